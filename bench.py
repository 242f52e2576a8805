"""Benchmark of the MLA paged-decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = the whole hot path on one batch: split plan, attention over the
pages, LSE combine (three kernels of libmla_gb300.so, called through the C ABI)
on the named workload (default: the B=64, H=128 decode workload).  Inputs are
seeded synthetic data (workloads/gen.py), resident in HBM before timing.

Timing: W >= 3 untimed warm-up steps; then K steps, each bracketed by CUDA
events on the launching stream, with a 512 MiB L2 flush (a buffer write)
between steps outside the events; barrier + synchronize on both sides of the
K steps; max over ranks.  Rank 0 prints one JSON line.

Metric: TFLOP/s, counting 2*576 + 2*512 = 2176 flops per (query row, visible
key); the line also carries KV GB/s (unique cache bytes read: 1152 B/token
bf16, 596 B/token fp8 incl. scales) and the fraction of the roofline
max(flops / tensor peak, KV bytes / HBM peak) for the step.

--impl reference times the fp64 CPU oracle (the reference of this build) on
a bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from workloads import gen  # noqa: E402

METRIC = "MLA decode TFLOP/s and KV GB/s at B=64,H=128 (1 GB300) + % of roofline"
FLOP_PER_ROW_KEY = 2 * 576 + 2 * 512
L2_FLUSH_BYTES = 512 << 20

WORKLOAD_TEXT = {
    "tiny": "tiny: B=2 s_q=1 H=16 seqlens {37,130}, bf16 cache, page 64",
    "decode": "decode: B=64 s_q=1 H=128 seqlens U[1024,4096], bf16 q and latent cache, page 64, scale 1/sqrt(192)",
    "mtp": "MTP verify: B=128 s_q=2 (causal) H=128 seqlen 4096, bf16, page 64",
    "mtp6": "MTP verify of five draft tokens: B=64 s_q=6 (causal) H=128 seqlen 4096, bf16, page 64",
    "fp8b": "fp8 cache variant B: B=256 s_q=2 (causal) H=128 seqlen 2048, 656-byte token records (e4m3 latent, 4 fp32 scales, bf16 RoPE)",
    "long": "long skewed: B=16 s_q=1 H=128 lognormal seqlens (mean 3500, sigma 1) + one 65536, bf16, page 64",
    "fp8": "fp8 cache: B=256 s_q=2 (causal) H=128 seqlen 2048, e4m3 cache + fp32 scale per token per 128-ch group",
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


KERNEL_SOURCES = ("mla_paged_decode_absorbed_gb300/csrc/mla_decode_kernel.cu",
                  "mla_paged_decode_absorbed_gb300/csrc/sm103_ptx.cuh",
                  "mla_paged_decode_absorbed_gb300/csrc/mla_internal.h")
NCU_SUMMARY = {"decode": "profiles/mla_decode_kernel_B64_H128_ncu_full.md",
               "mtp": "profiles/mla_decode_kernel_mtp_B128_ncu_full.md",
               "fp8": "profiles/mla_decode_kernel_fp8_B256_ncu_full.md"}


def measured_traffic(workload):
    """DRAM bytes per launch of the attention kernel from the committed ncu
    summary of this workload, or None when there is none or the kernel
    sources changed since it was captured (sha256 recorded beside it)."""
    import hashlib
    name = NCU_SUMMARY.get(workload)
    if name is None:
        return None
    try:
        text = open(os.path.join(ROOT, name)).read()
        h = hashlib.sha256()
        for f in KERNEL_SOURCES:
            with open(os.path.join(ROOT, f), "rb") as fh:
                h.update(fh.read())
        fields = dict(line.split(": ", 1) for line in text.splitlines() if line.startswith(("dram_bytes", "kernel_source")))
        if fields.get("kernel_source_sha256", "").strip() != h.hexdigest():
            return None
        return int(fields["dram_bytes_per_launch"])
    except Exception:
        return None


def work_of(inp):
    """(flops, kv_bytes) of one call: per row the visible keys, per request the
    cache bytes of the tokens the longest row sees."""
    flops = 0
    kv_bytes = 0
    per_tok = (656 if inp.rope_bf16 else 596) if inp.kv_fp8 else 1152
    for s in inp.seqlens.tolist():
        for i in range(inp.s_q):
            n = max(0, s - inp.s_q + i + 1)
            flops += inp.heads * n * FLOP_PER_ROW_KEY
        kv_bytes += max(0, s) * per_tok
    return flops, kv_bytes


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None
        self.path = None
        self.out = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.device_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            if self.out is not None:
                self.out.close()
                os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            self.proc.wait()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def replica_inputs(workload: str, rank: int):
    """Each data-parallel replica decodes its own independent batch of the
    same workload (weak scaling): same recipe, seed offset by the rank."""
    return gen.make_inputs(workload, seed=gen.workload_spec(workload).seed + 1000 * rank)


def max_over_ranks(values, device):
    """Element-wise MAX of per-rank timings (a no-op without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return list(values)
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def _request_flops(inp, b):
    s = int(inp.seqlens[b])
    return sum(inp.heads * max(0, s - inp.s_q + i + 1) for i in range(inp.s_q)) * FLOP_PER_ROW_KEY


def oracle_sample(inp, seconds: float):
    """Rows of the first requests of the workload (all their heads and tokens)
    sized, from a one-request calibration run, to about `seconds` of oracle
    work on the host cores; the whole batch when it takes less."""
    import oracle
    R = inp.s_q * inp.heads
    first = torch.arange(0, R, dtype=torch.int64)
    t0 = time.perf_counter()
    oracle.mla_decode_inputs(inp, rows=first)
    rate = _request_flops(inp, 0) / max(time.perf_counter() - t0, 1e-6)
    budget = rate * seconds
    rows, flops = [], 0
    for b in range(inp.batch):
        f = _request_flops(inp, b)
        if rows and flops + f > budget:
            break
        rows.extend(range(b * R, (b + 1) * R))
        flops += f
    return torch.tensor(rows, dtype=torch.int64), flops, len(rows) // R


def reference_arm(args):
    """The fp64 CPU oracle on a bounded sample of the workload, per step."""
    import oracle
    world, rank, _ = dist_env()
    if rank != 0:
        return
    inp = gen.make_inputs(args.workload)
    R = inp.s_q * inp.heads
    rows_t, flops, nreq = oracle_sample(inp, 2.0)   # about 2 s of host work per step
    for _ in range(args.warmup):
        oracle.mla_decode_inputs(inp, rows=rows_t)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.mla_decode_inputs(inp, rows=rows_t)
    dt = (time.perf_counter() - t0) / args.steps
    tflops = flops / dt / 1e12
    cores = oracle.num_threads()
    sample = (f"{nreq} of {inp.batch} requests x {R} rows of the {args.workload} workload per step "
              f"({flops/1e9:.2f} GFLOP)")
    line = {
        "impl": "reference", "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, workloads/gen.py)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "sample": sample},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def absorption_gemms(inp, flush, hbm_gbs, tflops_peak, iters: int = 10):
    """Times the absorption GEMMs (mla_absorb_q, mla_project_out) on this
    workload's token rows (B*s_q) and heads, with random bf16 weights of the
    MLA shape (H x 512 x 128), L2 flushed before each launch.  Each is HBM-bound
    on its weights at few tokens and tensor-bound at many; reported against
    the bound that applies."""
    import mla_paged_decode_absorbed_gb300 as mla
    T, H = inp.batch * inp.s_q, inp.heads
    g = torch.Generator(device="cuda").manual_seed(4242)
    rn = lambda *shape: (torch.randn(shape, device="cuda", generator=g) / 8).to(torch.bfloat16)
    q_nope, q_rope, w_uk, w_uv, outl = rn(T, H, 128), rn(T, H, 64), rn(H, 512, 128), rn(H, 512, 128), rn(T, H, 512)
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device="cuda")
    o = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    res = {}
    for name, fn, nbytes in (
            ("absorb_q", lambda: mla.mla_absorb_q(q_nope, q_rope, w_uk, q), H * 512 * 128 * 2 + T * H * (192 + 576) * 2),
            ("project_out", lambda: mla.mla_project_out(outl, w_uv, o), H * 512 * 128 * 2 + T * H * (512 + 128) * 2)):
        flops = 2.0 * T * H * 512 * 128
        for _ in range(3):
            fn()
        times = []
        for it in range(iters):
            flush.fill_(it & 0xFF)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        ms = sorted(times)[len(times) // 2]
        hbm = nbytes / (hbm_gbs * 1e9) >= flops / (tflops_peak * 1e12)
        ach = (nbytes / (ms * 1e-3) / 1e9) if hbm else (flops / (ms * 1e-3) / 1e12)
        peak = hbm_gbs if hbm else tflops_peak
        res[name] = {"us": ms * 1e3, "bound": "hbm" if hbm else "tensor", "achieved": ach,
                     "unit": "GB/s" if hbm else "TFLOP/s", "peak": peak, "frac": ach / peak,
                     "algorithmic_bytes": nbytes, "flops": flops}
    res["shape"] = f"tokens={T} heads={H}, weights [H,512,128] bf16, L2 flushed before each launch"
    return res


def cpu_model() -> str:
    """CPU model of this host: lscpu's model name (Arm hosts have no model
    name in /proc/cpuinfo), else /proc/cpuinfo, else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_one_core(name: str, **kw):
    """The oracle on one host core over every row of a small workload: GFLOP/s."""
    import oracle
    inp = gen.make_inputs(name, **kw)
    flops, _ = work_of(inp)
    oracle.set_num_threads(1)
    try:
        oracle.mla_decode_inputs(inp)          # warm caches and the library
        t0 = time.perf_counter()
        reps = 0
        while True:
            oracle.mla_decode_inputs(inp)
            reps += 1
            dt = time.perf_counter() - t0
            if dt >= 1.0 or reps >= 50:
                break
    finally:
        oracle.set_num_threads(os.cpu_count() or 1)
    return {"gflops": reps * flops / dt / 1e9, "seconds_per_call": dt / reps, "gflop_per_call": flops / 1e9}


def cpu_baseline(inp, seconds: float = 12.0):
    """Time the oracle on a bounded sample of the workload (rank 0, N=1):
    about `seconds` of host work on all cores; a sample smaller than that is
    repeated.  Also the oracle on ONE core over every row of the tiny workload
    and of a four-request cut of the decode workload, and the CPU model."""
    import oracle
    R = inp.s_q * inp.heads
    rows_t, flops, nreq = oracle_sample(inp, seconds)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.mla_decode_inputs(inp, rows=rows_t)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= 0.8 * seconds or reps >= 20:
            break
    cores = oracle.num_threads()
    per_core = {"tiny (every row)": oracle_one_core("tiny"),
                "decode B=4 (every row)": oracle_one_core("decode", batch=4)}
    return {"value": reps * flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{nreq} of {inp.batch} requests x {R} rows ({flops/1e9:.2f} GFLOP), run {reps}x in {dt:.1f} s",
            "cpu_model": cpu_model(), "one_core": per_core}


def roofline_of(inp, flops, kv_bytes, kms, hbm_gbs, tflops_peak, peak_src, workload):
    """Roofline entry of the attention kernel: HBM-bound (cache bytes / HBM
    peak) or tensor-bound (flops / dense 16-bit tensor peak), whichever takes
    longer at the measured peaks."""
    name = "mla_decode_kernel<bf16>" if not inp.kv_fp8 else "mla_decode_kernel<fp8>"
    if kv_bytes / (hbm_gbs * 1e9) >= flops / (tflops_peak * 1e12):
        ach = kv_bytes / (kms * 1e-3) / 1e9
        return {"kernel": name, "bound": "hbm", "achieved": ach, "peak": hbm_gbs, "unit": "GB/s", "frac": ach / hbm_gbs,
                "traffic": measured_traffic(workload), "peak_source": f"{peak_src} hbm_gbs (burst, kernel timed alone)",
                "algorithmic_bytes_per_launch": kv_bytes}
    ach = flops / (kms * 1e-3) / 1e12
    return {"kernel": name, "bound": "tensor", "achieved": ach, "peak": tflops_peak, "unit": "TFLOP/s",
            "frac": ach / tflops_peak, "traffic": measured_traffic(workload),
            "peak_source": f"{peak_src} bf16_tflops (burst, kernel timed alone; fp16 has the same dense rate)",
            "algorithmic_flops_per_launch": flops}


def time_workload(mla, inp, dev, stream, flush, steps, warmup, clock_dev, sync_ranks):
    """Device-resident inputs of `inp`, W warm-up steps, then K timed steps
    (events around each step on the launching stream, L2 flushed between
    steps outside the events), then the attention kernel alone in a second
    loop of the same steps.  Clocks are sampled over both loops."""
    q = inp.q.to(dev)
    kv = inp.kv.to(dev)
    sc = inp.kv_scales.to(dev) if inp.kv_scales is not None else None
    bt = inp.block_table.to(dev)
    sl = inp.seqlens.to(dev)
    dec = mla.MlaDecoder(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq, kv_fp8=inp.kv_fp8,
                         rope_bf16=inp.rope_bf16, device=dev)
    d, ws = dec.desc, dec.workspace
    out = torch.empty((inp.batch, inp.s_q, inp.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((inp.batch, inp.s_q, inp.heads), dtype=torch.float32, device=dev)

    def step(ev_a=None, ev_b=None):
        # The three kernels chain by programmatic dependent launch; events
        # between them (kernel timing) serialise the launches, so the step
        # loop runs without them and the kernel loop with them.
        mla.mla_plan(d, sl, ws, stream)
        if ev_a is not None:
            ev_a.record(stream)
        mla.mla_decode_attention(d, q, kv, sc, bt, sl, inp.s_q, inp.softmax_scale, out, lse, ws, stream)
        if ev_b is not None:
            ev_b.record(stream)
        mla.mla_combine_workspace(d, out, lse, ws, stream)

    for _ in range(warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    st = dec.device_error()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device error during warm-up: {mla.status_string(st)}")
    ev = lambda: torch.cuda.Event(enable_timing=True)
    starts, ends = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    k_a, k_b = [ev() for _ in range(steps)], [ev() for _ in range(steps)]
    clocks = ClockSampler(clock_dev)
    sync_ranks()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    for i in range(steps):
        flush.fill_(i & 0xFF)
        step(k_a[i], k_b[i])
    torch.cuda.synchronize()
    sync_ranks()
    clk = clocks.stop()
    st = dec.device_error()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device error in the timed steps: {mla.status_string(st)}")
    ms = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / steps
    kms = sum(a.elapsed_time(b) for a, b in zip(k_a, k_b)) / steps
    return {"ms": ms, "kms": kms, "clocks": clk, "dec": dec, "desc": d, "ws": ws,
            "tensors": (q, kv, sc, bt, sl, out, lse)}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode", choices=list(gen.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the per-workload map (the other six workloads)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        reference_arm(args)
        return

    import mla_paged_decode_absorbed_gb300 as mla

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    # each replica decodes its own batch of independent requests (weak scaling)
    inp = replica_inputs(args.workload, rank)
    flops, kv_bytes = work_of(inp)
    hbm_gbs, tflops_peak, tflops_sust, peak_src = load_peaks()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    props = torch.cuda.get_device_properties(dev)
    clock_dev = f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local)
    sync_ranks = (lambda: torch.distributed.barrier()) if world > 1 else (lambda: None)
    res = time_workload(mla, inp, dev, stream, flush, args.steps, args.warmup, clock_dev, sync_ranks)
    ms, kms = max_over_ranks([res["ms"], res["kms"]], dev)
    dec, d, ws = res["dec"], res["desc"], res["ws"]
    q, kv, sc, bt, sl, out, lse = res["tensors"]
    clk = res["clocks"]

    # end to end through the C ABI call with host buffers: H2D of the step's
    # inputs (q, block table, seqlens) from pinned memory, decode, D2H of out + lse
    e2e = None
    if not args.no_e2e:
        q_h = inp.q.pin_memory()
        bt_h = inp.block_table.pin_memory()
        sl_h = inp.seqlens.pin_memory()
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()

        def e2e_step():
            q.copy_(q_h, non_blocking=True)
            bt.copy_(bt_h, non_blocking=True)
            sl.copy_(sl_h, non_blocking=True)
            mla.mla_decode(d, q, kv, sc, bt, sl, inp.s_q, inp.softmax_scale, out, lse, ws, stream)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        e_s = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        e_e = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            e_s[i].record(stream)
            e2e_step()
            e_e[i].record(stream)
        torch.cuda.synchronize()
        ems = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / args.steps
        ems = max_over_ranks([ems], dev)[0]
        h2d = q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4
        d2h = out_h.numel() * 2 + lse_h.numel() * 4
        e2e = {"value": world * flops / (ems * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems}
        st = dec.device_error()
        if st != mla.MLA_OK:
            raise RuntimeError(f"device error in e2e leg: {mla.status_string(st)}")

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    tflops = world * flops / (ms * 1e-3) / 1e12
    kv_gbs = world * kv_bytes / (ms * 1e-3) / 1e9
    t_roof = max(flops / (tflops_peak * 1e12), kv_bytes / (hbm_gbs * 1e9))
    k_tflops = flops / (kms * 1e-3) / 1e12
    k_gbs = kv_bytes / (kms * 1e-3) / 1e9
    roof = roofline_of(inp, flops, kv_bytes, kms, hbm_gbs, tflops_peak, peak_src, args.workload)
    line = {
        "metric": METRIC, "value": tflops, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if not inp.kv_fp8 else ("fp16 (e4m3 latent + bf16 RoPE cache)" if inp.rope_bf16 else "fp16 (e4m3 cache)"),
        "data": "synthetic (seeded, workloads/gen.py)",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "l2": "flushed between steps (512 MiB buffer write)",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "clusters": dec.num_clusters, "step": "plan + attention + combine kernels (programmatic dependent launch)",
                   "kernel_timing": "attention kernel timed with events around it in a second loop of the same steps"},
        "kv_gbs": kv_gbs, "pct_roofline": t_roof / (ms * 1e-3),
        "decode_kernel_ms": kms, "decode_kernel_tflops": k_tflops, "decode_kernel_kv_gbs": k_gbs,
        "roofline": roof,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
    }
    if e2e is not None:
        line["e2e"] = e2e
    line["absorption_gemms"] = absorption_gemms(inp, flush, hbm_gbs, tflops_peak)
    if world == 1 and not args.no_workloads:
        # every other named workload, each in its own launch configuration,
        # timed the same way (fewer steps), with its own clock record
        wl = {}
        for name in gen.WORKLOADS:
            if name == args.workload:
                continue
            w_inp = gen.make_inputs(name)
            w_flops, w_bytes = work_of(w_inp)
            r = time_workload(mla, w_inp, dev, stream, flush, min(args.steps, 10), 3, clock_dev, sync_ranks)
            wl[name] = {
                "workload": WORKLOAD_TEXT[name], "step_ms": r["ms"], "kernel_ms": r["kms"],
                "tflops": w_flops / (r["ms"] * 1e-3) / 1e12, "kv_gbs": w_bytes / (r["ms"] * 1e-3) / 1e9,
                "pct_roofline": max(w_flops / (tflops_peak * 1e12), w_bytes / (hbm_gbs * 1e9)) / (r["ms"] * 1e-3),
                "roofline": roofline_of(w_inp, w_flops, w_bytes, r["kms"], hbm_gbs, tflops_peak, peak_src, name),
                "clocks": r["clocks"], "steps": min(args.steps, 10), "warmup": 3,
            }
            del r, w_inp
            torch.cuda.empty_cache()
        line["workloads"] = wl
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
