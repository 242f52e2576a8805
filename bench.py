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
NCU_SUMMARY = {"decode": "profiles/mla_decode_kernel_B64_H128_ncu_full.md"}


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


def cpu_baseline(inp, seconds: float = 12.0):
    """Time the oracle on a bounded sample of the workload (rank 0, N=1):
    about `seconds` of host work; a sample smaller than that is repeated."""
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
    return {"value": reps * flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{nreq} of {inp.batch} requests x {R} rows ({flops/1e9:.2f} GFLOP), run {reps}x in {dt:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="decode", choices=list(gen.WORKLOADS))
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
    q = inp.q.to(dev)
    kv = inp.kv.to(dev)
    sc = inp.kv_scales.to(dev) if inp.kv_scales is not None else None
    bt = inp.block_table.to(dev)
    sl = inp.seqlens.to(dev)
    dec = mla.MlaDecoder(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq, kv_fp8=inp.kv_fp8,
                         rope_bf16=inp.rope_bf16,
                         device=dev)
    d = dec.desc
    ws = dec.workspace
    out = torch.empty((inp.batch, inp.s_q, inp.heads, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((inp.batch, inp.s_q, inp.heads), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

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
        mla.mla_combine(d, out, lse, ws, stream)

    for _ in range(args.warmup):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    st = dec.device_error()
    if st != mla.MLA_OK:
        raise RuntimeError(f"device error during warm-up: {mla.status_string(st)}")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    k_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    props = torch.cuda.get_device_properties(dev)
    clocks = ClockSampler(f"GPU-{props.uuid}" if getattr(props, "uuid", None) else str(local))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    # the attention kernel alone (events around it), same inputs and flushes
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(k_a[i], k_b[i])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kern_ms = [a.elapsed_time(b) for a, b in zip(k_a, k_b)]
    ms = sum(step_ms) / len(step_ms)
    kms = sum(kern_ms) / len(kern_ms)
    ms, kms = max_over_ranks([ms, kms], dev)

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

    hbm_gbs, tflops_peak, tflops_sust, peak_src = load_peaks()
    tflops = world * flops / (ms * 1e-3) / 1e12
    kv_gbs = world * kv_bytes / (ms * 1e-3) / 1e9
    t_roof = max(flops / (tflops_peak * 1e12), kv_bytes / (hbm_gbs * 1e9))
    k_tflops = flops / (kms * 1e-3) / 1e12
    k_gbs = kv_bytes / (kms * 1e-3) / 1e9
    hbm_bound = kv_bytes / (hbm_gbs * 1e9) >= flops / (tflops_peak * 1e12)
    if hbm_bound:
        roof = {"kernel": "mla_decode_kernel<bf16>" if not inp.kv_fp8 else "mla_decode_kernel<fp8>", "bound": "hbm",
                "achieved": k_gbs, "peak": hbm_gbs, "unit": "GB/s", "frac": k_gbs / hbm_gbs,
                "traffic": measured_traffic(args.workload), "peak_source": f"{peak_src} hbm_gbs (burst, kernel timed alone)",
                "algorithmic_bytes_per_launch": kv_bytes}
    else:
        roof = {"kernel": "mla_decode_kernel<bf16>" if not inp.kv_fp8 else "mla_decode_kernel<fp8>", "bound": "tensor",
                "achieved": k_tflops, "peak": tflops_peak, "unit": "TFLOP/s", "frac": k_tflops / tflops_peak,
                "traffic": None, "peak_source": f"{peak_src} bf16_tflops (burst, kernel timed alone)",
                "algorithmic_flops_per_launch": flops}
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
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
