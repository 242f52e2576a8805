"""Parity of the CUDA path (through the C ABI) with the fp64 CPU oracle.

Every case is compared on every output row, the full-size workloads included
(in the launch configuration the benchmark times).  Tolerances (max abs / relative L2
/ lse abs): bf16 cache 2e-2 / 5e-3 / 1e-3, fp8 cache 6e-2 / 2e-2 / 1e-3.
Indexing (block table, page offsets, causal limit) is checked bit-exactly with
planted one-hot attention.
"""
import math

import numpy as np
import pytest
import torch

import mla_paged_decode_absorbed_gb300 as mla
import oracle
from oracle import plan_ref
from workloads import gen
from tests.gpu_helpers import TOL_BF16, TOL_FP8, compare, run_gpu, to_device

pytestmark = pytest.mark.gpu

# Split units of at most this many pieces are merged inside the attention
# kernel; units of more pieces are combine jobs (workspace header word 6).
FUSE_MAX = 3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    mla.library()
    torch.cuda.set_device(0)


def _check(inp, tol=None, rows=None, **kw):
    """The CUDA path against the oracle under the stated tolerances (the fp8
    caches included: lse within 1e-3 on every row)."""
    tol = tol or (TOL_FP8 if inp.kv_fp8 else TOL_BF16)
    out_g, lse_g, status, _ = run_gpu(inp, **kw)
    assert status == mla.MLA_OK, mla.status_string(status)
    if rows is None:
        out_r, lse_r = oracle.mla_decode_inputs(inp)
        return compare(out_g, lse_g, out_r, lse_r, tol)
    out_r, lse_r = oracle.mla_decode_inputs(inp, rows=rows)
    assert np.isfinite(out_g).all()
    return compare(out_g[rows.numpy()], lse_g[rows.numpy()], out_r, lse_r, tol)


# ------------------------------------------------------------------ workloads
def test_tiny_workload_every_output():
    _check(gen.make_inputs("tiny"))


@pytest.mark.parametrize("name,kw", [
    ("decode", dict(batch=6)),
    ("mtp", dict(batch=2)),
    ("long", dict(seqlens=[20000, 3000, 64, 700])),
    ("fp8", dict(batch=3)),
    ("fp8b", dict(batch=3)),
])
def test_reduced_workloads_every_output(name, kw):
    _check(gen.make_inputs(name, **kw))


@pytest.mark.parametrize("name", ["decode", "mtp", "long", "fp8", "mtp6", "fp8b"])
def test_full_size_workloads_every_row(name):
    """Each full-size workload in the benchmark's launch configuration (the
    default clusters and plan), compared with the oracle on EVERY output row.
    The oracle runs all rows on the host cores (tens of seconds for the
    largest workloads)."""
    _check(gen.make_inputs(name))


# ------------------------------------------------------------------ splits and shapes
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("clusters,ovh", [(1, 1), (2, 2), (3, 1), (7, 3)])
def test_forced_splits_match(clusters, ovh, fp8):
    """Many segments per cluster (ring stages and barrier phases carry over
    segment and unit boundaries, including empty units), split units merged
    in the kernel and in the combine kernel; for the fp8 cache also the
    per-page exchange of converted blocks between the two CTAs."""
    inp = gen.make_inputs("x", seqlens=[1000, 64, 1, 2500, 130], heads=32, s_q=2, kv_fp8=fp8, seed=31)
    _check(inp, max_clusters=clusters, plan_overhead=ovh)


@pytest.mark.parametrize("seqlens,heads,s_q,fp8", [
    ([1], 16, 1, False),                 # a single key
    ([64, 128, 192], 16, 1, False),      # page-aligned ends (no tail to mask)
    ([1, 0, 2], 8, 2, False),            # no visible key for some rows
    ([300, 77], 20, 3, False),           # rows of several tokens in one block, H not dividing 128
    ([129, 70], 16, 8, False),           # 8 tokens x 16 heads = one full block
    ([500, 257], 256, 1, False),         # two row blocks per request
    ([200], 128, 16, False),             # 16 row blocks, causal across blocks
    ([65, 3, 128], 16, 1, True),         # fp8 tails and a 3-key request
    ([333], 40, 5, True),                # fp8 with causal verify of 5 tokens
    ([4096, 700, 3], 128, 6, False),     # five draft tokens, 768 rows per request, a request shorter than s_q
    ([2000, 5, 130], 128, 6, True),      # the same with the fp8 cache
])
def test_edge_shapes(seqlens, heads, s_q, fp8):
    _check(gen.make_inputs("x", seqlens=seqlens, heads=heads, s_q=s_q, kv_fp8=fp8, seed=sum(seqlens) + heads))


@pytest.mark.parametrize("seqlens,heads,s_q,clusters", [
    ([65, 3, 128], 16, 1, 0),            # tails and a 3-key request
    ([1], 4, 1, 0),                      # a single key (lse is that key's score)
    ([2000, 5, 130], 128, 6, 0),         # five draft tokens, a request shorter than s_q
    ([1000, 64, 1, 2500, 130], 32, 2, 3),  # many segments per cluster, split units merged
])
def test_fp8_variant_b(seqlens, heads, s_q, clusters):
    """fp8 variant B: 656-byte token records (e4m3 latent with four scales
    inside the record, RoPE kept in bf16)."""
    inp = gen.make_inputs("x", seqlens=seqlens, heads=heads, s_q=s_q, kv_fp8=True, rope_bf16=True,
                          seed=sum(seqlens) + heads + 5)
    _check(inp, max_clusters=clusters)


def test_fp8_variant_b_bad_page_is_reported():
    inp = gen.make_inputs("x", seqlens=[300, 50], heads=16, s_q=1, kv_fp8=True, rope_bf16=True, seed=4)
    inp.block_table[0, 2] = inp.num_pages + 5
    out_g, lse_g, status, _ = run_gpu(inp)
    assert status == mla.MLA_ERR_DEVICE_BOUNDS
    assert np.isfinite(out_g).all()
    out_r, lse_r = oracle.mla_decode(inp.q[1:], inp.kv, inp.block_table[1:], inp.seqlens[1:], 1, inp.softmax_scale,
                                     kv_dtype=oracle.KV_FP8B)
    compare(out_g[16:], lse_g[16:], out_r, lse_r, TOL_FP8)


def test_full_pool_no_spare_and_max_pages():
    inp = gen.make_inputs("x", seqlens=[64 * 7, 64 * 3 + 5], heads=16, s_q=1, seed=5, spare_frac=0.0)
    _check(inp)


# ------------------------------------------------------------------ exact indexing
def _planted(seqlens, heads, s_q, seed):
    """Every head of every token gets one planted key with a huge score; the
    output must then be that key's latent row, bit for bit."""
    inp = gen.make_inputs("x", seqlens=seqlens, heads=heads, s_q=s_q, seed=seed)
    g = torch.Generator().manual_seed(seed)
    kv = (torch.randn(inp.kv.shape, generator=g) * 0.01).to(torch.bfloat16)
    q = torch.zeros(inp.q.shape, dtype=torch.bfloat16)
    want = {}
    R = s_q * heads
    for b, sl in enumerate(seqlens):
        for i in range(s_q):
            n = sl - s_q + i + 1
            if n <= 0:
                continue
            for h in range(heads):
                ch = (i * heads + h) % 512   # distinct per row of a request
                t = int(torch.randint(0, n, (1,), generator=g))
                page = int(inp.block_table[b, t // 64])
                kv[page, t % 64, ch] = 1.0
                q[b, i, h, ch] = 2000.0
                want[b * R + i * heads + h] = (page, t % 64)
    inp.kv, inp.q = kv, q
    return inp, want


@pytest.mark.parametrize("seqlens,heads,s_q,clusters", [
    ([130, 37, 700], 16, 1, 0),
    ([1000, 4096], 128, 2, 0),
    ([3000, 65, 1], 32, 3, 5),
])
def test_planted_one_hot_is_bit_exact(seqlens, heads, s_q, clusters):
    inp, want = _planted(seqlens, heads, s_q, seed=77 + heads)
    out_g, lse_g, status, _ = run_gpu(inp, max_clusters=clusters)
    assert status == mla.MLA_OK
    kv = inp.kv.float().numpy()
    for r, (p, s) in want.items():
        assert np.array_equal(out_g[r], kv[p, s, :512]), f"row {r} did not read page {p} slot {s}"
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(out_g, lse_g, out_r, lse_r, TOL_BF16)


def test_causal_limit_hides_later_draft_tokens():
    inp = gen.make_inputs("x", seqlens=[100, 64], heads=16, s_q=2, seed=3)
    kv = (inp.kv.float() * 0.01).to(torch.bfloat16)
    q = (inp.q.float() * 0.01).to(torch.bfloat16)
    for b, sl in enumerate([100, 64]):
        t = sl - 1
        page = int(inp.block_table[b, t // 64])
        kv[page, t % 64, 5] = 1.0
        q[b, :, :, 5] = 2000.0
    inp.kv, inp.q = kv, q
    out_g, lse_g, status, _ = run_gpu(inp)
    assert status == mla.MLA_OK
    o = out_g.reshape(2, 2, 16, 512)
    assert (o[:, 1, :, 5] == 1.0).all()          # token 1 sees the last key
    assert (np.abs(o[:, 0, :, 5]) < 0.5).all()   # token 0 does not
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(out_g, lse_g, out_r, lse_r, TOL_BF16)


def test_verify_equals_batch_extension_on_gpu():
    inp = gen.make_inputs("x", seqlens=[700, 129, 4000], heads=64, s_q=2, seed=9)
    out2, lse2, st, _ = run_gpu(inp)
    assert st == mla.MLA_OK
    out2 = out2.reshape(3, 2, 64, 512)
    lse2 = lse2.reshape(3, 2, 64)
    for i in range(2):
        one = gen.make_inputs("x", seqlens=[700, 129, 4000], heads=64, s_q=1, seed=9)
        one.q = inp.q[:, i:i + 1].contiguous()
        one.kv, one.block_table = inp.kv, inp.block_table
        one.seqlens = (inp.seqlens - 1 + i).to(torch.int32)
        o1, l1, st, _ = run_gpu(one)
        assert st == mla.MLA_OK
        np.testing.assert_allclose(o1.reshape(3, 64, 512), out2[:, i], atol=1.6e-2, rtol=0)
        np.testing.assert_allclose(l1.reshape(3, 64), lse2[:, i], atol=2e-5, rtol=0)


# ------------------------------------------------------------------ the plan
@pytest.mark.parametrize("seqlens,heads,s_q,clusters,ovh", [
    ([37, 130], 16, 1, 0, 0),
    ([1000, 64, 1, 2500, 130, 0], 128, 2, 9, 3),      # two row blocks, clusters split between them
    ([1000, 64, 1, 2500, 130, 0], 128, 6, 4, 2),      # six row blocks on four clusters: one after another
    ([4097, 300, 65], 128, 6, 0, 2),                  # six row blocks, every cluster
    (list(range(1, 4000, 97)), 64, 1, 0, 1),
])
def test_device_plan_equals_reference_plan(seqlens, heads, s_q, clusters, ovh):
    inp = gen.make_inputs("x", seqlens=seqlens, heads=heads, s_q=s_q, seed=1)
    d = mla.make_desc(inp.batch, s_q, heads, inp.num_pages, inp.max_pages_per_seq, max_clusters=clusters,
                      plan_overhead=ovh)
    ws = mla.alloc_workspace(d)
    G = mla.mla_num_clusters(d)
    sl = inp.seqlens.cuda()
    mla.mla_plan(d, sl, ws)
    torch.cuda.synchronize()
    lay = mla.mla_get_workspace_layout(d, G)
    w = ws.cpu()
    hdr = w[lay.header:lay.header + 28].view(torch.int32).tolist()
    ref = plan_ref.make_plan(seqlens, s_q, heads, inp.max_pages_per_seq, G, ovh or plan_ref.DEFAULT_OVERHEAD)
    many = sum(1 for u in range(ref.units) if ref.piece_count(u) > FUSE_MAX)
    assert hdr == [0, ref.W, ref.pre[-1], ref.units, G, ref.overhead, many]
    assert w[lay.sync:lay.sync + 12 * G].view(torch.int32).eq(0).all()
    pre = w[lay.pre:lay.pre + 4 * (ref.units + 1 + ref.n_rb)].view(torch.int32).tolist()
    assert pre == ref.pre + ref.rb_ends
    cl_first = w[lay.cl_first:lay.cl_first + 4 * G].view(torch.int32).tolist()
    assert cl_first == [ref.first_unit(c) for c in range(G)]


# ------------------------------------------------------------------ device errors
@pytest.mark.parametrize("fp8", [False, True])
def test_page_id_out_of_pool_is_reported_not_faulted(fp8):
    inp = gen.make_inputs("x", seqlens=[300, 50], heads=16, s_q=1, kv_fp8=fp8, seed=4)
    inp.block_table[0, 2] = inp.num_pages + 5
    out_g, lse_g, status, _ = run_gpu(inp)
    assert status == mla.MLA_ERR_DEVICE_BOUNDS
    assert np.isfinite(out_g).all()
    # the other request is untouched by the bad entry
    out_r, lse_r = oracle.mla_decode(inp.q[1:], inp.kv, inp.block_table[1:], inp.seqlens[1:], 1, inp.softmax_scale,
                                     kv_scales=inp.kv_scales, kv_dtype=oracle.KV_FP8 if fp8 else oracle.KV_BF16)
    compare(out_g[16:], lse_g[16:], out_r, lse_r, TOL_FP8 if fp8 else TOL_BF16)


def test_seqlen_beyond_block_table_is_reported():
    inp = gen.make_inputs("x", seqlens=[100, 64], heads=16, s_q=1, seed=4)
    inp.seqlens[1] = 64 * inp.max_pages_per_seq + 1
    _, _, status, _ = run_gpu(inp)
    assert status == mla.MLA_ERR_DEVICE_BOUNDS


def test_error_word_clears_on_next_good_call():
    inp = gen.make_inputs("x", seqlens=[100, 64], heads=16, s_q=1, seed=4)
    bad = gen.make_inputs("x", seqlens=[100, 64], heads=16, s_q=1, seed=4)
    bad.block_table[0, 0] = -7
    _, _, st, dec = run_gpu(bad)
    assert st == mla.MLA_ERR_DEVICE_BOUNDS
    _, _, st, _ = run_gpu(inp, decoder=dec)
    assert st == mla.MLA_OK


# ------------------------------------------------------------------ determinism, streams, graphs
@pytest.mark.parametrize("fp8", [False, True])
def test_repeated_calls_are_bitwise_identical(fp8):
    inp = gen.make_inputs("x", seqlens=[3000, 17, 900], heads=128, s_q=1, kv_fp8=fp8, seed=6)
    t = to_device(inp)
    o1, l1, _, dec = run_gpu(inp, tensors=t, max_clusters=5)
    o2, l2, _, _ = run_gpu(inp, tensors=t, decoder=dec)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_side_stream_and_cuda_graph_replay():
    """The step runs on a side stream and captures into a CUDA graph.  The
    plan is recomputed on the device at every replay, so writing new seqlens
    and block-table entries into the same device tensors between replays
    changes the work: each replay is checked against the oracle on the inputs
    it saw."""
    inp = gen.make_inputs("x", seqlens=[1500, 33], heads=64, s_q=2, seed=8)
    q, kv, sc, bt, sl = to_device(inp)
    dec = mla.MlaDecoder(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq)
    out = torch.empty((inp.batch, inp.s_q, inp.heads, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((inp.batch, inp.s_q, inp.heads), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dec(q, kv, bt, sl, inp.softmax_scale, out=out, lse=lse, stream=s)
    s.synchronize()
    ref_o, ref_l = out.clone(), lse.clone()
    out.zero_()
    lse.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec(q, kv, bt, sl, inp.softmax_scale, out=out, lse=lse, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    assert dec.device_error() == mla.MLA_OK

    def check_replay():
        out_r, lse_r = oracle.mla_decode_inputs(inp)
        compare(out.float().cpu().numpy().reshape(-1, 512).astype(np.float64),
                lse.cpu().numpy().reshape(-1).astype(np.float64), out_r, lse_r, TOL_BF16)

    check_replay()
    # new lengths (request 0 shorter, request 1 longer) and a reshuffled block
    # table over the same pool, written in place; the captured graph replays
    # with them and must follow: its plan is rebuilt from the new seqlens
    for seqlens in ([700, 900], [64, 1501], [1501, 0]):
        maxp = inp.max_pages_per_seq
        need = [(n + 63) // 64 for n in seqlens]
        assert max(need) <= maxp and sum(need) <= inp.num_pages
        perm = torch.randperm(inp.num_pages, generator=torch.Generator().manual_seed(sum(seqlens)))
        table = torch.full((inp.batch, maxp), -1, dtype=torch.int32)
        cur = 0
        for b, n in enumerate(need):
            table[b, :n] = perm[cur:cur + n].to(torch.int32)
            cur += n
        # the pages now owned may be old spare (NaN) pages: refill the pool with finite values
        kv_new = (torch.randn(inp.kv.shape, generator=torch.Generator().manual_seed(3 + sum(seqlens)))).to(torch.bfloat16)
        inp.kv, inp.block_table = kv_new, table
        inp.seqlens = torch.tensor(seqlens, dtype=torch.int32)
        kv.copy_(kv_new)
        bt.copy_(table)
        sl.copy_(inp.seqlens)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert dec.device_error() == mla.MLA_OK
        check_replay()


# ------------------------------------------------------------------ split merges
@pytest.mark.parametrize("clusters,fp8", [(3, False), (5, False), (12, False), (40, False), (5, True), (40, True)])
def test_merge_in_kernel_and_in_combine(clusters, fp8):
    """Units split into 2..FUSE_MAX pieces are merged by the attention
    kernel's last finisher; units with more pieces by the combine kernel.
    Both must match."""
    seqlens = [9000, 64, 3100, 700, 1, 2000]
    inp = gen.make_inputs("x", seqlens=seqlens, heads=128, s_q=1, kv_fp8=fp8, seed=40 + clusters)
    d = mla.make_desc(inp.batch, 1, 128, inp.num_pages, inp.max_pages_per_seq, max_clusters=clusters)
    G = mla.mla_num_clusters(d)
    ref = plan_ref.make_plan(seqlens, 1, 128, inp.max_pages_per_seq, G, plan_ref.DEFAULT_OVERHEAD)
    counts = {ref.piece_count(u) for u in range(ref.units)}
    assert counts & set(range(2, FUSE_MAX + 1)) or max(counts) > FUSE_MAX, counts
    _check(inp, max_clusters=clusters)


def test_attention_rerun_without_replanning():
    """The attention kernel leaves the merge counters and slot flags clear, so
    plan once, then attention + combine twice gives the same result."""
    inp = gen.make_inputs("x", seqlens=[5000, 2500, 300], heads=128, s_q=1, seed=77)
    q, kv, sc, bt, sl = to_device(inp)
    d = mla.make_desc(inp.batch, 1, 128, inp.num_pages, inp.max_pages_per_seq, max_clusters=9)
    ws = mla.alloc_workspace(d)
    G = mla.mla_num_clusters(d)
    lay = mla.mla_get_workspace_layout(d, G)
    outs = []
    mla.mla_plan(d, sl, ws)
    for _ in range(2):
        out = torch.zeros((inp.batch, 1, 128, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.zeros((inp.batch, 1, 128), dtype=torch.float32, device="cuda")
        mla.mla_decode_attention(d, q, kv, None, bt, sl, 1, inp.softmax_scale, out, lse, ws)
        mla.mla_combine_workspace(d, out, lse, ws)
        torch.cuda.synchronize()
        assert ws[lay.sync:lay.sync + 12 * G].view(torch.int32).eq(0).all()
        outs.append((out.clone(), lse.clone()))
    assert mla.mla_get_device_error(ws) == mla.MLA_OK
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(outs[0][0].float().cpu().numpy().reshape(-1, 512).astype(np.float64),
            outs[0][1].cpu().numpy().reshape(-1).astype(np.float64), out_r, lse_r, TOL_BF16)


# ------------------------------------------------------------------ timeout path
@pytest.mark.parametrize("fp8", [False, True])
def test_pipeline_timeout_is_reported_and_the_context_stays_usable(fp8):
    """A stall request (workspace header word 7, written after the plan) makes
    every scorer wait on a barrier nothing signals.  The bounded wait runs out
    (about a second), both CTAs of every cluster take the abort path and tear
    down, the call reports MLA_ERR_DEVICE_TIMEOUT, and the next call on the
    same context (whose plan clears the request) is correct.  No fault, trap
    or unbounded wait is involved."""
    import time
    inp = gen.make_inputs("x", seqlens=[700, 300], heads=16, s_q=1, kv_fp8=fp8, seed=12)
    t = to_device(inp)
    q, kv, sc, bt, sl = t
    d = mla.make_desc(inp.batch, 1, 16, inp.num_pages, inp.max_pages_per_seq, kv_fp8=fp8)
    ws = mla.alloc_workspace(d)
    lay = mla.mla_get_workspace_layout(d, mla.mla_num_clusters(d))
    out = torch.zeros((inp.batch, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((inp.batch, 1, 16), dtype=torch.float32, device="cuda")
    mla.mla_plan(d, sl, ws)
    ws[lay.header + 28:lay.header + 32].view(torch.int32).fill_(1)
    t0 = time.monotonic()
    mla.mla_decode_attention(d, q, kv, sc, bt, sl, 1, inp.softmax_scale, out, lse, ws)
    mla.mla_combine_workspace(d, out, lse, ws)
    assert mla.mla_get_device_error(ws) == mla.MLA_ERR_DEVICE_TIMEOUT
    assert time.monotonic() - t0 < 30
    out_g, lse_g, status, dec = run_gpu(inp, tensors=t)
    assert status == mla.MLA_OK
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(out_g, lse_g, out_r, lse_r, TOL_FP8 if fp8 else TOL_BF16)
