"""mla_combine on caller-supplied split-KV partials, against the oracle.

The partials are the oracle's own results over disjoint, page-aligned key
ranges of each request (the cache partitioning of the best-practice digest,
section 1.4): each range is attended by the oracle separately (block table
shifted to the range's first page, seqlen cut to the range), per new token so
that the causal limit of every row is respected.  The merge of those partials
must equal the oracle on the whole key range, at the bf16 tolerances.  Rows of
a partial that saw no key (lse -inf) are filled with NaN, which the kernel must
never read; a request with no partial gets out 0 and lse -inf.
"""
import numpy as np
import pytest
import torch

import mla_paged_decode_absorbed_gb300 as mla
import oracle
from workloads import gen
from tests.gpu_helpers import TOL_BF16, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    mla.library()
    torch.cuda.set_device(0)


def oracle_partials(inp, cuts_per_request):
    """o_part [K, R, 512], lse_part [K, R] (float64) and indptr [B+1] for the
    key ranges [c_j, c_{j+1}) of each request (cuts are key offsets, multiples
    of 64, starting at 0; the last range ends at the request's seqlen)."""
    B, s_q, H = inp.batch, inp.s_q, inp.heads
    R = s_q * H
    o_parts, l_parts, indptr = [], [], [0]
    for b in range(B):
        n = int(inp.seqlens[b])
        cuts = list(cuts_per_request[b])
        for j, a in enumerate(cuts):
            assert a % 64 == 0
            end = cuts[j + 1] if j + 1 < len(cuts) else n
            o = np.zeros((R, 512))
            l = np.full((R,), -np.inf)
            bt = inp.block_table[b:b + 1, a // 64:].contiguous()
            for i in range(s_q):
                visible = n - s_q + i + 1                      # keys row (i, h) sees in the whole problem
                m = max(0, min(end, visible) - a)
                if m == 0:
                    continue
                oi, li = oracle.mla_decode(inp.q[b:b + 1, i:i + 1].contiguous(), inp.kv, bt,
                                           torch.tensor([m], dtype=torch.int32), 1, inp.softmax_scale)
                o[i * H:(i + 1) * H] = oi
                l[i * H:(i + 1) * H] = li
            o[~np.isfinite(l)] = np.nan                        # rows that saw no key: must not be read
            o_parts.append(o)
            l_parts.append(l)
        indptr.append(len(o_parts))
    K = len(o_parts)
    o_part = np.stack(o_parts) if K else np.zeros((0, R, 512))
    l_part = np.stack(l_parts) if K else np.zeros((0, R))
    return o_part, l_part, np.array(indptr, dtype=np.int32)


def run_combine(inp, o_part, l_part, indptr):
    d = mla.make_desc(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq)
    out = torch.full((inp.batch, inp.s_q, inp.heads, 512), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((inp.batch, inp.s_q, inp.heads), 7.0, dtype=torch.float32, device="cuda")
    mla.mla_combine(d, torch.from_numpy(o_part).float().cuda(), torch.from_numpy(l_part).float().cuda(),
                    torch.from_numpy(indptr).cuda(), out, lse)
    torch.cuda.synchronize()
    return (out.float().cpu().numpy().reshape(-1, 512).astype(np.float64),
            lse.cpu().numpy().reshape(-1).astype(np.float64))


@pytest.mark.parametrize("seqlens,heads,s_q,cuts", [
    # 1, 2, 3 and 40 pieces; the 5000-key request is cut every other page
    ([3000, 700, 64, 5000], 16, 2, [[0], [0, 320], [0, 64, 128], list(range(0, 5000, 128))]),
    # full 128-head rows, uneven pieces; the last piece of request 0 holds only its last key
    ([4097, 2500, 1300], 128, 1, [[0, 1024, 4096], [0, 64, 2048], [0, 640, 1216, 1280]]),
    # causal verify of six tokens: the last piece holds the last two keys, so the
    # first four tokens see none of it (lse -inf, NaN rows in the partial)
    ([1026, 300], 64, 6, [[0, 512, 1024], [0, 256]]),
])
def test_merge_of_oracle_partials_equals_whole_range(seqlens, heads, s_q, cuts):
    inp = gen.make_inputs("x", seqlens=seqlens, heads=heads, s_q=s_q, seed=sum(seqlens) + 17)
    o_part, l_part, indptr = oracle_partials(inp, cuts)
    out_g, lse_g = run_combine(inp, o_part, l_part, indptr)
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(out_g, lse_g, out_r, lse_r, TOL_BF16)


def test_request_without_partials_and_rows_without_keys():
    """Request 1 has no partial (empty range); request 0's single partial has
    -inf rows for the tokens that see no key: those rows are zero, lse -inf."""
    inp = gen.make_inputs("x", seqlens=[2, 900], heads=8, s_q=4, seed=3)
    o_part, l_part, _ = oracle_partials(inp, [[0], [0]])
    o_part, l_part = o_part[:1], l_part[:1]            # keep request 0's partial only
    indptr = np.array([0, 1, 1], dtype=np.int32)
    out_g, lse_g = run_combine(inp, o_part, l_part, indptr)
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    R = 4 * 8
    compare(out_g[:R], lse_g[:R], out_r[:R], lse_r[:R], TOL_BF16)
    assert (out_g[R:] == 0).all() and np.isneginf(lse_g[R:]).all()
    assert np.isneginf(lse_g[:2 * 8]).all() and (out_g[:2 * 8] == 0).all()   # tokens 0, 1 see no key


def test_merge_matches_the_decode_path_on_a_full_size_shape():
    """Decode-sized rows (B=64, H=128) cut into four page-aligned ranges per
    request: the merge of the oracle's partials equals mla_decode's own result
    within the bf16 tolerances (both against the oracle)."""
    inp = gen.make_inputs("decode", batch=8)
    cuts = []
    for n in inp.seqlens.tolist():
        pages = (n + 63) // 64
        cuts.append(sorted({0, 64 * (pages // 4), 64 * (pages // 2), 64 * (3 * pages // 4)}))
    o_part, l_part, indptr = oracle_partials(inp, cuts)
    out_g, lse_g = run_combine(inp, o_part, l_part, indptr)
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(out_g, lse_g, out_r, lse_r, TOL_BF16)
