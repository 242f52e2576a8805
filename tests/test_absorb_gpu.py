"""Parity of the absorption GEMMs (mla_absorb_q, mla_project_out) with the
fp64 oracle, and of the absorbed pipeline (absorb -> decode -> project) with
standard MLA attention (latent up-projected by W_UK / W_UV, 192-wide heads).

Each GEMM output is bf16 from an fp32 accumulation of exact bf16 products, so
every element must lie within one bf16 rounding (2^-8 relative) of the fp64
product, plus a small absolute slack for the fp32 sum.  The RoPE part of the
absorbed q is a copy and must be bit-exact.
"""
import math

import numpy as np
import pytest
import torch

import mla_paged_decode_absorbed_gb300 as mla
import oracle
from tests.gpu_helpers import TOL_BF16, compare

pytestmark = pytest.mark.gpu

BF16_REL = 2.0 ** -8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    mla.library()
    torch.cuda.set_device(0)


def _bf16(g, shape, scale=1.0):
    return (torch.randn(shape, generator=g, dtype=torch.float64) * scale).to(torch.bfloat16)


def _within_bf16(gpu, ref, slack):
    gpu = gpu.to(torch.float64).numpy() if isinstance(gpu, torch.Tensor) else gpu
    err = np.abs(gpu - ref)
    bound = BF16_REL * np.abs(ref) + slack
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"error {err[worst]} > {bound[worst]} at {worst}"


@pytest.mark.parametrize("T,H", [(1, 1), (5, 16), (64, 128), (200, 3), (257, 4)])
def test_absorb_q_matches_oracle(T, H):
    g = torch.Generator().manual_seed(1000 + 7 * T + H)
    q_nope, q_rope = _bf16(g, (T, H, 128)), _bf16(g, (T, H, 64))
    w_uk = _bf16(g, (H, 512, 128), 1.0 / 8.0)
    q = torch.full((T, H, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q(q_nope.cuda(), q_rope.cuda(), w_uk.cuda(), q)
    torch.cuda.synchronize()
    ref = oracle.absorb_q(q_nope, q_rope, w_uk)
    got = q.cpu()
    _within_bf16(got[..., :512], ref[..., :512], 1e-5)
    assert torch.equal(got[..., 512:], q_rope), "the RoPE part of q must be copied bit-exactly"


@pytest.mark.parametrize("T,H", [(1, 1), (7, 16), (64, 128), (300, 2), (256, 5)])
def test_project_out_matches_oracle(T, H):
    g = torch.Generator().manual_seed(2000 + 7 * T + H)
    out = _bf16(g, (T, H, 512))
    w_uv = _bf16(g, (H, 512, 128), 1.0 / 8.0)
    o = torch.full((T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    mla.mla_project_out(out.cuda(), w_uv.cuda(), o)
    torch.cuda.synchronize()
    _within_bf16(o.cpu(), oracle.project_out(out, w_uv), 1e-5)


def test_absorbed_pipeline_equals_standard_mla():
    """absorb -> mla_decode -> project on the GPU, against standard MLA in
    fp64 on the same bf16 inputs.  Each stage is also held to its own bound
    against the oracle run on exactly what the GPU stage consumed."""
    g = torch.Generator().manual_seed(77)
    B, s_q, H = 3, 2, 16
    seqlens = [5, 130, 64]
    pages = [(s + 63) // 64 for s in seqlens]
    P = sum(pages) + 3
    perm = torch.randperm(P, generator=g)
    maxp = max(pages)
    bt = torch.full((B, maxp), -1, dtype=torch.int32)
    k = 0
    for b in range(B):
        for j in range(pages[b]):
            bt[b, j] = int(perm[k])
            k += 1
    latent = _bf16(g, (P, 64, 512))
    krope = _bf16(g, (P, 64, 64))
    kv = torch.cat([latent, krope], dim=-1).contiguous()
    w_uk = _bf16(g, (H, 512, 128), 1.0 / 8.0)
    w_uv = _bf16(g, (H, 512, 128), 1.0 / 8.0)
    T = B * s_q
    q_nope, q_rope = _bf16(g, (T, H, 128)), _bf16(g, (T, H, 64))
    scale = 1.0 / math.sqrt(192.0)
    sl = torch.tensor(seqlens, dtype=torch.int32)

    # GPU: absorb, decode, project
    q = torch.empty((T, H, 576), dtype=torch.bfloat16, device="cuda")
    mla.mla_absorb_q(q_nope.cuda(), q_rope.cuda(), w_uk.cuda(), q)
    dec = mla.MlaDecoder(B, s_q, H, P, maxp)
    out, lse = dec(q.view(B, s_q, H, 576), kv.cuda(), bt.cuda(), sl.cuda(), scale)
    o = torch.empty((T, H, 128), dtype=torch.bfloat16, device="cuda")
    mla.mla_project_out(out.view(T, H, 512), w_uv.cuda(), o)
    torch.cuda.synchronize()
    assert dec.device_error() == mla.MLA_OK

    # stage by stage against the oracle on the GPU's own intermediates
    q_g = q.cpu()
    _within_bf16(q_g[..., :512], oracle.absorb_q(q_nope, q_rope, w_uk)[..., :512], 1e-5)
    out_r, lse_r = oracle.mla_decode(q_g.view(B, s_q, H, 576), kv, bt, sl, s_q, scale)
    out_g = out.float().cpu().numpy().reshape(-1, 512).astype(np.float64)
    lse_g = lse.cpu().numpy().reshape(-1).astype(np.float64)
    compare(out_g, lse_g, out_r, lse_r, TOL_BF16)
    _within_bf16(o.cpu(), oracle.project_out(out.cpu().view(T, H, 512), w_uv), 1e-5)

    # end to end against standard attention (192-wide heads, V = c W_UV)
    lat = latent.to(torch.float64).numpy()
    kr = krope.to(torch.float64).numpy()
    wk = w_uk.to(torch.float64).numpy()
    wv = w_uv.to(torch.float64).numpy()
    qn = q_nope.to(torch.float64).numpy().reshape(B, s_q, H, 128)
    qr = q_rope.to(torch.float64).numpy().reshape(B, s_q, H, 64)
    o_g = o.float().cpu().numpy().astype(np.float64).reshape(B, s_q, H, 128)
    diffs, norms = [], []
    for b in range(B):
        rows = [int(bt[b, t // 64]) for t in range(seqlens[b])]
        c = np.stack([lat[rows[t], t % 64] for t in range(seqlens[b])])
        kro = np.stack([kr[rows[t], t % 64] for t in range(seqlens[b])])
        for i in range(s_q):
            n = seqlens[b] - s_q + i + 1
            for h in range(H):
                kk = np.concatenate([c[:n] @ wk[h], kro[:n]], axis=1)
                vv = c[:n] @ wv[h]
                s = kk @ np.concatenate([qn[b, i, h], qr[b, i, h]]) * scale
                p = np.exp(s - s.max())
                ref = (p / p.sum()) @ vv
                diffs.append(o_g[b, i, h] - ref)
                norms.append(ref)
    d, r = np.concatenate(diffs), np.concatenate(norms)
    # The stage checks above carry the precise bounds.  This one guards the
    # composition (token order, head index, weight orientation), whose
    # mistakes give O(1) relative errors; the bf16 roundings of the absorbed
    # q, P, the attention output and o stay far below these bounds.  W_UV
    # scales the output (|o| reaches ~8 here), so the max bound is relative.
    assert np.linalg.norm(d) / np.linalg.norm(r) <= 2 * TOL_BF16[1]
    assert np.abs(d).max() <= 1e-2 * np.abs(r).max()
