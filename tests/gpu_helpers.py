"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and compare it with the oracle under the stated tolerances."""
from __future__ import annotations

import numpy as np
import torch

import mla_paged_decode_absorbed_gb300 as mla

# max abs error, relative L2 error, lse abs error
TOL_BF16 = (2e-2, 5e-3, 1e-3)
TOL_FP8 = (6e-2, 2e-2, 1e-3)


def to_device(inp, device="cuda"):
    q = inp.q.to(device)
    kv = inp.kv.to(device)
    sc = inp.kv_scales.to(device) if inp.kv_scales is not None else None
    bt = inp.block_table.to(device)
    sl = inp.seqlens.to(device)
    return q, kv, sc, bt, sl


def run_gpu(inp, max_clusters: int = 0, plan_overhead: int = 0, decoder=None, tensors=None):
    """out [rows, 512] float64, lse [rows] float64, device status, decoder."""
    dec = decoder or mla.MlaDecoder(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq,
                                    kv_fp8=inp.kv_fp8, max_clusters=max_clusters, plan_overhead=plan_overhead,
                                    rope_bf16=inp.rope_bf16)
    q, kv, sc, bt, sl = tensors or to_device(inp)
    out, lse = dec(q, kv, bt, sl, inp.softmax_scale, kv_scales=sc)
    torch.cuda.synchronize()
    status = dec.device_error()
    o = out.float().cpu().numpy().reshape(-1, 512).astype(np.float64)
    l = lse.cpu().numpy().reshape(-1).astype(np.float64)
    return o, l, status, dec


def fp16_k_lse_shift(inp, rows=None):
    """Per row, how far the oracle's lse moves when the dequantised fp8 cache
    (e4m3 x scale) is rounded to fp16 before use -- the rounding the fp8
    variant's 16-bit tensor-core operands cannot avoid.  Computed on the CPU
    by running the oracle twice on fp64 caches built here with torch (the
    exact product and its fp16 rounding); nothing comes from the CUDA path."""
    import oracle
    if getattr(inp, "rope_bf16", False):  # variant B records
        rec = inp.kv
        lat = rec[:, :, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
        sc4 = rec[:, :, 512:528].contiguous().view(torch.float32).to(torch.float64)
        rope = rec[:, :, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
        exact = torch.cat([lat * sc4.repeat_interleave(128, dim=-1), rope], dim=-1)
    else:
        codes = inp.kv.view(torch.float8_e4m3fn).to(torch.float64)
        sc = inp.kv_scales.to(torch.float64)
        grp = torch.tensor([0] * 128 + [1] * 128 + [2] * 128 + [3] * 128 + [4] * 64)
        exact = codes * sc[:, :, grp]
    rounded = exact.to(torch.float16).to(torch.float64)
    q = inp.q.to(torch.float64)
    _, l_ex = oracle.mla_decode(q, exact, inp.block_table, inp.seqlens, inp.s_q, inp.softmax_scale,
                                kv_dtype=oracle.KV_F64, rows=rows)
    _, l_16 = oracle.mla_decode(q, rounded, inp.block_table, inp.seqlens, inp.s_q, inp.softmax_scale,
                                kv_dtype=oracle.KV_F64, rows=rows)
    l_16, l_ex = np.asarray(l_16), np.asarray(l_ex)
    fin = np.isfinite(l_16) & np.isfinite(l_ex)  # rows with no visible key have lse = -inf
    d = np.zeros_like(l_ex)
    d[fin] = np.abs(l_16[fin] - l_ex[fin])
    return d


def compare(out_g, lse_g, out_r, lse_r, tol, lse_extra=None):
    """Element-wise comparison; returns the measured errors.  `lse_extra`
    (per row) widens the lse bound by an error the arithmetic cannot avoid
    (see fp16_k_lse_shift)."""
    max_abs_tol, rel_tol, lse_tol = tol
    assert out_g.shape == out_r.shape and lse_g.shape == lse_r.shape
    assert np.isfinite(out_g).all(), "GPU output has NaN/Inf"
    empty = ~np.isfinite(lse_r)
    assert np.isneginf(lse_r[empty]).all()
    assert np.isneginf(lse_g[empty]).all(), "rows with no visible key must have lse = -inf"
    assert (out_g[empty] == 0).all(), "rows with no visible key must be zero"
    full = ~empty
    if not full.any():
        return 0.0, 0.0, 0.0
    assert np.isfinite(lse_g[full]).all()
    d = out_g[full] - out_r[full]
    max_abs = float(np.abs(d).max())
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(out_r[full]), 1e-30))
    lse_d = np.abs(lse_g[full] - lse_r[full])
    lse_err = float(lse_d.max())
    bound = lse_tol + (np.asarray(lse_extra)[full] if lse_extra is not None else 0.0)
    assert max_abs <= max_abs_tol, f"max abs error {max_abs} > {max_abs_tol}"
    assert rel <= rel_tol, f"relative L2 error {rel} > {rel_tol}"
    worst = int(np.argmax(lse_d - bound))
    assert (lse_d <= bound).all(), f"lse error {float(lse_d[worst])} > {float(np.broadcast_to(bound, lse_d.shape)[worst])}"
    return max_abs, rel, lse_err
