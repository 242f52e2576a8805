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


def compare(out_g, lse_g, out_r, lse_r, tol):
    """Element-wise comparison under the stated tolerances (max abs, relative
    L2, lse abs on every row); returns the measured errors."""
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
    assert max_abs <= max_abs_tol, f"max abs error {max_abs} > {max_abs_tol}"
    assert rel <= rel_tol, f"relative L2 error {rel} > {rel_tol}"
    assert lse_err <= lse_tol, f"lse error {lse_err} > {lse_tol}"
    return max_abs, rel, lse_err
