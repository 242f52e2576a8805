"""CPU oracle for MLA paged decode (absorbed form).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library in
``mla_paged_decode_absorbed_gb300`` never imports, links or calls it, and the
two share no code: the oracle is plain fp64 C (``mla_oracle.c``) compiled with
gcc, loaded here with ctypes.

Pinned by ``tests/test_oracle_pins.py`` against: the non-absorbed MLA form
(which also pins ``absorb_q`` and ``project_out``, the absorption GEMMs),
closed forms (single key, identical keys, a hand-derived two-key example),
softmax rows summing to one, the split/LSE-merge identity, the batch-extension
equivalence of causal verify, a dense library softmax, and torch's bf16/e4m3
decoders.  ``plan_ref`` is the reference for the split planner's integer plan.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "_liboracle_mla.so")
_lock = threading.Lock()
_lib = None

KV_BF16, KV_FP8, KV_F64, KV_FP8B = 0, 1, 2, 3  # KV_FP8B: fp8 variant B, [P, 64, 656] token records


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_mla_decode.restype = ctypes.c_int
            lib.oracle_mla_decode.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
            lib.oracle_bf16_to_f64.restype = ctypes.c_double
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_e4m3_to_f64.restype = ctypes.c_double
            lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.restype = None
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads the next oracle calls use (a timing knob; results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def bf16_to_f64(code: int) -> float:
    return float(_load().oracle_bf16_to_f64(code))


def e4m3_to_f64(code: int) -> float:
    return float(_load().oracle_e4m3_to_f64(code))


def _np(t, dtype):
    """Contiguous numpy array of ``t`` (torch tensor or array) as ``dtype``;
    same-size integer types are reinterpreted, anything else converted."""
    import torch
    if isinstance(t, torch.Tensor):
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        elif t.dtype == torch.float8_e4m3fn:
            t = t.view(torch.uint8)
        t = t.numpy()
    a = np.asarray(t)
    dt = np.dtype(dtype)
    if a.dtype != dt:
        if a.dtype.itemsize == dt.itemsize and a.dtype.kind in "iu" and dt.kind in "iu":
            a = a.view(dt)
        else:
            a = a.astype(dt)
    return np.ascontiguousarray(a)


def mla_decode(q, kv, block_table, seqlens, s_q: int, softmax_scale: float, *, kv_scales=None,
               kv_dtype: int = KV_BF16, rows=None, return_p: bool = False
               ) -> Tuple[np.ndarray, np.ndarray] | Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Reference out [n, 512] and lse [n] (float64) for the flat query rows
    ``rows`` (b*s_q*H + i*H + h; None = all rows in order).

    q: [B, s_q, H, 576] bf16 (or float64 when kv_dtype == KV_F64)
    kv: [P, 64, 576] bf16 / uint8 e4m3 codes / float64; kv_scales: [P, 64, 5] fp32 for fp8.
    """
    lib = _load()
    qshape = tuple(q.shape)
    B, sq, H = int(qshape[0]), int(qshape[1]), int(qshape[2])
    if sq != s_q:
        raise ValueError("q.shape[1] must equal s_q")
    if kv_dtype == KV_F64:
        qa = _np(q, np.float64)
        kva = _np(kv, np.float64)
    else:
        qa = _np(q, np.uint16)
        kva = _np(kv, np.uint16 if kv_dtype == KV_BF16 else np.uint8)
        if kv_dtype == KV_FP8B and (kva.ndim != 3 or kva.shape[2] != 656):
            raise ValueError("fp8 variant B cache must be uint8 [P, 64, 656]")
    sca = _np(kv_scales, np.float32) if kv_scales is not None else None
    bta = _np(block_table, np.int32)
    sla = _np(seqlens, np.int32)
    P = int(kva.shape[0])
    maxp = int(bta.shape[1])
    if rows is None:
        n = B * s_q * H
        rows_a = None
    else:
        rows_a = _np(rows, np.int64)
        n = int(rows_a.size)
    out = np.zeros((n, 512), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    pbuf = None
    p_stride = 0
    if return_p:
        p_stride = max(1, int(sla.max()))
        pbuf = np.zeros((n, p_stride), dtype=np.float64)
    rc = lib.oracle_mla_decode(
        qa.ctypes.data, kva.ctypes.data, sca.ctypes.data if sca is not None else None, kv_dtype,
        bta.ctypes.data, sla.ctypes.data, B, s_q, H, P, maxp, float(softmax_scale),
        rows_a.ctypes.data if rows_a is not None else None, n,
        out.ctypes.data, lse.ctypes.data, pbuf.ctypes.data if pbuf is not None else None, p_stride)
    if rc != 0:
        raise RuntimeError(f"oracle_mla_decode failed with status {rc}")
    if return_p:
        return out, lse, pbuf
    return out, lse


def mla_decode_inputs(inp, rows=None, return_p: bool = False):
    """Oracle on a ``workloads.gen.Inputs`` bundle."""
    dt = (KV_FP8B if getattr(inp, "rope_bf16", False) else KV_FP8) if inp.kv_fp8 else KV_BF16
    return mla_decode(inp.q, inp.kv, inp.block_table, inp.seqlens, inp.s_q, inp.softmax_scale,
                      kv_scales=inp.kv_scales, kv_dtype=dt, rows=rows, return_p=return_p)


# ------------------------------------------------------- absorption GEMMs
# Matrix absorption for MLA (best-practice digest §2.4.3, the
# `--mla_use_matrix_absorption` switch; the algebra is standard MLA): the key
# up-projection W_UK is folded into the query and the value up-projection W_UV
# is applied to the latent output.  Plain fp64 definitions.

def _f64(t) -> np.ndarray:
    """Values of ``t`` (torch tensor of any float dtype, or array) in fp64."""
    import torch
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def absorb_q(q_nope, q_rope, w_uk) -> np.ndarray:
    """q[t, h] = [W_UK[h] @ q_nope[t, h] ; q_rope[t, h]]  (fp64 [T, H, 576]).

    q_nope [T, H, 128], q_rope [T, H, 64], w_uk [H, 512, 128] (any float or
    bf16 tensor/array; bf16 values are taken exactly)."""
    qn, qr, w = _f64(q_nope), _f64(q_rope), _f64(w_uk)
    lat = np.einsum("hcd,thd->thc", w, qn)
    return np.concatenate([lat, qr], axis=-1)


def project_out(out_latent, w_uv) -> np.ndarray:
    """o[t, h] = W_UV[h]^T @ out_latent[t, h]  (fp64 [T, H, 128]).

    out_latent [T, H, 512], w_uv [H, 512, 128]."""
    o, w = _f64(out_latent), _f64(w_uv)
    return np.einsum("hcd,thc->thd", w, o)
