"""Python binding of the GB300 MLA paged-decode library (absorbed form).

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libmla_gb300.so`` (C ABI in ``include/mla.h``).  PyTorch supplies
device memory and the current stream.  There is no CPU fallback: if the
library cannot be loaded the calls raise.

Functions mirror the C entry points: ``mla_workspace_size``, ``mla_plan``,
``mla_decode_attention``, ``mla_combine_workspace``, ``mla_combine`` (merge
of caller-supplied fp32 partials), ``mla_decode``, ``mla_get_device_error``.  Each checks its tensors' dtype, shape, contiguity
and device against the descriptor before the call (``check_decode_tensors``),
since the C ABI sees only pointers.  ``MlaDecoder`` bundles a descriptor and
a cached workspace for repeated calls.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_LAUNCH = -4
MLA_ERR_DEVICE_BOUNDS = -5
MLA_ERR_DEVICE_TIMEOUT = -6
MLA_ERR_CUDA = -7
MLA_ERR_DEVICE_RANGE = -8

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_KV_FP8_E4M3_ROPE_BF16 = 2  # fp8 variant B: [P, 64, 656] token records
FP8B_RECORD = 656

PAGE, D_QK, D_V = 64, 576, 512


class MlaDesc(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("s_q", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("d_qk", ctypes.c_int32),
        ("d_v", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("max_clusters", ctypes.c_int32),
        ("plan_overhead", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 5),
    ]


class MlaWorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in ("header", "cl_first", "pre", "lse_part", "o_part", "sync", "total")]


class MlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None
_lock = threading.Lock()


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"CUDA library {LIB_PATH} is not built; run __graft_entry__.build()")
            lib = ctypes.CDLL(LIB_PATH)
            vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
            dp = ctypes.POINTER(MlaDesc)
            lib.mla_workspace_size.restype = sz
            lib.mla_workspace_size.argtypes = [dp, ctypes.c_int]
            lib.mla_num_clusters.restype = ctypes.c_int
            lib.mla_num_clusters.argtypes = [dp]
            lib.mla_plan.restype = ctypes.c_int
            lib.mla_plan.argtypes = [dp, vp, vp, sz, vp]
            lib.mla_decode_attention.restype = ctypes.c_int
            lib.mla_decode_attention.argtypes = [dp, vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, vp, sz, vp]
            lib.mla_combine_workspace.restype = ctypes.c_int
            lib.mla_combine_workspace.argtypes = [dp, vp, vp, vp, sz, vp]
            lib.mla_combine.restype = ctypes.c_int
            lib.mla_combine.argtypes = [dp, vp, vp, vp, i32, vp, vp, vp]
            lib.mla_decode.restype = ctypes.c_int
            lib.mla_decode.argtypes = [dp, vp, vp, vp, vp, vp, i32, ctypes.c_float, vp, vp, vp, sz, vp]
            lib.mla_get_device_error.restype = ctypes.c_int
            lib.mla_get_device_error.argtypes = [vp, vp]
            lib.mla_status_string.restype = ctypes.c_char_p
            lib.mla_status_string.argtypes = [ctypes.c_int]
            lib.mla_absorb_q.restype = ctypes.c_int
            lib.mla_absorb_q.argtypes = [vp, vp, vp, i32, i32, vp, vp, vp]
            lib.mla_project_out.restype = ctypes.c_int
            lib.mla_project_out.argtypes = [vp, vp, i32, i32, vp, vp, vp]
            lib.mla_get_workspace_layout.restype = ctypes.c_int
            lib.mla_get_workspace_layout.argtypes = [dp, ctypes.c_int, ctypes.POINTER(MlaWorkspaceLayout)]
            _lib = lib
    return _lib


def library():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def status_string(status: int) -> str:
    return _load().mla_status_string(int(status)).decode()


def make_desc(batch: int, s_q: int, num_heads: int, num_pages: int, max_pages_per_seq: int,
              kv_fp8: bool = False, max_clusters: int = 0, plan_overhead: int = 0,
              rope_bf16: bool = False) -> MlaDesc:
    """rope_bf16 (with kv_fp8): fp8 variant B, 656-byte token records."""
    d = MlaDesc()
    d.batch, d.s_q, d.num_heads = batch, s_q, num_heads
    d.num_pages, d.max_pages_per_seq = num_pages, max_pages_per_seq
    d.page_size, d.d_qk, d.d_v = PAGE, D_QK, D_V
    if rope_bf16 and not kv_fp8:
        raise ValueError("rope_bf16 is a layout of the fp8 cache")
    d.kv_dtype = (MLA_KV_FP8_E4M3_ROPE_BF16 if rope_bf16 else MLA_KV_FP8_E4M3) if kv_fp8 else MLA_KV_BF16
    d.max_clusters, d.plan_overhead = max_clusters, plan_overhead
    return d


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _check(status: int, what: str):
    if status != MLA_OK:
        raise MlaError(status, what)


def mla_workspace_size(desc: MlaDesc, num_sms: int = 0) -> int:
    return int(_load().mla_workspace_size(ctypes.byref(desc), int(num_sms)))


def mla_num_clusters(desc: MlaDesc) -> int:
    n = int(_load().mla_num_clusters(ctypes.byref(desc)))
    _check(n if n < 0 else MLA_OK, "mla_num_clusters")
    return n


def mla_get_workspace_layout(desc: MlaDesc, num_clusters: int) -> MlaWorkspaceLayout:
    lay = MlaWorkspaceLayout()
    _check(_load().mla_get_workspace_layout(ctypes.byref(desc), int(num_clusters), ctypes.byref(lay)),
           "mla_get_workspace_layout")
    return lay


def alloc_workspace(desc: MlaDesc, device=None) -> torch.Tensor:
    n = mla_workspace_size(desc, 0)
    if n == 0:
        raise MlaError(MLA_ERR_INVALID_ARG, "mla_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def check_decode_tensors(desc: MlaDesc, q, kv, kv_scales, block_table, seqlens, out, lse, cuda: bool = True):
    """Checks a decode call's tensors against the descriptor (dtype, shape,
    contiguity and, with ``cuda``, the device) and returns ``kv`` as the
    library reads it (an e4m3 tensor viewed as bytes).  The C ABI sees only
    pointers, so this is where a tensor too small for the descriptor is
    caught before a kernel reads past it."""
    B, sq, H = desc.batch, desc.s_q, desc.num_heads
    _expect(q, "q", torch.bfloat16, (B, sq, H, D_QK), cuda)
    if desc.kv_dtype == MLA_KV_FP8_E4M3_ROPE_BF16:
        _expect(kv, "kv", torch.uint8, (desc.num_pages, PAGE, FP8B_RECORD), cuda)
        if kv_scales is not None:
            raise ValueError("fp8 variant B keeps its scales inside the token records")
    elif desc.kv_dtype == MLA_KV_FP8_E4M3:
        if isinstance(kv, torch.Tensor) and kv.dtype == torch.float8_e4m3fn:
            kv = kv.view(torch.uint8)
        _expect(kv, "kv", torch.uint8, (desc.num_pages, PAGE, D_QK), cuda)
        _expect(kv_scales, "kv_scales", torch.float32, (desc.num_pages, PAGE, 5), cuda)
    else:
        _expect(kv, "kv", torch.bfloat16, (desc.num_pages, PAGE, D_QK), cuda)
        if kv_scales is not None:
            raise ValueError("kv_scales is only for the fp8 cache")
    _expect(block_table, "block_table", torch.int32, (B, desc.max_pages_per_seq), cuda)
    _expect(seqlens, "seqlens", torch.int32, (B,), cuda)
    _expect(out, "out", torch.bfloat16, (B, sq, H, D_V), cuda)
    _expect(lse, "lse", torch.float32, (B, sq, H), cuda)
    return kv


def _check_workspace(desc: MlaDesc, workspace, cuda: bool = True):
    _expect(workspace, "workspace", torch.uint8, None, cuda)


def mla_plan(desc: MlaDesc, seqlens: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    _expect(seqlens, "seqlens", torch.int32, (desc.batch,))
    _check_workspace(desc, workspace)
    _check(_load().mla_plan(ctypes.byref(desc), _ptr(seqlens), _ptr(workspace), workspace.numel(),
                            _stream(stream)), "mla_plan")


def mla_decode_attention(desc: MlaDesc, q, kv, kv_scales, block_table, seqlens, s_q: int, softmax_scale: float,
                         out, lse, workspace, stream=None) -> None:
    kv = check_decode_tensors(desc, q, kv, kv_scales, block_table, seqlens, out, lse)
    _check_workspace(desc, workspace)
    _check(_load().mla_decode_attention(ctypes.byref(desc), _ptr(q), _ptr(kv), _ptr(kv_scales), _ptr(block_table),
                                        _ptr(seqlens), int(s_q), float(softmax_scale), _ptr(out), _ptr(lse),
                                        _ptr(workspace), workspace.numel(), _stream(stream)),
           "mla_decode_attention")


def mla_combine_workspace(desc: MlaDesc, out, lse, workspace, stream=None) -> None:
    """Step 3 of mla_decode: merges the split pieces a previous
    mla_decode_attention left in ``workspace``."""
    _expect(out, "out", torch.bfloat16, (desc.batch, desc.s_q, desc.num_heads, D_V))
    _expect(lse, "lse", torch.float32, (desc.batch, desc.s_q, desc.num_heads))
    _check_workspace(desc, workspace)
    _check(_load().mla_combine_workspace(ctypes.byref(desc), _ptr(out), _ptr(lse), _ptr(workspace),
                                         workspace.numel(), _stream(stream)), "mla_combine_workspace")


def mla_combine(desc: MlaDesc, o_part, lse_part, split_indptr, out, lse, stream=None) -> None:
    """LSE merge of caller-supplied split-KV partials: ``o_part`` fp32
    [num_partials, s_q*H, 512], ``lse_part`` fp32 [num_partials, s_q*H],
    ``split_indptr`` int32 [B+1] (request b owns partials
    split_indptr[b]..split_indptr[b+1]-1), into ``out`` / ``lse``."""
    R = desc.s_q * desc.num_heads
    n = int(o_part.shape[0]) if isinstance(o_part, torch.Tensor) else -1
    _expect(o_part, "o_part", torch.float32, (n, R, D_V))
    _expect(lse_part, "lse_part", torch.float32, (n, R))
    _expect(split_indptr, "split_indptr", torch.int32, (desc.batch + 1,))
    _expect(out, "out", torch.bfloat16, (desc.batch, desc.s_q, desc.num_heads, D_V))
    _expect(lse, "lse", torch.float32, (desc.batch, desc.s_q, desc.num_heads))
    _check(_load().mla_combine(ctypes.byref(desc), _ptr(o_part) if n > 0 else None,
                               _ptr(lse_part) if n > 0 else None, _ptr(split_indptr), n, _ptr(out), _ptr(lse),
                               _stream(stream)), "mla_combine")


def mla_decode(desc: MlaDesc, q, kv, kv_scales, block_table, seqlens, s_q: int, softmax_scale: float, out, lse,
               workspace, stream=None) -> None:
    """The C ``mla_decode`` on caller-provided tensors (checked against the descriptor)."""
    kv = check_decode_tensors(desc, q, kv, kv_scales, block_table, seqlens, out, lse)
    _check_workspace(desc, workspace)
    _check(_load().mla_decode(ctypes.byref(desc), _ptr(q), _ptr(kv), _ptr(kv_scales), _ptr(block_table),
                              _ptr(seqlens), int(s_q), float(softmax_scale), _ptr(out), _ptr(lse),
                              _ptr(workspace), workspace.numel(), _stream(stream)), "mla_decode")


def mla_absorb_q(q_nope, q_rope, w_uk, q, workspace=None, stream=None) -> None:
    """q[t, h] = [W_UK[h] @ q_nope[t, h] ; q_rope[t, h]] (bf16 tensors:
    q_nope [T, H, 128], q_rope [T, H, 64], w_uk [H, 512, 128], q [T, H, 576])."""
    T, H = int(q_nope.shape[0]), int(q_nope.shape[1])
    _expect(q_nope, "q_nope", torch.bfloat16, (T, H, 128))
    _expect(q_rope, "q_rope", torch.bfloat16, (T, H, 64))
    _expect(w_uk, "w_uk", torch.bfloat16, (H, 512, 128))
    _expect(q, "q", torch.bfloat16, (T, H, 576))
    _check(_load().mla_absorb_q(_ptr(q_nope), _ptr(q_rope), _ptr(w_uk), T, H, _ptr(q), _ptr(workspace),
                                _stream(stream)), "mla_absorb_q")


def mla_project_out(out, w_uv, o, workspace=None, stream=None) -> None:
    """o[t, h] = W_UV[h]^T @ out[t, h] (bf16 tensors: out [T, H, 512],
    w_uv [H, 512, 128], o [T, H, 128])."""
    T, H = int(out.shape[0]), int(out.shape[1])
    _expect(out, "out", torch.bfloat16, (T, H, 512))
    _expect(w_uv, "w_uv", torch.bfloat16, (H, 512, 128))
    _expect(o, "o", torch.bfloat16, (T, H, 128))
    _check(_load().mla_project_out(_ptr(out), _ptr(w_uv), T, H, _ptr(o), _ptr(workspace), _stream(stream)),
           "mla_project_out")


def mla_get_device_error(workspace: torch.Tensor, stream=None) -> int:
    return int(_load().mla_get_device_error(_ptr(workspace), _stream(stream)))


def _expect(t: torch.Tensor, name: str, dtype, shape=None, cuda: bool = True):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


class MlaDecoder:
    """Descriptor + workspace for repeated decode calls on one configuration."""

    def __init__(self, batch: int, s_q: int, num_heads: int, num_pages: int, max_pages_per_seq: int,
                 kv_fp8: bool = False, max_clusters: int = 0, plan_overhead: int = 0, device=None,
                 rope_bf16: bool = False):
        self.desc = make_desc(batch, s_q, num_heads, num_pages, max_pages_per_seq, kv_fp8, max_clusters,
                              plan_overhead, rope_bf16)
        self.device = torch.device(device or "cuda")
        with torch.cuda.device(self.device):
            self.workspace = alloc_workspace(self.desc, self.device)
            self.num_clusters = mla_num_clusters(self.desc)

    def __call__(self, q: torch.Tensor, kv: torch.Tensor, block_table: torch.Tensor, seqlens: torch.Tensor,
                 softmax_scale: float, kv_scales: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                 stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
        d = self.desc
        B, sq, H = d.batch, d.s_q, d.num_heads
        dev = q.device if isinstance(q, torch.Tensor) else self.device
        if out is None:
            out = torch.empty((B, sq, H, D_V), dtype=torch.bfloat16, device=dev)
        if lse is None:
            lse = torch.empty((B, sq, H), dtype=torch.float32, device=dev)
        mla_decode(d, q, kv, kv_scales, block_table, seqlens, sq, softmax_scale, out, lse, self.workspace, stream)
        return out, lse

    def device_error(self, stream=None) -> int:
        return mla_get_device_error(self.workspace, stream)


def noalloc_function():
    """The C ``mla_decode_noalloc`` with its argument types declared."""
    fn = _load().mla_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(MlaDesc)] + [ctypes.c_void_p] * 5 + [ctypes.c_int32, ctypes.c_float,
                                                                       ctypes.c_void_p, ctypes.c_void_p,
                                                                       ctypes.c_int, ctypes.c_void_p]
    return fn


def mla_noalloc_get_device_error(stream=None) -> int:
    """Device error status of the last mla_decode_noalloc on this device
    (synchronises the stream)."""
    fn = _load().mla_noalloc_get_device_error
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p]
    return int(fn(_stream(stream)))


def mla_decode_noalloc(desc: MlaDesc, q, kv, kv_scales, block_table, seqlens, s_q: int, softmax_scale: float,
                       out, lse, check_device_error: bool = False, stream=None) -> int:
    """Raw call of the C ``mla_decode_noalloc`` (scratch inside the library,
    no workspace argument, no device allocation).  Returns the status when
    ``check_device_error`` is set (the call then synchronises the stream)."""
    kv = check_decode_tensors(desc, q, kv, kv_scales, block_table, seqlens, out, lse)
    st = noalloc_function()(ctypes.byref(desc), _ptr(q), _ptr(kv), _ptr(kv_scales), _ptr(block_table), _ptr(seqlens), int(s_q),
            float(softmax_scale), _ptr(out), _ptr(lse), 1 if check_device_error else 0, _stream(stream))
    if st not in (MLA_OK, MLA_ERR_DEVICE_BOUNDS, MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_RANGE):
        raise MlaError(st, "mla_decode_noalloc")
    return st
