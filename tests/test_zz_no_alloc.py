"""mla_decode_noalloc: the decode step for callers that cannot allocate device
memory at call time (serving loops or plugin hosts that reserve all memory up
front; C callers that own only their inputs and outputs).  Its scratch is a
fixed array inside the library, so this test calls it through the C ABI twice
in a row, on different inputs, and checks each result against the fp64 oracle
and against mla_decode with a caller-provided workspace, under the parity
tolerances.  A device error of a call made without check_device_error is read
back through mla_noalloc_get_device_error.  It runs last (file name) so a
failure here never hides the other tests, and it passes both alone in a fresh
process and after the rest of the suite."""
import ctypes

import numpy as np
import pytest
import torch

import mla_paged_decode_absorbed_gb300 as mla
import oracle
from workloads import gen
from tests.gpu_helpers import TOL_BF16, TOL_FP8, compare, to_device

pytestmark = pytest.mark.gpu


def _both(inp, max_clusters=0):
    q, kv, sc, bt, sl = to_device(inp)
    d = mla.make_desc(inp.batch, inp.s_q, inp.heads, inp.num_pages, inp.max_pages_per_seq, kv_fp8=inp.kv_fp8,
                      max_clusters=max_clusters)
    shape_o = (inp.batch, inp.s_q, inp.heads, 512)
    shape_l = (inp.batch, inp.s_q, inp.heads)
    ws = mla.alloc_workspace(d)
    o_ref = torch.empty(shape_o, dtype=torch.bfloat16, device="cuda")
    l_ref = torch.empty(shape_l, dtype=torch.float32, device="cuda")
    mla.mla_decode(d, q, kv, sc, bt, sl, inp.s_q, inp.softmax_scale, o_ref, l_ref, ws)
    o = torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda")
    l = torch.full(shape_l, float("nan"), dtype=torch.float32, device="cuda")
    st = mla.mla_decode_noalloc(d, q, kv, sc, bt, sl, inp.s_q, inp.softmax_scale, o, l, check_device_error=True)
    assert st == mla.MLA_OK, mla.status_string(st)
    torch.cuda.synchronize()
    assert mla.mla_get_device_error(ws) == mla.MLA_OK
    f = lambda t: t.float().cpu().numpy().reshape(-1, 512).astype(np.float64)
    g = lambda t: t.cpu().numpy().reshape(-1).astype(np.float64)
    tol = TOL_FP8 if inp.kv_fp8 else TOL_BF16
    out_r, lse_r = oracle.mla_decode_inputs(inp)
    compare(f(o), g(l), out_r, lse_r, tol)
    compare(f(o), g(l), f(o_ref), g(l_ref), tol)


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.fail("gpu test needs a CUDA device")
    torch.cuda.set_device(0)
    # first call: many split requests, so the partials in the library's scratch are used
    _both(gen.make_inputs("x", seqlens=[3000, 64, 1, 2500, 130, 900], heads=128, s_q=2, seed=41), max_clusters=7)
    # second call right after, different shapes and cache type, default clusters
    _both(gen.make_inputs("x", seqlens=[37, 4096, 700], heads=16, s_q=1, kv_fp8=True, seed=42))


def test_noalloc_device_error_is_read_back_without_syncing_in_the_call():
    """A page id outside the pool, run without check_device_error: the call
    returns at once, mla_noalloc_get_device_error reports the bounds error,
    and the next good call clears it."""
    if not torch.cuda.is_available():
        pytest.fail("gpu test needs a CUDA device")
    inp = gen.make_inputs("x", seqlens=[300, 50], heads=16, s_q=1, seed=4)
    good = inp.block_table.clone()
    inp.block_table[0, 2] = inp.num_pages + 5
    q, kv, sc, bt, sl = to_device(inp)
    d = mla.make_desc(inp.batch, 1, 16, inp.num_pages, inp.max_pages_per_seq)
    o = torch.empty((inp.batch, 1, 16, 512), dtype=torch.bfloat16, device="cuda")
    l = torch.empty((inp.batch, 1, 16), dtype=torch.float32, device="cuda")
    assert mla.mla_decode_noalloc(d, q, kv, sc, bt, sl, 1, inp.softmax_scale, o, l) == mla.MLA_OK
    assert mla.mla_noalloc_get_device_error() == mla.MLA_ERR_DEVICE_BOUNDS
    bt.copy_(good)
    assert mla.mla_decode_noalloc(d, q, kv, sc, bt, sl, 1, inp.softmax_scale, o, l) == mla.MLA_OK
    assert mla.mla_noalloc_get_device_error() == mla.MLA_OK


def test_noalloc_rejects_what_the_scratch_cannot_hold():
    d = mla.make_desc(65536, 16, 1024, 10, 1)     # 8,388,608 (row block, request) units
    st = mla.noalloc_function()(ctypes.byref(d), 256, 256, None, 256, 256, 16, 0.07, 256, 256, 0, None)
    assert st == mla.MLA_ERR_WORKSPACE
