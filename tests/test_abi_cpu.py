"""Host-side checks that need no GPU: the C ABI library builds, loads and
exports every symbol include/mla.h declares; host validation returns the
documented status codes without touching the device; and the reference split
plan has the properties the kernels rely on."""
import ctypes
import os
import random
import re
import subprocess

import pytest

import mla_paged_decode_absorbed_gb300 as mla
from mla_paged_decode_absorbed_gb300 import build as mla_build
from oracle import plan_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def lib():
    mla_build.build()
    return mla.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*(mla_[a-z_]+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for need in ("mla_decode", "mla_plan", "mla_decode_attention", "mla_combine", "mla_combine_workspace",
                 "mla_workspace_size",
                 "mla_get_device_error", "mla_status_string", "mla_num_clusters", "mla_get_workspace_layout"):
        assert need in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", mla.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def _desc(**kw):
    base = dict(batch=2, s_q=1, num_heads=16, num_pages=4, max_pages_per_seq=3)
    base.update(kw)
    return mla.make_desc(**base)


def test_workspace_size_is_host_only(lib):
    d = _desc()
    n = mla.mla_workspace_size(d, 152)
    lay = mla.mla_get_workspace_layout(d, 76)
    assert n == lay.total and n % 256 == 0
    assert lay.o_part >= lay.lse_part >= lay.sync >= lay.pre >= lay.cl_first >= lay.header
    assert lay.lse_part - lay.sync >= 3 * 76 * 4
    assert lay.total - lay.o_part >= 2 * 76 * 128 * 512 * 2
    # capping clusters shrinks the partial buffers
    assert mla.mla_workspace_size(_desc(max_clusters=4), 152) < n


@pytest.mark.parametrize("field,value,status", [
    ("page_size", 32, mla.MLA_ERR_UNSUPPORTED),
    ("d_qk", 512, mla.MLA_ERR_UNSUPPORTED),
    ("d_v", 576, mla.MLA_ERR_UNSUPPORTED),
    ("kv_dtype", 7, mla.MLA_ERR_UNSUPPORTED),
    ("batch", 0, mla.MLA_ERR_INVALID_ARG),
    ("s_q", 0, mla.MLA_ERR_INVALID_ARG),
    ("s_q", 17, mla.MLA_ERR_INVALID_ARG),
    ("num_heads", 0, mla.MLA_ERR_INVALID_ARG),
    ("num_pages", 0, mla.MLA_ERR_INVALID_ARG),
    ("max_clusters", -1, mla.MLA_ERR_INVALID_ARG),
])
def test_bad_descriptor_is_rejected_before_any_launch(lib, field, value, status):
    d = _desc()
    setattr(d, field, value)
    assert lib.mla_workspace_size(ctypes.byref(d), 152) == 0
    fake = 1 << 20  # never dereferenced: validation fails first
    rc = lib.mla_decode(ctypes.byref(d), fake, fake, None, fake, fake, d.s_q, 0.07, fake, fake, fake, 1 << 30, None)
    assert rc == status


def test_reserved_fields_must_be_zero(lib):
    d = _desc()
    d.reserved[2] = 1
    assert lib.mla_decode(ctypes.byref(d), 256, 256, None, 256, 256, 1, 0.07, 256, 256, 256, 1 << 30, None) \
        == mla.MLA_ERR_INVALID_ARG


def test_pointer_and_scalar_validation(lib):
    d = _desc()
    ok = 1 << 20
    args = dict(q=ok, kv=ok, sc=None, bt=ok, sl=ok, s_q=1, scale=0.07, out=ok, lse=ok, ws=ok)

    def call(**kw):
        a = dict(args)
        a.update(kw)
        return lib.mla_decode(ctypes.byref(d), a["q"], a["kv"], a["sc"], a["bt"], a["sl"], a["s_q"], a["scale"],
                              a["out"], a["lse"], a["ws"], 1 << 30, None)

    assert call(q=None) == mla.MLA_ERR_INVALID_ARG
    assert call(q=ok + 8) == mla.MLA_ERR_INVALID_ARG          # q must be 16-byte aligned
    assert call(kv=ok + 2) == mla.MLA_ERR_INVALID_ARG
    assert call(lse=ok + 2) == mla.MLA_ERR_INVALID_ARG
    assert call(sc=ok) == mla.MLA_ERR_INVALID_ARG              # scales only with the fp8 cache
    assert call(s_q=2) == mla.MLA_ERR_INVALID_ARG              # must match the descriptor
    assert call(scale=0.0) == mla.MLA_ERR_INVALID_ARG
    assert call(scale=float("nan")) == mla.MLA_ERR_INVALID_ARG
    assert call(ws=None) == mla.MLA_ERR_WORKSPACE
    assert call(ws=ok + 16) == mla.MLA_ERR_WORKSPACE           # workspace must be 256-byte aligned
    d8 = _desc(kv_fp8=True)
    assert lib.mla_decode(ctypes.byref(d8), ok, ok, None, ok, ok, 1, 0.07, ok, ok, ok, 1 << 30, None) \
        == mla.MLA_ERR_INVALID_ARG                             # fp8 needs scales
    for code in range(-8, 1):
        assert lib.mla_status_string(code).decode() != "unknown status"


def test_combine_of_caller_partials_validates_before_any_launch(lib):
    d = _desc()
    ok = 1 << 20
    call = lambda o, l, ip, n, out, lse: lib.mla_combine(ctypes.byref(d), o, l, ip, n, out, lse, None)
    assert call(ok, ok, ok, -1, ok, ok) == mla.MLA_ERR_INVALID_ARG        # negative partial count
    assert call(ok, ok, None, 4, ok, ok) == mla.MLA_ERR_INVALID_ARG       # no split_indptr
    assert call(None, ok, ok, 4, ok, ok) == mla.MLA_ERR_INVALID_ARG       # partials without o_part
    assert call(ok + 8, ok, ok, 4, ok, ok) == mla.MLA_ERR_INVALID_ARG     # o_part must be 16-byte aligned
    assert call(ok, ok + 2, ok, 4, ok, ok) == mla.MLA_ERR_INVALID_ARG
    assert call(ok, ok, ok, 4, ok + 8, ok) == mla.MLA_ERR_INVALID_ARG     # out must be 16-byte aligned
    assert call(ok, ok, ok, 4, ok, None) == mla.MLA_ERR_INVALID_ARG
    bad = _desc()
    bad.page_size = 32
    assert lib.mla_combine(ctypes.byref(bad), ok, ok, ok, 4, ok, ok, None) == mla.MLA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ plan properties
def _check_plan(plan):
    covered = {}
    slots = set()
    for c in range(plan.G):
        for p in plan.pieces(c):
            if plan.tiles[p.unit] == 0:
                covered.setdefault(p.unit, []).append(("empty", c))
                continue
            assert 0 <= p.page_lo < p.page_hi <= plan.tiles[p.unit]
            covered.setdefault(p.unit, []).append((p.page_lo, p.page_hi, c, p.split, p.slot))
            if p.split:
                assert p.slot not in slots
                assert p.slot in (2 * c, 2 * c + 1)
                slots.add(p.slot)
    combined = {}
    for c in range(plan.G):
        r = plan.combine_unit(c)
        if r is not None:
            u, pieces = r
            assert u not in combined
            combined[u] = pieces
    for u in range(plan.units):
        segs = covered.get(u, [])
        if plan.tiles[u] == 0:
            assert len(segs) == 1
            continue
        segs.sort()
        assert segs[0][0] == 0 and segs[-1][1] == plan.tiles[u]
        for a, b in zip(segs, segs[1:]):
            assert a[1] == b[0]
        if len(segs) == 1:
            assert not segs[0][3] and u not in combined
        else:
            assert all(s[3] for s in segs)
            assert sorted((s[2], s[4]) for s in segs) == sorted(combined[u])


@pytest.mark.parametrize("seed", range(12))
def test_reference_plan_covers_every_page_once(seed):
    rng = random.Random(seed)
    B = rng.randint(1, 40)
    s_q = rng.choice([1, 1, 2, 3, 5])
    H = rng.choice([16, 20, 64, 128, 256])
    maxp = rng.randint(1, 80)
    seqlens = [rng.choice([0, 1, 63, 64, 65, rng.randint(0, maxp * 64)]) for _ in range(B)]
    G = rng.randint(1, 80)
    ovh = rng.choice([1, 2, 4])
    _check_plan(plan_ref.make_plan(seqlens, s_q, H, maxp, G, ovh))


def test_reference_plan_runs_row_blocks_in_lockstep():
    """With several row blocks and at least as many clusters, cluster
    r * Gl + g covers the same stretch of pages of the same requests for
    every row block r (whose units have equal page counts here), so the
    row blocks of a request read each page at about the same time; the
    clusters past n_rb * Gl get nothing."""
    for s_q, H, G in ((2, 128, 76), (6, 128, 76), (2, 128, 9), (3, 64, 20)):
        seqlens = [4096, 2048, 640, 3000 - 3000 % 64, 64]
        plan = plan_ref.make_plan(seqlens, s_q, H, 64, G, 2)
        n_rb = plan.n_rb
        assert n_rb > 1
        gl = G // n_rb
        for r in range(n_rb):
            assert plan.pre[r * plan.B] == r * gl * plan.W
        for g in range(gl):
            views = []
            for r in range(n_rb):
                views.append([(p.b, p.page_lo, p.page_hi, p.split) for p in plan.pieces(r * gl + g)])
            assert all(v == views[0] for v in views), (s_q, H, G, g, views)
        for c in range(n_rb * gl, G):
            assert plan.pieces(c) == []
        _check_plan(plan)


def test_reference_plan_on_named_workloads():
    from workloads import gen
    for name in ("tiny", "decode", "long"):
        inp = gen.make_inputs(name) if name == "tiny" else None
        if inp is None:
            import torch
            g = torch.Generator("cpu").manual_seed(gen.workload_spec(name).seed)
            sl = gen._seqlens_for(name, gen.workload_spec(name).batch, g).tolist()
            maxp = max((s + 63) // 64 for s in sl)
            plan = plan_ref.make_plan(sl, 1, 128, maxp, 76, plan_ref.DEFAULT_OVERHEAD)
        else:
            plan = plan_ref.make_plan(inp.seqlens.tolist(), 1, 16, inp.max_pages_per_seq, 76, plan_ref.DEFAULT_OVERHEAD)
        _check_plan(plan)


def test_absorption_entry_points_reject_bad_arguments_without_a_gpu(lib):
    """Host validation of mla_absorb_q / mla_project_out returns
    MLA_ERR_INVALID_ARG and launches nothing (no device memory is touched:
    the pointers below are never dereferenced)."""
    A = 1 << 20  # a 16-byte aligned fake address
    bad = mla.MLA_ERR_INVALID_ARG
    assert lib.mla_absorb_q(A, A, A, 0, 4, A, None, None) == bad          # no tokens
    assert lib.mla_absorb_q(A, A, A, 3, 0, A, None, None) == bad          # no heads
    assert lib.mla_absorb_q(A, A, A, 3, 2000, A, None, None) == bad       # too many heads
    assert lib.mla_absorb_q(None, A, A, 3, 4, A, None, None) == bad       # NULL input
    assert lib.mla_absorb_q(A + 8, A, A, 3, 4, A, None, None) == bad      # misaligned q_nope
    assert lib.mla_absorb_q(A, A, A, 3, 4, A, A + 16, None) == bad        # workspace not 256-aligned
    assert lib.mla_project_out(A, A, 0, 4, A, None, None) == bad
    assert lib.mla_project_out(A, None, 3, 4, A, None, None) == bad
    assert lib.mla_project_out(A, A, 3, 4, A + 2, None, None) == bad


def test_fp8_variant_b_descriptor_and_arguments(lib):
    """fp8 variant B (656-byte records, scales inside): a valid descriptor
    sizes a workspace like the other fp8 layout, kv_scales must be NULL, and
    the binding refuses the layout without the fp8 cache."""
    d = _desc(kv_fp8=True, rope_bf16=True)
    assert d.kv_dtype == mla.MLA_KV_FP8_E4M3_ROPE_BF16
    assert mla.mla_workspace_size(d, 152) == mla.mla_workspace_size(_desc(kv_fp8=True), 152) > 0
    ok = 1 << 20
    assert lib.mla_decode(ctypes.byref(d), ok, ok, ok, ok, ok, 1, 0.07, ok, ok, ok, 1 << 30, None) \
        == mla.MLA_ERR_INVALID_ARG                             # the scales live in the records
    assert lib.mla_decode(ctypes.byref(d), ok, ok + 8, None, ok, ok, 1, 0.07, ok, ok, ok, 1 << 30, None) \
        == mla.MLA_ERR_INVALID_ARG                             # the records must be 16-byte aligned
    with pytest.raises(ValueError):
        _desc(rope_bf16=True)
