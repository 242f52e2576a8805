"""The seeded input generator (workloads/gen.py) against its stated recipe:
shapes and seqlen distributions of the named workloads, the shuffled page
pool and block table, NaN poisoning of memory no request owns, the fp8 scale
rule (amax / 448 per group) and the variant-B record layout."""
import math

import numpy as np
import pytest
import torch

from workloads import gen

SPECS = {  # name: (batch, s_q, heads, fp8)
    "tiny": (2, 1, 16, False), "decode": (64, 1, 128, False), "mtp": (128, 2, 128, False),
    "long": (16, 1, 128, False), "fp8": (256, 2, 128, True), "mtp6": (64, 6, 128, False),
    "fp8b": (256, 2, 128, True),
}


@pytest.mark.parametrize("name", list(SPECS))
def test_named_workloads_match_their_recipe(name):
    spec = gen.workload_spec(name)
    assert (spec.batch, spec.s_q, spec.heads, spec.kv_fp8) == SPECS[name]
    assert spec.seed == 20260000 + gen.WORKLOADS.index(name) + 1
    sl = gen._seqlens_for(name, spec.batch, torch.Generator("cpu").manual_seed(spec.seed))
    assert sl.dtype == torch.int32 and sl.numel() == spec.batch
    if name == "decode":
        assert int(sl.min()) >= 1024 and int(sl.max()) <= 4096 and len(set(sl.tolist())) > 32
    elif name in ("mtp", "mtp6"):
        assert (sl == 4096).all()
    elif name in ("fp8", "fp8b"):
        assert (sl == 2048).all()
    elif name == "long":
        assert int(sl[0]) == 65536 and int(sl[1:].min()) >= 64 and int(sl[1:].max()) <= 32768
    else:
        assert sl.tolist() == [37, 130]


def test_long_seqlens_are_lognormal_with_arithmetic_mean_3500():
    # mu = ln 3500 - sigma^2 / 2 with sigma = 1: median e^mu ~ 2123; clipping
    # at 32768 takes ~1.2% off the mean (3457)
    sl = gen._seqlens_for("long", 200_001, torch.Generator("cpu").manual_seed(5))[1:].double()
    assert 3380 < float(sl.mean()) < 3530
    assert abs(float(sl.median()) - 3500 * math.exp(-0.5)) < 40
    z = (sl.clamp(65, 32767).log() - (math.log(3500) - 0.5))
    assert abs(float(z.std()) - 1.0) < 0.02


@pytest.mark.parametrize("fp8,rope_bf16", [(False, False), (True, False), (True, True)])
def test_page_pool_block_table_and_poisoning(fp8, rope_bf16):
    seqlens = [1, 64, 65, 0, 300]
    inp = gen.make_inputs("x", seqlens=seqlens, heads=4, s_q=1, kv_fp8=fp8, rope_bf16=rope_bf16, seed=11)
    pages = [(s + 63) // 64 for s in seqlens]
    owned = sum(pages)
    assert inp.num_pages == owned + math.ceil(0.05 * owned)
    assert inp.max_pages_per_seq == max(pages)
    bt = inp.block_table
    ids = []
    for b, n in enumerate(pages):
        assert (bt[b, n:] == -1).all()
        ids += bt[b, :n].tolist()
    assert len(ids) == owned == len(set(ids)) and all(0 <= i < inp.num_pages for i in ids)
    # which (page, slot) a request owns
    own = torch.zeros((inp.num_pages, 64), dtype=torch.bool)
    for b, s in enumerate(seqlens):
        for t in range(s):
            own[int(bt[b, t // 64]), t % 64] = True
    if not fp8:
        kv = inp.kv.float()
        assert torch.isnan(kv[~own]).all() and torch.isfinite(kv[own]).all()
    elif not rope_bf16:
        assert (inp.kv[~own] == 0x7F).all() and torch.isnan(inp.kv_scales[~own]).all()
        assert torch.isfinite(inp.kv_scales[own]).all() and (inp.kv_scales[own] > 0).all()
    else:
        rec = inp.kv
        sc = rec[..., 512:528].contiguous().view(torch.float32)
        rope = rec[..., 528:656].contiguous().view(torch.bfloat16).float()
        assert inp.kv_scales is None
        assert (rec[~own][:, :512] == 0x7F).all() and torch.isnan(sc[~own]).all() and torch.isnan(rope[~own]).all()
        assert torch.isfinite(sc[own]).all() and (sc[own] > 0).all() and torch.isfinite(rope[own]).all()


@pytest.mark.parametrize("rope_bf16", [False, True])
def test_fp8_scale_is_group_amax_over_448(rope_bf16):
    """With scale = amax / 448, the largest |code| of every owned group is
    exactly 448, the e4m3 maximum."""
    inp = gen.make_inputs("x", seqlens=[200, 77], heads=4, s_q=1, kv_fp8=True, rope_bf16=rope_bf16, seed=13)
    groups = gen.FP8_GROUPS[:4] if rope_bf16 else gen.FP8_GROUPS
    codes = inp.kv[..., :576].contiguous() if not rope_bf16 else inp.kv[..., :512].contiguous()
    vals = codes.view(torch.float8_e4m3fn).float()
    own = torch.zeros((inp.num_pages, 64), dtype=torch.bool)
    for b, s in enumerate(inp.seqlens.tolist()):
        for t in range(s):
            own[int(inp.block_table[b, t // 64]), t % 64] = True
    for c0, c1 in groups:
        amax = vals[..., c0:c1].abs().amax(dim=-1)
        assert (amax[own] == 448.0).all()


def test_values_are_standard_normal_and_draws_are_seeded():
    a = gen.make_inputs("decode", batch=4)
    b = gen.make_inputs("decode", batch=4)
    c = gen.make_inputs("decode", batch=4, seed=99)
    assert torch.equal(a.q, b.q) and torch.equal(a.block_table, b.block_table)
    assert not torch.equal(a.q, c.q)
    q = a.q.float().flatten()
    assert abs(float(q.mean())) < 0.01 and abs(float(q.std()) - 1.0) < 0.01
    kv = a.kv.float()
    kv = kv[torch.isfinite(kv)]
    assert abs(float(kv.mean())) < 0.01 and abs(float(kv.std()) - 1.0) < 0.01
