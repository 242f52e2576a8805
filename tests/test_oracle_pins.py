"""Pins of the CPU oracle against things other than itself.

Each check is chosen so that a plausible slip in the oracle (a wrong channel
split, a dropped RoPE term, a wrong causal offset, a log base, a transposed
gather, a wrong fp8 group) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import KV_BF16, KV_F64, KV_FP8
from workloads import gen

SCALE = 1.0 / math.sqrt(192.0)


def _dense_cache_f64(P, rng):
    return rng.standard_normal((P, 64, 576))


def _table(rng, B, pages_per, P):
    perm = rng.permutation(P)
    maxp = max(pages_per)
    bt = -np.ones((B, maxp), dtype=np.int32)
    cur = 0
    for b, n in enumerate(pages_per):
        bt[b, :n] = perm[cur:cur + n]
        cur += n
    return bt


def _gather(kv, bt, b, n):
    """Dense [n, 576] keys of request b, gathered with numpy fancy indexing."""
    t = np.arange(n)
    return kv[bt[b, t // 64], t % 64]


# --------------------------------------------------------------- decoders
def test_bf16_decoder_matches_torch_for_every_code():
    codes = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = codes.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(c) for c in range(1 << 16)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_e4m3_decoder_matches_torch_for_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(c) for c in range(256)])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), np.nonzero(~same)
    assert oracle.e4m3_to_f64(0x7E) == 448.0 and np.isnan(oracle.e4m3_to_f64(0x7F))


# --------------------------------------------------------- non-absorbed form
@pytest.mark.parametrize("s_q", [1, 2])
def test_absorbed_equals_non_absorbed_mla(s_q):
    """Standard MLA (latent up-projected by W_UK / W_UV, 192-wide heads) equals
    the absorbed computation the oracle does, after W_UV^T on its output."""
    rng = np.random.default_rng(11 + s_q)
    B, H = 2, 3
    seqlens = np.array([5, 70], dtype=np.int32)
    pages = [(int(s) + 63) // 64 for s in seqlens]
    P = sum(pages) + 2
    bt = _table(rng, B, pages, P)
    latent = rng.standard_normal((P, 64, 512))
    krope = rng.standard_normal((P, 64, 64))
    W_UK = rng.standard_normal((H, 512, 128)) / 8.0
    W_UV = rng.standard_normal((H, 512, 128)) / 8.0
    q_nope = rng.standard_normal((B, s_q, H, 128))
    q_rope = rng.standard_normal((B, s_q, H, 64))

    # absorbed inputs: q_h = [W_UK_h q_nope_h ; q_rope_h], KV row = [c_t ; k_rope_t]
    q_abs = oracle.absorb_q(q_nope.reshape(B * s_q, H, 128), q_rope.reshape(B * s_q, H, 64),
                            W_UK).reshape(B, s_q, H, 576)
    kv = np.concatenate([latent, krope], axis=-1)
    out_abs, lse_abs = oracle.mla_decode(q_abs, kv, bt, seqlens, s_q, SCALE, kv_dtype=KV_F64)
    o_abs = oracle.project_out(out_abs.reshape(B * s_q, H, 512), W_UV).reshape(B, s_q, H, 128)
    out_abs = out_abs.reshape(B, s_q, H, 512)
    lse_abs = lse_abs.reshape(B, s_q, H)

    for b in range(B):
        for i in range(s_q):
            n = int(seqlens[b]) - s_q + i + 1
            c = _gather(latent, bt, b, n)
            kr = _gather(krope, bt, b, n)
            for h in range(H):
                k = np.concatenate([c @ W_UK[h], kr], axis=1)          # [n, 192]
                v = c @ W_UV[h]                                        # [n, 128]
                qh = np.concatenate([q_nope[b, i, h], q_rope[b, i, h]])
                s = k @ qh / math.sqrt(192.0)
                p = np.exp(s - s.max())
                out_std = (p / p.sum()) @ v
                lse_std = s.max() + math.log(p.sum())
                np.testing.assert_allclose(W_UV[h].T @ out_abs[b, i, h], out_std, rtol=1e-10, atol=1e-12)
                np.testing.assert_allclose(o_abs[b, i, h], out_std, rtol=1e-10, atol=1e-12)
                assert abs(lse_abs[b, i, h] - lse_std) < 1e-10


# ----------------------------------------------------------------- closed forms
def test_single_key_returns_its_value_and_score():
    inp = gen.make_inputs("x", seqlens=[1, 1], heads=4, s_q=1, seed=3)
    out, lse = oracle.mla_decode_inputs(inp)
    kv = inp.kv.to(torch.float64).numpy()
    q = inp.q.to(torch.float64).numpy()
    bt = inp.block_table.numpy()
    for b in range(2):
        k0 = kv[bt[b, 0], 0]
        for h in range(4):
            r = b * 4 + h
            assert np.array_equal(out[r], k0[:512])
            assert lse[r] == pytest.approx(SCALE * float(q[b, 0, h] @ k0), abs=1e-12)


def test_identical_scores_give_mean_of_values():
    """Latent q zero and all RoPE rows equal: every score is the same, so the
    weights are uniform, out is the mean latent and lse = s + ln n."""
    rng = np.random.default_rng(5)
    n = 150
    P = 4
    bt = np.array([[2, 0, 3]], dtype=np.int32)
    kv = rng.standard_normal((P, 64, 576))
    rope = rng.standard_normal(64)
    kv[:, :, 512:] = rope
    q = np.zeros((1, 1, 2, 576))
    q[..., 512:] = rng.standard_normal((1, 1, 2, 64))
    out, lse = oracle.mla_decode(q, kv, bt, np.array([n], np.int32), 1, SCALE, kv_dtype=KV_F64)
    lat = _gather(kv, bt, 0, n)[:, :512]
    for h in range(2):
        s = SCALE * float(q[0, 0, h, 512:] @ rope)
        np.testing.assert_allclose(out[h], lat.mean(axis=0), rtol=0, atol=1e-13)
        assert lse[h] == pytest.approx(s + math.log(n), abs=1e-12)


@pytest.mark.parametrize("shift", [1.0e4, -1.0e4])
def test_common_score_shift_leaves_out_and_moves_lse(shift):
    """Adding the same amount to every key's score (through a RoPE channel
    equal for all keys) leaves the softmax weights, and so out, unchanged and
    moves lse by exactly that amount.  At +-1e4 a softmax without the maximum
    subtracted overflows (or underflows to 0/0) in fp64, so this also fails
    if the oracle's stabilisation is missing or wrong."""
    rng = np.random.default_rng(21)
    n = 230
    bt = np.array([[3, 0, 4, 1]], dtype=np.int32)
    kv = rng.standard_normal((5, 64, 576))
    kv[:, :, 575] = 1.0
    q = rng.standard_normal((1, 1, 3, 576))
    q[..., 575] = 0.0
    o0, l0 = oracle.mla_decode(q, kv, bt, np.array([n], np.int32), 1, SCALE, kv_dtype=KV_F64)
    q[..., 575] = shift / SCALE
    o1, l1 = oracle.mla_decode(q, kv, bt, np.array([n], np.int32), 1, SCALE, kv_dtype=KV_F64)
    assert np.isfinite(o1).all() and np.isfinite(l1).all()
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0 + shift, rtol=0, atol=1e-9)


def test_two_key_hand_derivation():
    """Scores 0 and 1 (scale 1): p = (1, e)/(1+e), lse = ln(1+e)."""
    q = np.zeros((1, 1, 1, 576))
    q[0, 0, 0, 0] = 1.0
    q[0, 0, 0, 512] = 1.0
    kv = np.zeros((1, 64, 576))
    kv[0, 0, 1] = 2.0                      # key 0: score 0, value e_1 * 2
    kv[0, 1, 0] = 0.5                      # key 1: score 0.5 + 0.5 = 1
    kv[0, 1, 512] = 0.5
    kv[0, 1, 1] = -1.0
    kv[0, 2:] = np.nan                     # never visible
    out, lse = oracle.mla_decode(q, kv, np.array([[0]], np.int32), np.array([2], np.int32), 1, 1.0,
                                 kv_dtype=KV_F64)
    e = math.e
    p0, p1 = 1.0 / (1.0 + e), e / (1.0 + e)
    want = np.zeros(512)
    want[0] = 0.5 * p1
    want[1] = 2.0 * p0 - p1
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-15)
    assert lse[0] == pytest.approx(math.log(1.0 + e), abs=1e-15)


def test_softmax_rows_sum_to_one():
    inp = gen.make_inputs("tiny")
    out, lse, p = oracle.mla_decode_inputs(inp, return_p=True)
    R = inp.s_q * inp.heads
    for r in range(out.shape[0]):
        n = int(inp.seqlens[r // R])
        assert abs(p[r, :n].sum() - 1.0) < 1e-12
        assert (p[r, :n] > 0).all() and (p[r, n:] == 0).all()


def test_empty_visible_set_gives_zero_and_minus_inf():
    inp = gen.make_inputs("x", seqlens=[1, 0], heads=2, s_q=2, seed=4)
    out, lse = oracle.mla_decode_inputs(inp)
    # request 0 (seqlen 1, s_q 2): token 0 sees nothing, token 1 sees key 0
    assert (out[0:2] == 0).all() and np.isneginf(lse[0:2]).all()
    assert np.isfinite(lse[2:4]).all()
    assert (out[4:] == 0).all() and np.isneginf(lse[4:]).all()


# --------------------------------------------------------------- identities
def test_lse_merge_of_disjoint_key_ranges_equals_whole():
    rng = np.random.default_rng(9)
    n, cut_pages = 300, 2
    P = 6
    kv = rng.standard_normal((P, 64, 576))
    bt = np.array([[4, 1, 5, 0, 3]], dtype=np.int32)
    q = rng.standard_normal((1, 1, 3, 576))
    whole_o, whole_l = oracle.mla_decode(q, kv, bt, np.array([n], np.int32), 1, SCALE, kv_dtype=KV_F64)
    # keys [0, 128): same table, seqlen 128; keys [128, 300): table shifted by two pages
    o1, l1 = oracle.mla_decode(q, kv, bt, np.array([64 * cut_pages], np.int32), 1, SCALE, kv_dtype=KV_F64)
    bt2 = np.ascontiguousarray(bt[:, cut_pages:])
    o2, l2 = oracle.mla_decode(q, kv, bt2, np.array([n - 64 * cut_pages], np.int32), 1, SCALE, kv_dtype=KV_F64)
    l = np.logaddexp(l1, l2)
    o = np.exp(l1 - l)[:, None] * o1 + np.exp(l2 - l)[:, None] * o2
    np.testing.assert_allclose(l, whole_l, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o, whole_o, rtol=0, atol=1e-12)


def test_causal_verify_equals_batch_extension():
    """Row i of an s_q=2 verify call equals an s_q=1 call whose seqlen ends at
    that token (the batch-extension formulation the pages replace)."""
    inp = gen.make_inputs("x", seqlens=[37, 130, 64], heads=4, s_q=2, seed=12)
    out2, lse2 = oracle.mla_decode_inputs(inp)
    out2 = out2.reshape(3, 2, 4, 512)
    lse2 = lse2.reshape(3, 2, 4)
    for i in range(2):
        sl = (inp.seqlens - 1 + i).to(torch.int32)
        o1, l1 = oracle.mla_decode(inp.q[:, i:i + 1].contiguous(), inp.kv, inp.block_table, sl, 1,
                                   inp.softmax_scale)
        assert np.array_equal(o1.reshape(3, 4, 512), out2[:, i])
        assert np.array_equal(l1.reshape(3, 4), lse2[:, i])


def test_causal_probe_last_key_hidden_from_first_draft_token():
    rng = np.random.default_rng(21)
    n = 100
    P = 2
    kv = rng.standard_normal((P, 64, 576)) * 0.1
    bt = np.array([[1, 0]], dtype=np.int32)
    q = rng.standard_normal((1, 2, 1, 576)) * 0.1
    t_last = n - 1
    pg, sl = bt[0, t_last // 64], t_last % 64
    kv[:, :, 3] = 0.0
    kv[pg, sl, :] = 0.0
    kv[pg, sl, 3] = 1.0
    q[0, :, 0, 3] = 400.0                  # huge score only on the last key
    out, lse = oracle.mla_decode(q, kv, bt, np.array([n], np.int32), 2, SCALE, kv_dtype=KV_F64)
    assert out[1, 3] == pytest.approx(1.0, abs=1e-9)      # token 1 sees it: one-hot
    assert abs(out[0, 3]) < 0.5                           # token 0 does not


def test_matches_dense_torch_softmax():
    inp = gen.make_inputs("tiny")
    out, lse = oracle.mla_decode_inputs(inp)
    kv = inp.kv.to(torch.float64)
    q = inp.q.to(torch.float64)
    R = inp.s_q * inp.heads
    for b in range(inp.batch):
        n = int(inp.seqlens[b])
        t = torch.arange(n)
        K = kv[inp.block_table[b, t // 64].long(), t % 64]           # [n, 576]
        S = inp.softmax_scale * q[b, 0] @ K.T                        # [H, n]
        Pm = torch.softmax(S, dim=-1)
        ref = Pm @ K[:, :512]
        np.testing.assert_allclose(out[b * R:(b + 1) * R], ref.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b * R:(b + 1) * R], torch.logsumexp(S, dim=-1).numpy(), atol=1e-12)


def test_fp8_cache_equals_library_dequantized_cache():
    """The oracle's fp8 path equals its fp64 path run on torch's e4m3 decode
    times the per-group scales (pins the channel-group mapping)."""
    inp = gen.make_inputs("x", seqlens=[70, 129], heads=4, s_q=2, kv_fp8=True, seed=8)
    out8, lse8 = oracle.mla_decode_inputs(inp)
    vals = inp.kv.view(torch.float8_e4m3fn).to(torch.float64)
    sc = inp.kv_scales.to(torch.float64)
    groups = torch.tensor([0] * 128 + [1] * 128 + [2] * 128 + [3] * 128 + [4] * 64)
    deq = vals * sc[:, :, groups]
    o64, l64 = oracle.mla_decode(inp.q.to(torch.float64), deq, inp.block_table, inp.seqlens, 2,
                                 inp.softmax_scale, kv_dtype=KV_F64)
    np.testing.assert_allclose(out8, o64, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse8, l64, rtol=0, atol=1e-12)
    # and close to the unquantized values the cache was drawn from (information only)
    assert np.isfinite(out8).all()


def test_poisoned_memory_is_never_read():
    for name in ("tiny",):
        inp = gen.make_inputs(name, poison=True)
        out, lse = oracle.mla_decode_inputs(inp)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
    inp = gen.make_inputs("x", seqlens=[65, 3], heads=2, s_q=1, kv_fp8=True, seed=2)
    out, lse = oracle.mla_decode_inputs(inp)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


def test_bad_page_id_is_an_error():
    inp = gen.make_inputs("x", seqlens=[70], heads=2, s_q=1, seed=2)
    bt = inp.block_table.clone()
    bt[0, 1] = inp.num_pages + 3
    with pytest.raises(RuntimeError):
        oracle.mla_decode(inp.q, inp.kv, bt, inp.seqlens, 1, inp.softmax_scale)


def test_fp8_cache_decodes_like_torch_in_the_oracle():
    """The oracle's fp8 path (e4m3 codes times the per-token group scales)
    equals its fp64 path on the cache dequantised independently with torch's
    float8_e4m3fn decoder, bit for bit."""
    inp = gen.make_inputs("x", seqlens=[70, 5, 1], heads=8, s_q=2, kv_fp8=True, seed=3)
    codes = inp.kv.view(torch.float8_e4m3fn).to(torch.float64)
    grp = torch.tensor([0] * 128 + [1] * 128 + [2] * 128 + [3] * 128 + [4] * 64)
    exact = codes * inp.kv_scales.to(torch.float64)[:, :, grp]
    o_f, l_f = oracle.mla_decode(inp.q.to(torch.float64), exact, inp.block_table, inp.seqlens, inp.s_q,
                                 inp.softmax_scale, kv_dtype=oracle.KV_F64)
    o_c, l_c = oracle.mla_decode_inputs(inp)
    assert np.array_equal(o_f, o_c) and np.array_equal(l_f, l_c)


def test_fp8_variant_b_records_decode_like_torch():
    """The oracle's fp8 variant B path (656-byte token records) equals its
    fp64 path on the same cache decoded independently with torch: e4m3 codes
    with float8_e4m3fn, the scales as float32, the RoPE as bfloat16."""
    inp = gen.make_inputs("x", seqlens=[70, 5, 1], heads=8, s_q=2, kv_fp8=True, rope_bf16=True, seed=9)
    rec = inp.kv
    assert rec.shape[-1] == 656 and inp.kv_scales is None
    lat = rec[:, :, :512].contiguous().view(torch.float8_e4m3fn).to(torch.float64)
    sc = rec[:, :, 512:528].contiguous().view(torch.float32).to(torch.float64)
    rope = rec[:, :, 528:].contiguous().view(torch.bfloat16).to(torch.float64)
    dense = torch.cat([lat * sc.repeat_interleave(128, dim=-1), rope], dim=-1)
    o_f, l_f = oracle.mla_decode(inp.q.to(torch.float64), dense, inp.block_table, inp.seqlens, inp.s_q,
                                 inp.softmax_scale, kv_dtype=KV_F64)
    o_b, l_b = oracle.mla_decode_inputs(inp)
    assert np.array_equal(o_f, o_b) and np.array_equal(l_f, l_b)
    # a single key returns its own latent row (the dequantised codes)
    one = gen.make_inputs("x", seqlens=[1], heads=2, s_q=1, kv_fp8=True, rope_bf16=True, seed=2)
    o1, _ = oracle.mla_decode_inputs(one)
    r0 = one.kv[int(one.block_table[0, 0]), 0]
    want = r0[:512].contiguous().view(torch.float8_e4m3fn).to(torch.float64) * \
        r0[512:528].contiguous().view(torch.float32).to(torch.float64).repeat_interleave(128)
    assert np.array_equal(o1[0], want.numpy()) and np.array_equal(o1[1], want.numpy())


def test_fp8_q_quantisation_breaks_the_lse_bound():
    """Why there is no fp8 (kind::f8f6f4) QK path: even with the dequantised
    cache exact, rounding q to e4m3 (per-row scale amax/448) moves lse far past
    the 1e-3 bound; tensor-core block scales are powers of two, so the cache's
    fp32 scales could not be applied exactly either."""
    inp = gen.make_inputs("x", seqlens=[2048, 700], heads=64, s_q=1, kv_fp8=True, seed=3)
    k8 = inp.kv.view(torch.float8_e4m3fn).to(torch.float64)
    grp = torch.tensor([0] * 128 + [1] * 128 + [2] * 128 + [3] * 128 + [4] * 64)
    exact = k8 * inp.kv_scales.to(torch.float64)[:, :, grp]
    q = inp.q.to(torch.float64)
    qs = q.abs().amax(dim=-1, keepdim=True).clamp_min(1e-30) / 448.0
    q8 = (q / qs).to(torch.float8_e4m3fn).to(torch.float64) * qs
    _, l_ex = oracle.mla_decode(q, exact, inp.block_table, inp.seqlens, 1, inp.softmax_scale, kv_dtype=KV_F64)
    _, l_q8 = oracle.mla_decode(q8, exact, inp.block_table, inp.seqlens, 1, inp.softmax_scale, kv_dtype=KV_F64)
    err = np.abs(np.asarray(l_q8) - np.asarray(l_ex))
    assert err.max() > 1e-2 and np.median(err) > 1e-3
