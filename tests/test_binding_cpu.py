"""The Python binding's tensor checks (no GPU): every decode entry point checks
its tensors against the descriptor before the C call, which sees only
pointers and could not tell a tensor too small for the descriptor."""
import pytest
import torch

import mla_paged_decode_absorbed_gb300 as mla

B, SQ, H, P, MAXP = 3, 2, 16, 7, 4


def _tensors(kv_dtype=mla.MLA_KV_BF16):
    t = {
        "q": torch.zeros((B, SQ, H, 576), dtype=torch.bfloat16),
        "kv": torch.zeros((P, 64, 576), dtype=torch.bfloat16),
        "kv_scales": None,
        "block_table": torch.zeros((B, MAXP), dtype=torch.int32),
        "seqlens": torch.zeros((B,), dtype=torch.int32),
        "out": torch.zeros((B, SQ, H, 512), dtype=torch.bfloat16),
        "lse": torch.zeros((B, SQ, H), dtype=torch.float32),
    }
    if kv_dtype == mla.MLA_KV_FP8_E4M3:
        t["kv"] = torch.zeros((P, 64, 576), dtype=torch.uint8)
        t["kv_scales"] = torch.ones((P, 64, 5), dtype=torch.float32)
    elif kv_dtype == mla.MLA_KV_FP8_E4M3_ROPE_BF16:
        t["kv"] = torch.zeros((P, 64, mla.FP8B_RECORD), dtype=torch.uint8)
    return t


def _desc(kv_dtype=mla.MLA_KV_BF16):
    return mla.make_desc(B, SQ, H, P, MAXP, kv_fp8=kv_dtype != mla.MLA_KV_BF16,
                         rope_bf16=kv_dtype == mla.MLA_KV_FP8_E4M3_ROPE_BF16)


def _run(d, t, cuda=False):
    return mla.check_decode_tensors(d, t["q"], t["kv"], t["kv_scales"], t["block_table"], t["seqlens"], t["out"],
                                    t["lse"], cuda=cuda)


@pytest.mark.parametrize("kv_dtype", [mla.MLA_KV_BF16, mla.MLA_KV_FP8_E4M3, mla.MLA_KV_FP8_E4M3_ROPE_BF16])
def test_matching_tensors_pass(kv_dtype):
    t = _tensors(kv_dtype)
    assert _run(_desc(kv_dtype), t) is t["kv"]


def test_e4m3_cache_is_viewed_as_bytes():
    t = _tensors(mla.MLA_KV_FP8_E4M3)
    t["kv"] = torch.zeros((P, 64, 576), dtype=torch.float8_e4m3fn)
    kv = _run(_desc(mla.MLA_KV_FP8_E4M3), t)
    assert kv.dtype == torch.uint8 and kv.data_ptr() == t["kv"].data_ptr()


@pytest.mark.parametrize("name,bad,kv_dtype", [
    ("q", torch.zeros((B, SQ, H, 576), dtype=torch.float32), mla.MLA_KV_BF16),         # dtype
    ("q", torch.zeros((B, 1, H, 576), dtype=torch.bfloat16), mla.MLA_KV_BF16),         # s_q
    ("kv", torch.zeros((P - 1, 64, 576), dtype=torch.bfloat16), mla.MLA_KV_BF16),      # too few pages
    ("kv", torch.zeros((P, 64, 576), dtype=torch.uint8), mla.MLA_KV_BF16),             # fp8 cache, bf16 desc
    ("kv", torch.zeros((P, 64, 576), dtype=torch.uint8), mla.MLA_KV_FP8_E4M3_ROPE_BF16),  # variant A bytes
    ("kv_scales", torch.ones((P, 64, 5)), mla.MLA_KV_BF16),                            # scales without fp8
    ("kv_scales", None, mla.MLA_KV_FP8_E4M3),                                          # fp8 without scales
    ("kv_scales", torch.ones((P, 64, 4)), mla.MLA_KV_FP8_E4M3),                        # 4 groups, not 5
    ("kv_scales", torch.ones((P, 64, 5)), mla.MLA_KV_FP8_E4M3_ROPE_BF16),              # variant B has them inline
    ("block_table", torch.zeros((B, MAXP + 1), dtype=torch.int32), mla.MLA_KV_BF16),
    ("block_table", torch.zeros((B, MAXP), dtype=torch.int64), mla.MLA_KV_BF16),
    ("seqlens", torch.zeros((B + 1,), dtype=torch.int32), mla.MLA_KV_BF16),
    ("out", torch.zeros((B, SQ, H, 512), dtype=torch.float32), mla.MLA_KV_BF16),
    ("out", torch.zeros((B, SQ, H, 1024), dtype=torch.bfloat16)[..., ::2], mla.MLA_KV_BF16),  # not contiguous
    ("lse", torch.zeros((B, SQ, H + 1), dtype=torch.float32), mla.MLA_KV_BF16),
    ("lse", [0.0], mla.MLA_KV_BF16),                                                   # not a tensor
])
def test_mismatched_tensor_is_rejected(name, bad, kv_dtype):
    t = _tensors(kv_dtype)
    t[name] = bad
    with pytest.raises(ValueError):
        _run(_desc(kv_dtype), t)


def test_host_tensors_are_rejected_before_the_library_is_called():
    d, t = _desc(), _tensors()
    ws = torch.zeros(1 << 20, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        _run(d, t, cuda=True)
    args = (t["q"], t["kv"], t["kv_scales"], t["block_table"], t["seqlens"], SQ, 0.07, t["out"], t["lse"])
    for call in (lambda: mla.mla_decode(d, *args, ws), lambda: mla.mla_decode_attention(d, *args, ws),
                 lambda: mla.mla_decode_noalloc(d, *args), lambda: mla.mla_plan(d, t["seqlens"], ws),
                 lambda: mla.mla_combine_workspace(d, t["out"], t["lse"], ws),
                 lambda: mla.mla_combine(d, torch.zeros((2, SQ * H, 512)), torch.zeros((2, SQ * H)),
                                         torch.zeros((B + 1,), dtype=torch.int32), t["out"], t["lse"])):
        with pytest.raises(ValueError, match="CUDA tensor"):
            call()
