"""Seeded synthetic inputs for MLA paged decode (absorbed form).

This module only draws inputs: shapes, seeds, random values, the shuffled page
pool and the NaN poisoning of memory that no request owns.  It contains none of
the attention arithmetic, so both the CPU oracle and the CUDA path can consume
what it produces without sharing any of the method.

Workloads (one per named configuration):

* ``tiny``      B=2,   s_q=1, H=16,  seqlens {37, 130}
* ``decode``    B=64,  s_q=1, H=128, seqlens uniform integers in [1024, 4096]
* ``mtp``       B=128, s_q=2, H=128, every seqlen 4096 (causal MTP verify)
* ``long``      B=16,  s_q=1, H=128, lognormal seqlens (arithmetic mean 3500,
                sigma 1.0) clipped to [64, 32768], request 0 set to 65536
* ``fp8``       B=256, s_q=2, H=128, every seqlen 2048, KV stored as e4m3 with
                one fp32 scale per token per channel group
* ``mtp6``      B=64,  s_q=6, H=128, every seqlen 4096 (five draft tokens)
* ``fp8b``      as ``fp8``, with the cache in fp8 variant B: a 656-byte record
                per token (e4m3 latent, 4 fp32 scales, RoPE kept bf16)

Recipe (fixed, documented so a reader can regenerate any case):

* seed: ``torch.Generator('cpu').manual_seed(20260000 + k)`` where k is the
  1-based position of the workload in the list above; draw order is seqlens,
  page permutation, q, kv.
* q and the latent KV are N(0, 1) drawn in fp32 and rounded to bf16.
* page pool: ``sum(ceil(seqlen/64))`` owned pages plus 5% spare pages
  (rounded up).  A random permutation of all page ids is dealt to requests in
  order; the rest are spare.  Unused block-table entries hold -1.
* poisoning: spare pages and the slots past ``seqlen`` in each request's last
  page hold NaN (bf16) or the e4m3 NaN code 0x7F with NaN scales (fp8), so any
  read of memory a request does not own shows up in its output.
* fp8 cache: groups are channels [0,128), [128,256), [256,384), [384,512),
  [512,576); scale = amax(|group|)/448 (1.0 when the group is all zero); the
  code is the e4m3 (OCP E4M3FN) value of x/scale clamped to [-448, 448],
  encoded with torch's float8_e4m3fn conversion.
* fp8 variant B: the four latent groups are quantised the same way; the token
  record is bytes [0,512) e4m3 latent codes, [512,528) the four fp32 scales,
  [528,656) the 64 RoPE channels as bf16 (the fp32 draw rounded to bf16).
  Poisoned slots hold code 0x7F, NaN scales and NaN RoPE.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

PAGE = 64          # tokens per KV page
D_QK = 576         # 512 latent + 64 RoPE channels per query head / KV token
D_V = 512          # output channels (the latent part of each KV row)
FP8_GROUPS = ((0, 128), (128, 256), (256, 384), (384, 512), (512, 576))
FP8B_RECORD = 656  # fp8 variant B bytes per token: 512 e4m3 + 4 fp32 scales + 64 bf16 RoPE
SOFTMAX_SCALE = 1.0 / math.sqrt(192.0)

WORKLOADS = ("tiny", "decode", "mtp", "long", "fp8", "mtp6", "fp8b")


@dataclasses.dataclass
class Workload:
    name: str
    batch: int
    s_q: int
    heads: int
    kv_fp8: bool
    seed: int


def workload_spec(name: str) -> Workload:
    table = {
        "tiny": (2, 1, 16, False),
        "decode": (64, 1, 128, False),
        "mtp": (128, 2, 128, False),
        "long": (16, 1, 128, False),
        "fp8": (256, 2, 128, True),
        # five draft tokens per request (s_q = 6, 768 query rows per request)
        "mtp6": (64, 6, 128, False),
        # fp8 variant B: latent e4m3 with 4 group scales, RoPE kept bf16 (656 B/token)
        "fp8b": (256, 2, 128, True),
    }
    if name not in table:
        raise KeyError(f"unknown workload {name!r}; known: {WORKLOADS}")
    b, s_q, h, fp8 = table[name]
    return Workload(name, b, s_q, h, fp8, 20260000 + WORKLOADS.index(name) + 1)


@dataclasses.dataclass
class Inputs:
    """One decode call's inputs, all on the CPU."""

    name: str
    batch: int
    s_q: int
    heads: int
    q: torch.Tensor                 # bf16 [B, s_q, H, 576]
    kv: torch.Tensor                # bf16 [P, 64, 576], uint8 e4m3 codes [P, 64, 576], or (fp8 variant B)
                                    # uint8 [P, 64, 656] token records
    kv_scales: Optional[torch.Tensor]  # fp32 [P, 64, 5] for the fp8 cache (variant A), else None
    block_table: torch.Tensor       # int32 [B, max_pages_per_seq], -1 = unused
    seqlens: torch.Tensor           # int32 [B]
    softmax_scale: float
    kv_fp8: bool
    rope_bf16: bool = False         # fp8 variant B: the token record keeps RoPE in bf16

    @property
    def num_pages(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_pages_per_seq(self) -> int:
        return int(self.block_table.shape[1])


def _seqlens_for(name: str, batch: int, g: torch.Generator) -> torch.Tensor:
    if name == "tiny":
        return torch.tensor([37, 130], dtype=torch.int32)
    if name == "decode":
        return torch.randint(1024, 4097, (batch,), generator=g, dtype=torch.int64).to(torch.int32)
    if name == "mtp":
        return torch.full((batch,), 4096, dtype=torch.int32)
    if name == "long":
        sigma = 1.0
        mu = math.log(3500.0) - 0.5 * sigma * sigma
        z = torch.randn((batch,), generator=g, dtype=torch.float64)
        s = torch.exp(mu + sigma * z).round().clamp(64, 32768).to(torch.int32)
        s[0] = 65536
        return s
    if name == "fp8":
        return torch.full((batch,), 2048, dtype=torch.int32)
    if name == "mtp6":
        return torch.full((batch,), 4096, dtype=torch.int32)
    if name == "fp8b":
        return torch.full((batch,), 2048, dtype=torch.int32)
    raise KeyError(name)


def make_inputs(name: str, *, poison: bool = True, seqlens: Optional[Sequence[int]] = None,
                batch: Optional[int] = None, heads: Optional[int] = None, s_q: Optional[int] = None,
                kv_fp8: Optional[bool] = None, seed: Optional[int] = None,
                spare_frac: float = 0.05, rope_bf16: Optional[bool] = None) -> Inputs:
    """Draw the inputs of workload ``name``.

    The keyword overrides build smaller or edge-case variants with the same
    recipe (explicit seqlens, batch, heads, s_q, cache dtype or seed).
    """
    spec = workload_spec(name) if name in WORKLOADS else Workload(name, 1, 1, 16, False, 1)
    if seed is None:
        seed = spec.seed
    g = torch.Generator("cpu").manual_seed(seed)
    B = batch if batch is not None else spec.batch
    H = heads if heads is not None else spec.heads
    sq = s_q if s_q is not None else spec.s_q
    fp8 = kv_fp8 if kv_fp8 is not None else spec.kv_fp8
    rb16 = rope_bf16 if rope_bf16 is not None else name == "fp8b"
    if rb16 and not fp8:
        raise ValueError("rope_bf16 is a layout of the fp8 cache")
    if seqlens is not None:
        sl = torch.tensor(list(seqlens), dtype=torch.int32)
        B = int(sl.numel())
    else:
        sl = _seqlens_for(name, B, g)
    if int(sl.numel()) != B:
        raise ValueError("seqlens length does not match batch")

    pages_per = [(int(s) + PAGE - 1) // PAGE for s in sl.tolist()]
    owned = sum(pages_per)
    spare = int(math.ceil(owned * spare_frac))
    num_pages = max(1, owned + spare)
    maxp = max(1, max(pages_per) if pages_per else 1)
    perm = torch.randperm(num_pages, generator=g).to(torch.int32)
    bt = torch.full((B, maxp), -1, dtype=torch.int32)
    cur = 0
    for b, n in enumerate(pages_per):
        if n:
            bt[b, :n] = perm[cur:cur + n]
        cur += n
    spare_ids = perm[cur:]

    q = torch.randn((B, sq, H, D_QK), generator=g, dtype=torch.float32).to(torch.bfloat16)
    kv32 = torch.randn((num_pages, PAGE, D_QK), generator=g, dtype=torch.float32)

    # memory no request owns: spare pages and the tail of each last page
    unowned = torch.zeros((num_pages, PAGE), dtype=torch.bool)
    if spare_ids.numel():
        unowned[spare_ids.long()] = True
    for b, s in enumerate(sl.tolist()):
        n = pages_per[b]
        if n and s % PAGE:
            unowned[int(bt[b, n - 1]), s % PAGE:] = True

    scales = None
    if fp8 and rb16:
        # variant B token record: e4m3 latent [0,512), 4 fp32 scales [512,528)
        # (groups of 128 latent channels), RoPE bf16 [528,656)
        rec = torch.empty((num_pages, PAGE, FP8B_RECORD), dtype=torch.uint8)
        sc4 = torch.empty((num_pages, PAGE, 4), dtype=torch.float32)
        for gi, (c0, c1) in enumerate(FP8_GROUPS[:4]):
            grp = kv32[:, :, c0:c1]
            amax = grp.abs().amax(dim=-1)
            sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            sc4[:, :, gi] = sc
            x = (grp / sc.unsqueeze(-1)).clamp(-448.0, 448.0)
            rec[:, :, c0:c1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        rope = kv32[:, :, D_V:D_QK].to(torch.bfloat16)
        if poison:
            rec[unowned, :D_V] = 0x7F
            sc4[unowned] = float("nan")
            rope[unowned] = float("nan")
        rec[:, :, D_V:D_V + 16] = sc4.contiguous().view(torch.uint8).view(num_pages, PAGE, 16)
        rec[:, :, D_V + 16:] = rope.contiguous().view(torch.uint8).view(num_pages, PAGE, 128)
        kv = rec
    elif fp8:
        scales = torch.empty((num_pages, PAGE, len(FP8_GROUPS)), dtype=torch.float32)
        codes = torch.empty((num_pages, PAGE, D_QK), dtype=torch.uint8)
        for gi, (c0, c1) in enumerate(FP8_GROUPS):
            grp = kv32[:, :, c0:c1]
            amax = grp.abs().amax(dim=-1)
            sc = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
            scales[:, :, gi] = sc
            x = (grp / sc.unsqueeze(-1)).clamp(-448.0, 448.0)
            codes[:, :, c0:c1] = x.to(torch.float8_e4m3fn).view(torch.uint8)
        if poison:
            codes[unowned] = 0x7F
            scales[unowned] = float("nan")
        kv = codes
    else:
        kv = kv32.to(torch.bfloat16)
        if poison:
            kv[unowned] = float("nan")

    return Inputs(name=name, batch=B, s_q=sq, heads=H, q=q, kv=kv, kv_scales=scales,
                  block_table=bt, seqlens=sl, softmax_scale=SOFTMAX_SCALE, kv_fp8=fp8, rope_bf16=rb16)


def sample_rows(inp: Inputs, n: int, seed: int = 7) -> torch.Tensor:
    """A seeded sample of flat query-row ids (b*s_q*H + i*H + h) that always
    includes the first and last row of every request."""
    g = torch.Generator("cpu").manual_seed(seed)
    R = inp.s_q * inp.heads
    total = inp.batch * R
    must = []
    for b in range(inp.batch):
        must += [b * R, b * R + R - 1]
    rnd = torch.randint(0, total, (max(0, n - len(must)),), generator=g).tolist()
    return torch.tensor(sorted(set(must + rnd)), dtype=torch.int64)


def shard_requests(batch: int, rank: int, world: int) -> range:
    """Contiguous request shard of one data-parallel replica."""
    per = (batch + world - 1) // world
    lo = min(batch, rank * per)
    return range(lo, min(batch, lo + per))
