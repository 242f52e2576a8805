// MLA paged decode, absorbed form: the attention kernel for sm_103a.
//
// What it computes (PaddleNLP issue #10157, "Multi-head Latent Attention (MLA)
// 算子 / 总体概述"): per 64-token KV page, Data Load -> QK GEMM -> Softmax Update
// (+ P stored where the next MMA reads it) -> PV GEMM, with num_token > 1 per
// request (the MTP verify step of the same page, causal within the new tokens).
//
// Design for GB300 (the pages' Hopper warp-group schemes are prior art only):
//
// * One work unit is 128 query rows (token-major (i, h) rows of one request)
//   times a contiguous range of that request's pages, run by a cluster of two
//   CTAs with different jobs:
//     - the scorer (cluster rank 0) holds the whole Q block (576 channels) in
//       TMEM, computes S = Q K^T over each page with tcgen05 into a
//       double-buffered TMEM S, runs the fp32 online softmax, and streams the
//       16-bit P tile plus a per-row rescale factor into the accumulator's
//       shared memory (st.async, 16.5 KB per page, one direction);
//     - the accumulator (rank 1) holds the 128 x 512 fp32 output in all 512 of
//       its TMEM columns and runs O += P V with P read from shared memory, the
//       (rare) O rescales and the epilogue.
//   Each CTA TMA-loads the channel boxes of each page it needs into its own
//   3-stage ring (scorer: 576 channels, accumulator: 512); the second read of
//   a page comes from L2.
// * Why this split: a 128 x 512 fp32 accumulator fills a whole SM's TMEM, and
//   distributed shared memory moves only ~21 bytes per clock per SM pair (as
//   measured on GB300), so exchanging fp32 partial scores (32 KB per page each
//   way) costs more than the page itself; forwarding 16-bit P costs half and
//   goes one way.
// * Roles per CTA: warp 0 loads pages (TMA, 32 block-table entries per read);
//   warp 1 allocates TMEM and issues the MMAs from one lane; warps 2-5 (one
//   TMEM lane quarter each, one query row per thread) run the softmax
//   (scorer) or the rescale and epilogue (accumulator); warp 6 of the
//   accumulator returns P-buffer credits to the scorer.  The fp8-cache variant
//   adds warps 7-10, which read e4m3 pages with plain coalesced loads and write
//   fp16 into the ring (the MMAs then run in fp16).
// * Online softmax in base 2 with a lazy rescale: the running max only moves
//   (and O is only rescaled) when a tile's max exceeds it by more than 8 (a
//   factor 256); the final division by the row sum is exact either way.  This
//   trick is from FlashAttention-4 (Dao et al., 2025), not the pages.
// * Every barrier wait is bounded (about one second); a timeout sets an error
//   bit, tells the peer CTA to stop, and both CTAs tear down normally.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla_gb300 {
namespace {

using namespace mla_sm103;

constexpr int kBox = 64 * 64 * 2;                  // 64 tokens x 64 channels, 16-bit
constexpr int kStages = 3;
constexpr int kStageS = 9 * kBox;                  // scorer: channels 0..575
constexpr int kStageO = 8 * kBox;                  // accumulator: channels 0..511
constexpr int kPBytes = kRowsPerBlock * 64 * 2;    // P tile: 128 rows x 64 keys, SW128 K-major
constexpr int kVecBytes = kRowsPerBlock * 4;       // one fp32 per row

// Shared-memory layout (byte offsets from the 1024-aligned base; the same in
// both CTAs, each uses its part).
constexpr int kOffP = kStages * kStageO;           // accumulator: P tiles [2]
constexpr int kOffAlpha = kOffP + 2 * kPBytes;     // accumulator: rescale factors [2][128]
constexpr int kOffL = kOffAlpha + 2 * kVecBytes;   // accumulator: row sums [2][128]
constexpr int kOffBars = (kStages * kStageS > kOffL + 2 * kVecBytes) ? kStages * kStageS : kOffL + 2 * kVecBytes;
constexpr int kBarBytes = 256;
constexpr int kSmemMax = 232448;
constexpr int kSmem = kSmemMax;                    // layout + slack for aligning the base
constexpr int kAlignSlack = kSmem - kOffBars - kBarBytes;
static_assert(kAlignSlack >= 0, "shared memory layout too large");

// TMEM columns.  Scorer: Q (576 16-bit channels) then two S buffers.
constexpr uint32_t kColQ = 0, kColS0 = 288, kColS1 = 352;

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool kFp8>
struct Cfg {
  static constexpr int kThreads = kFp8 ? 352 : 224;
};

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t q_full;        // scorer: Q written to TMEM (softmax warps, 128)
  uint64_t s_full[2];     // scorer: QK done (commit)
  uint64_t s_free[2];     // scorer: S read by the softmax (128)
  uint64_t pbuf_free[2];  // scorer: accumulator finished with P tile b (remote, 1)
  uint64_t l_free[2];     // scorer: accumulator read row sums b (remote, 4)
  uint64_t p_full[2];     // accumulator: P tile + factors arrived (1 + tx)
  uint64_t corr_done[2];  // accumulator: O rescaled if needed for tile parity b (128).  Two
                          // of them: the rescale warps may finish tile t+1 before the MMA
                          // warp has observed tile t, which would overrun one barrier.
  uint64_t pv_done[2];    // accumulator: PV of tile with parity b done (commit)
  uint64_t o_full;        // accumulator: last PV of a segment done (commit)
  uint64_t o_free;        // accumulator: epilogue read O (128)
  uint64_t l_full[2];     // accumulator: row sums arrived (1 + tx)
  uint64_t drain;
  int abort_flag;
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block too large");

// One segment of a cluster's cost range: unit u (row block rb of request b),
// pages [page_lo, page_hi) of it.  `empty` units have no visible keys.
struct Seg {
  int u, b, rb, page_lo, page_hi, split, slot, empty;
};

// Walks the units of cluster c in order (the partition rule of mla_plan).
struct SegIter {
  const int32_t* pre;
  int U, B, ovh, c, lo_c, hi_c, u;

  __device__ bool next(Seg& s) {
    while (u < U) {
      const int p0 = __ldg(pre + u);
      if (p0 >= hi_c) {
        u = U;
        return false;
      }
      const int p1 = __ldg(pre + u + 1);
      const int cu = u++;
      const int tiles = p1 - p0 - ovh;
      s.u = cu;
      s.b = cu % B;
      s.rb = cu / B;
      if (tiles <= 0) {
        if (p0 < lo_c) continue;  // belongs to the previous cluster
        s.page_lo = s.page_hi = 0;
        s.split = 0;
        s.slot = -1;
        s.empty = 1;
        return true;
      }
      const int a = p0 + ovh;
      const int lo = max(a, lo_c), hi = min(p1, hi_c);
      if (lo >= hi) continue;
      s.page_lo = lo - a;
      s.page_hi = hi - a;
      s.split = (a < lo_c || p1 > hi_c) ? 1 : 0;
      s.slot = s.split ? (lo == lo_c ? 2 * c : 2 * c + 1) : -1;
      s.empty = 0;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ int clamp_seqlen(int s, int max_pages) {
  return s < 0 ? 0 : (s > max_pages * kPage ? max_pages * kPage : s);
}

__device__ __forceinline__ void signal_abort(Bars* bars, int32_t* err, uint32_t peer) {
  atomicOr(err, kErrTimeout);
  bars->abort_flag = 1;
  st_cluster_u32(mapa_shared(smem_u32(&bars->abort_flag), peer), 1u);
}

// Zero key rows [valid, 64) of `nbox` boxes of a 16-bit stage.  Cache slots
// past seqlen may hold anything, including NaN, and a masked weight of 0 times
// NaN would still poison the PV product.  Whole 128-byte rows, so the swizzle
// does not matter.
__device__ __forceinline__ void zero_tail_rows(uint8_t* stage, int valid, int nbox, int lane) {
  const int per_box = (kPage - valid) * 8;
  const int total = per_box * nbox;
  for (int i = lane; i < total; i += 32) {
    const int box = i / per_box, rem = i - box * per_box;
    const int row = valid + (rem >> 3), ch = rem & 7;
    *reinterpret_cast<uint4*>(stage + box * kBox + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
}

// e4m3 x2 -> two floats (exact through f16).
__device__ __forceinline__ void e4m3x2_to_f32(uint16_t v, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  float2 f = __half22float2(h);
  lo = f.x;
  hi = f.y;
}

// Tree reductions over 64 values (independent chains for ILP).
__device__ __forceinline__ float max64(const float (&x)[64]) {
  float m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) m[i] = fmaxf(fmaxf(fmaxf(x[8 * i], x[8 * i + 1]), fmaxf(x[8 * i + 2], x[8 * i + 3])),
                                           fmaxf(fmaxf(x[8 * i + 4], x[8 * i + 5]), fmaxf(x[8 * i + 6], x[8 * i + 7])));
  return fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
}

template <bool kFp8>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const bool scorer = rank == 0;
  if (pad > static_cast<uint32_t>(kAlignSlack)) {  // never expected: report, do nothing
    if (tid == 0) atomicOr(a.err, kErrTimeout);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), kFp8 ? 128 : 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    mbar_init(smem_u32(&bars->q_full), 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->s_free[i]), 128);
      mbar_init(smem_u32(&bars->pbuf_free[i]), 1);
      mbar_init(smem_u32(&bars->l_free[i]), 4);
      mbar_init(smem_u32(&bars->p_full[i]), 1);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
      mbar_init(smem_u32(&bars->l_full[i]), 1);
    }
    mbar_init(smem_u32(&bars->corr_done[0]), 128);
    mbar_init(smem_u32(&bars->corr_done[1]), 128);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->o_free), 128);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 0 && lane == 0 && !kFp8) tma_prefetch_desc(&kv_map);
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;
  const volatile int* abort_flag = &bars->abort_flag;

  const int c = static_cast<int>(cluster_id_x());
  const int W = __ldg(a.hdr + kHdrW);
  SegIter it0;
  it0.pre = a.pre;
  it0.U = a.U;
  it0.B = a.B;
  it0.ovh = a.overhead;
  it0.c = c;
  it0.lo_c = c * W;
  it0.hi_c = c * W + W;
  it0.u = __ldg(a.cl_first + c);

  const int nbox = scorer ? 9 : 8;                 // 64-channel boxes this CTA needs per page
  const int stage_bytes = scorer ? kStageS : kStageO;

  if (warp == 0) {
    // ---------------------------------------------------------------- loader
    // The whole warp walks the segments; lane 0 waits and issues the copies.
    // Page ids are read 32 at a time (one per lane) and shuffled out.
    SegIter it = it0;
    Seg s;
    // L2 prefetch of a segment's Q rows (contiguous), one segment ahead.
    auto prefetch_q = [&](const Seg& sg) {
      if (!scorer || lane != 0 || sg.empty) return;
      const int r0 = sg.rb * kRowsPerBlock;
      const int rows = min(kRowsPerBlock, a.R - r0);
      const uint8_t* base = reinterpret_cast<const uint8_t*>(a.q + (static_cast<size_t>(sg.b) * a.R + r0) * kDqk);
      const uint32_t total = static_cast<uint32_t>(rows) * kDqk * 2;
      for (uint32_t off = 0; off < total; off += 16384) prefetch_l2(base + off, min(16384u, total - off));
    };
    {
      SegIter look = it;
      Seg first;
      while (look.next(first))
        if (!first.empty) {
          prefetch_q(first);
          break;
        }
    }
    int stage = 0;
    uint32_t ph = 0;
    int last_par[kStages];
    for (int i = 0; i < kStages; ++i) last_par[i] = -1;
    bool ok = true;
    const uint32_t bytes = static_cast<uint32_t>(nbox * kBox);
    while (ok && it.next(s)) {
      if (s.empty) continue;
      {
        SegIter look = it;
        Seg nx;
        while (look.next(nx))
          if (!nx.empty) {
            prefetch_q(nx);
            break;
          }
      }
      if (kFp8) continue;  // the fp8 variant's dequant warps read pages themselves
      const int32_t* bt = a.block_table + static_cast<size_t>(s.b) * a.max_pages;
      for (int p0 = s.page_lo; ok && p0 < s.page_hi; p0 += 32) {
        const int my_p = p0 + lane;
        const int my_pid = my_p < s.page_hi ? __ldg(bt + my_p) : 0;
        const int cnt = min(32, s.page_hi - p0);
        for (int k = 0; k < cnt; ++k) {
          int pid = __shfl_sync(0xffffffffu, my_pid, k);
          if (lane == 0) {
            if (!mbar_wait(smem_u32(&bars->kv_empty[stage]), ph ^ 1u, abort_flag)) {
              ok = false;
              if (!*abort_flag) signal_abort(bars, a.err, peer);
            } else {
              if (pid < 0 || pid >= a.num_pages) {
                atomicOr(a.err, kErrBounds);
                pid = a.num_pages;  // outside the tensor map: TMA fills zeros, no fault
              }
              const uint32_t fb = smem_u32(&bars->kv_full[stage]);
              mbar_arrive_expect_tx(fb, bytes);
              uint8_t* dst = smem + stage * stage_bytes;
              for (int x = 0; x < nbox; ++x) tma_load_3d(smem_u32(dst + x * kBox), &kv_map, 64 * x, 0, pid, fb);
              last_par[stage] = static_cast<int>(ph);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // wait (time-bounded only) for the loads already in flight
      for (int i = 0; i < kStages; ++i)
        if (last_par[i] >= 0) mbar_wait(smem_u32(&bars->kv_full[i]), static_cast<uint32_t>(last_par[i]), nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    SegIter it = it0;
    Seg s;
    int stage = 0;
    uint32_t ph = 0, q_ph = 0, ofree_ph = 0;
    uint32_t t = 0;  // tile counter over the whole kernel
    bool ok = true;
    if (scorer) {
      // S[b] = Q K^T: 36 steps of K=16 over the 576 channels, A = Q in TMEM.
      const uint32_t idesc = idesc_f16_f32(128, 64, false, false, !kFp8);
      while (ok && it.next(s)) {
        if (s.empty) continue;
        if (!mbar_wait(smem_u32(&bars->q_full), q_ph, abort_flag)) { ok = false; break; }
        q_ph ^= 1u;
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t & 1u, sph = (t >> 1) & 1u;
          if (!mbar_wait(smem_u32(&bars->kv_full[stage]), ph, abort_flag)) { ok = false; break; }
          if (!mbar_wait(smem_u32(&bars->s_free[sb]), sph ^ 1u, abort_flag)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t b0 = smem_desc_sw128(smem_u32(smem + stage * kStageS), 16, 1024);
            const uint32_t dcol = tbase + (sb ? kColS1 : kColS0);
#pragma unroll
            for (int k = 0; k < 36; ++k)
              mma_ts(dcol, tbase + kColQ + 8 * k, b0 + static_cast<uint64_t>(((k >> 2) * kBox + (k & 3) * 32) >> 4),
                     idesc, k > 0 ? 1u : 0u);
            mma_commit(smem_u32(&bars->s_full[sb]));
            mma_commit(smem_u32(&bars->kv_empty[stage]));
          }
          __syncwarp();
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    } else {
      // O += P V: 4 steps of K=16 keys, two N=256 halves, A = P from shared memory.
      const uint32_t idesc = idesc_f16_f32(128, 256, false, true, !kFp8);
      while (ok && it.next(s)) {
        if (s.empty) continue;
        const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t & 1u;
          if (!mbar_wait(smem_u32(&bars->kv_full[stage]), ph, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + stage * kStageO;
          if (!kFp8) {
            const int valid = seqlen - j * kPage;
            if (valid < kPage) zero_tail_rows(st, valid > 0 ? valid : 0, 8, lane);
            __syncwarp();
          }
          if (!mbar_wait(smem_u32(&bars->corr_done[sb]), (t >> 1) & 1u, abort_flag)) { ok = false; break; }
          if (j == s.page_lo) {
            if (!mbar_wait(smem_u32(&bars->o_free), ofree_ph ^ 1u, abort_flag)) { ok = false; break; }
            ofree_ph ^= 1u;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint64_t pa = smem_desc_sw128(smem_u32(smem + kOffP + sb * kPBytes), 16, 1024);
            const uint64_t vb = smem_desc_sw128(smem_u32(st), 8192, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
              for (int h = 0; h < 2; ++h)
                mma_ss(tbase + 256 * h, pa + static_cast<uint64_t>((k * 32) >> 4),
                       vb + static_cast<uint64_t>((h * 4 * kBox + k * 2048) >> 4), idesc,
                       (j > s.page_lo || k > 0) ? 1u : 0u);
            mma_commit(smem_u32(&bars->kv_empty[stage]));
            mma_commit(smem_u32(&bars->pv_done[sb]));
            if (j + 1 == s.page_hi) mma_commit(smem_u32(&bars->o_full));
          }
          __syncwarp();
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && !*abort_flag && lane == 0) signal_abort(bars, a.err, peer);
    if (lane == 0) {
      mma_commit(smem_u32(&bars->drain));
      mbar_wait(smem_u32(&bars->drain), 0u, nullptr);
    }
    __syncwarp();
  } else if (warp < 6) {
    const int wq = warp & 3;
    const int L = wq * 32 + lane;  // query row within the block == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int ctid = tid - 64;     // 0..127
    SegIter it = it0;
    Seg s;
    uint32_t t = 0, seg_n = 0;
    bool ok = true;
    if (scorer) {
      // ------------------------------------------------------------ softmax (scorer)
      const uint32_t rP = mapa_shared(smem_u32(smem + kOffP), peer);
      const uint32_t rAlpha = mapa_shared(smem_u32(smem + kOffAlpha), peer);
      const uint32_t rL = mapa_shared(smem_u32(smem + kOffL), peer);
      const uint32_t rPfull0 = mapa_shared(smem_u32(&bars->p_full[0]), peer);
      const uint32_t rPfull1 = mapa_shared(smem_u32(&bars->p_full[1]), peer);
      const uint32_t rLfull0 = mapa_shared(smem_u32(&bars->l_full[0]), peer);
      const uint32_t rLfull1 = mapa_shared(smem_u32(&bars->l_full[1]), peer);
      uint32_t q_loaded = 0;
      float qmul = 1.f, qmul_next = 1.f;

      // Q row of this thread -> TMEM (all 576 channels, A operand of QK).  The
      // fp8-cache variant computes in fp16: the row is scaled by a power of
      // two so |q| <= 16384 (no overflow), undone on the scores.
      auto load_q = [&](const Seg& sg) -> float {
        const int r = sg.rb * kRowsPerBlock + L;
        const bool valid = r < a.R;
        const uint4* row =
            reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(sg.b) * a.R + (valid ? r : 0)) * kDqk);
        float qs = 1.f, qm = 1.f;
        if (kFp8 && valid) {
          float amax = 0.f;
          for (int v = 0; v < kDqk / 8; ++v) {
            const uint4 x = __ldg(row + v);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(x.x)), fabsf(bf16_hi(x.x))),
                                     fmaxf(fabsf(bf16_lo(x.y)), fabsf(bf16_hi(x.y)))));
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(bf16_lo(x.z)), fabsf(bf16_hi(x.z))),
                                     fmaxf(fabsf(bf16_lo(x.w)), fabsf(bf16_hi(x.w)))));
          }
          int k = 0;
          while (k < 126 && amax * ldexpf(1.f, -k) > 16384.f) ++k;
          qs = ldexpf(1.f, -k);
          qm = ldexpf(1.f, k);
        }
        for (int c2 = 0; c2 < 9; c2 += 2) {  // two 64-channel chunks of loads in flight
          uint4 x[16];
#pragma unroll
          for (int v = 0; v < 16; ++v)
            x[v] = (valid && (c2 + (v >> 3)) < 9) ? __ldg(row + c2 * 8 + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (c2 + h >= 9) break;
            uint32_t w[32];
#pragma unroll
            for (int v = 0; v < 8; ++v) {
              uint4 y = x[8 * h + v];
              if (kFp8) {
                y.x = pack_f16x2(bf16_lo(y.x) * qs, bf16_hi(y.x) * qs);
                y.y = pack_f16x2(bf16_lo(y.y) * qs, bf16_hi(y.y) * qs);
                y.z = pack_f16x2(bf16_lo(y.z) * qs, bf16_hi(y.z) * qs);
                y.w = pack_f16x2(bf16_lo(y.w) * qs, bf16_hi(y.w) * qs);
              }
              w[4 * v + 0] = y.x;
              w[4 * v + 1] = y.y;
              w[4 * v + 2] = y.z;
              w[4 * v + 3] = y.w;
            }
            tmem_st32(tbase + lane_off + kColQ + 32 * (c2 + h), w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->q_full));
        return qm;
      };

      while (ok && it.next(s)) {
        const int r = s.rb * kRowsPerBlock + L;
        const bool row_valid = r < a.R;
        const size_t out_row = static_cast<size_t>(s.b) * a.R + r;
        if (s.empty) {
          if (row_valid) a.lse[out_row] = -INFINITY;
          continue;
        }
        const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
        int n_vis = 0;
        if (row_valid) {
          n_vis = seqlen - a.s_q + r / a.H + 1;
          n_vis = n_vis < 0 ? 0 : (n_vis > seqlen ? seqlen : n_vis);
        }
        qmul = q_loaded ? qmul_next : load_q(s);
        q_loaded = 0;
        const float row_scale = a.scale_log2 * qmul;
        float m_ref = -INFINITY, l = 0.f;
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t & 1u, sph = (t >> 1) & 1u;
          if (!mbar_wait(smem_u32(&bars->s_full[sb]), sph, abort_flag)) { ok = false; break; }
          tc_fence_after();
          float x[64];
          {
            uint32_t v0[32], v1[32];
            const uint32_t col = tbase + lane_off + (sb ? kColS1 : kColS0);
            tmem_ld32(col, v0);
            tmem_ld32(col + 32, v1);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->s_free[sb]));
            const int nv = n_vis - j * kPage;  // keys of this page visible to the row
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = i < nv ? __uint_as_float(v0[i]) * row_scale : -INFINITY;
              x[32 + i] = 32 + i < nv ? __uint_as_float(v1[i]) * row_scale : -INFINITY;
            }
          }
          const float mt = max64(x);
          float alpha = 1.f;
          if (mt > m_ref + kRescaleLog2) {
            if (m_ref != -INFINITY) {
              alpha = ex2_approx(m_ref - mt);
              l *= alpha;
            }
            m_ref = mt;
          }
          uint32_t pk[32];
          float ps[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) ps[i] = 0.f;
          if (m_ref == -INFINITY) {
#pragma unroll
            for (int v = 0; v < 32; ++v) pk[v] = 0u;
          } else {
#pragma unroll
            for (int v = 0; v < 32; ++v) {
              const float p0 = ex2_approx(x[2 * v] - m_ref);
              const float p1 = ex2_approx(x[2 * v + 1] - m_ref);
              ps[v & 7] += p0 + p1;
              pk[v] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
          }
          l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));

          // P tile t and the factor to the accumulator (its buffer sb must be free)
          if (!mbar_wait(smem_u32(&bars->pbuf_free[sb]), sph ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t pbar = sb ? rPfull1 : rPfull0;
          const uint32_t prow = rP + sb * kPBytes + L * 128;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc)
            st_async_v4_u32(prow + ((cc ^ (L & 7)) << 4), pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3],
                            pbar);
          st_async_f32(rAlpha + sb * kVecBytes + L * 4, alpha, pbar);
        }
        if (!ok) break;

        // Q of the next segment with pages can go in now (its QK overlaps the
        // accumulator's last PV and epilogue of this one).
        {
          SegIter look = it;
          Seg nx;
          while (look.next(nx)) {
            if (!nx.empty) {
              qmul_next = load_q(nx);
              q_loaded = 1;
              break;
            }
          }
        }

        // lse here; the row sum goes to the accumulator for its epilogue
        const float lse_v = l > 0.f ? (m_ref + lg2_approx(l)) * kLn2 : -INFINITY;
        if (row_valid) {
          if (s.split)
            a.lse_part[static_cast<size_t>(s.slot) * kRowsPerBlock + L] = lse_v;
          else
            a.lse[out_row] = lse_v;
        }
        const uint32_t lb = seg_n & 1u, lph = (seg_n >> 1) & 1u;
        if (!mbar_wait(smem_u32(&bars->l_free[lb]), lph ^ 1u, abort_flag)) { ok = false; break; }
        st_async_f32(rL + lb * kVecBytes + L * 4, l, lb ? rLfull1 : rLfull0);
        ++seg_n;
      }
    } else {
      // ------------------------------------------------------------ rescale + epilogue (accumulator)
      const float* alpha_s = reinterpret_cast<const float*>(smem + kOffAlpha);
      const float* l_s = reinterpret_cast<const float*>(smem + kOffL);
      const uint32_t rLfree0 = mapa_shared(smem_u32(&bars->l_free[0]), peer);
      const uint32_t rLfree1 = mapa_shared(smem_u32(&bars->l_free[1]), peer);
      uint32_t ofull_ph = 0;
      while (ok && it.next(s)) {
        const int r = s.rb * kRowsPerBlock + L;
        const bool row_valid = r < a.R;
        const size_t out_row = static_cast<size_t>(s.b) * a.R + r;
        if (s.empty) {
          if (row_valid) {
            uint4* o = reinterpret_cast<uint4*>(a.out + out_row * kDv);
            for (int v = 0; v < kDv / 8; ++v) o[v] = make_uint4(0, 0, 0, 0);
          }
          continue;
        }
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t & 1u, sph = (t >> 1) & 1u;
          if (ctid == 0) mbar_arrive_expect_tx(smem_u32(&bars->p_full[sb]), kPBytes + kVecBytes);
          if (!mbar_wait<true>(smem_u32(&bars->p_full[sb]), sph, abort_flag)) { ok = false; break; }
          const float alpha = alpha_s[sb * kRowsPerBlock + L];
          if (__any_sync(0xffffffffu, alpha != 1.f) && j > s.page_lo) {
            // O must hold PV of the previous tile before it is rescaled
            const uint32_t pb = (t - 1u) & 1u, pph = ((t - 1u) >> 1) & 1u;
            if (!mbar_wait(smem_u32(&bars->pv_done[pb]), pph, abort_flag)) { ok = false; break; }
            tc_fence_after();
            for (int ch = 0; ch < 16; ++ch) {
              uint32_t o[32];
              tmem_ld32(tbase + lane_off + 32 * ch, o);
              tmem_wait_ld();
#pragma unroll
              for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
              tmem_st32(tbase + lane_off + 32 * ch, o);
            }
            tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->corr_done[sb]));
        }
        if (!ok) break;

        // epilogue: O / l -> out (bf16) or the fp32 partial slot
        if (!mbar_wait(smem_u32(&bars->o_full), ofull_ph, abort_flag)) { ok = false; break; }
        ofull_ph ^= 1u;
        const uint32_t lb = seg_n & 1u, lph = (seg_n >> 1) & 1u;
        if (ctid == 0) mbar_arrive_expect_tx(smem_u32(&bars->l_full[lb]), kVecBytes);
        if (!mbar_wait<true>(smem_u32(&bars->l_full[lb]), lph, abort_flag)) { ok = false; break; }
        const float l = l_s[lb * kRowsPerBlock + L];
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(lb ? rLfree1 : rLfree0);
        ++seg_n;
        tc_fence_after();
        const float inv_l = l > 0.f ? 1.f / l : 0.f;
        for (int ch = 0; ch < 16; ++ch) {
          uint32_t o[32];
          tmem_ld32(tbase + lane_off + 32 * ch, o);
          tmem_wait_ld();
          if (row_valid) {
            if (s.split) {
              float4* dst = reinterpret_cast<float4*>(a.o_part + (static_cast<size_t>(s.slot) * kRowsPerBlock + L) * kDv +
                                                      32 * ch);
#pragma unroll
              for (int v = 0; v < 8; ++v)
                dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                     __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(a.out + out_row * kDv + 32 * ch);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l);
                w.y = pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l);
                w.z = pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l);
                w.w = pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l);
                dst[v] = w;
              }
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->o_free));
      }
    }
    if (!ok && !*abort_flag) signal_abort(bars, a.err, peer);
  } else if (warp == 6) {
    // ---------------------------------------------------------------- credit relay (accumulator)
    // After PV of tile t, P buffer t%2 may be refilled by the scorer.
    if (!scorer && lane == 0) {
      const uint32_t rFree0 = mapa_shared(smem_u32(&bars->pbuf_free[0]), peer);
      const uint32_t rFree1 = mapa_shared(smem_u32(&bars->pbuf_free[1]), peer);
      SegIter it = it0;
      Seg s;
      uint32_t t = 0;
      bool ok = true;
      while (ok && it.next(s)) {
        if (s.empty) continue;
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t & 1u;
          if (!mbar_wait(smem_u32(&bars->pv_done[sb]), (t >> 1) & 1u, abort_flag)) { ok = false; break; }
          mbar_arrive_remote(sb ? rFree1 : rFree0);
        }
      }
      if (!ok && !*abort_flag) signal_abort(bars, a.err, peer);
    }
    __syncwarp();
  } else if (kFp8) {
    // ---------------------------------------------------------------- fp8 dequant (warps 7-10)
    // e4m3 x scale -> fp16 in the ring, swizzled as the MMA descriptors expect;
    // rows past seqlen are written as zeros.
    const int dq = tid - 224;  // 0..127
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(a.kv);
    SegIter it = it0;
    Seg s;
    int stage = 0;
    uint32_t ph = 0;
    bool ok = true;
    const int per_tok = nbox * 8;              // 16-byte output chunks per token
    const int chunks = kPage * per_tok;        // per page
    while (ok && it.next(s)) {
      if (s.empty) continue;
      const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
      const int32_t* bt = a.block_table + static_cast<size_t>(s.b) * a.max_pages;
      for (int p = s.page_lo; p < s.page_hi; ++p) {
        int pid = __ldg(bt + p);
        bool bad = pid < 0 || pid >= a.num_pages;
        if (bad) {
          if (dq == 0) atomicOr(a.err, kErrBounds);
          pid = 0;
        }
        const int valid = bad ? 0 : seqlen - p * kPage;
        uint8_t* dst = smem + stage * stage_bytes;
        bool out_of_range = false;
        // two halves of up to 18 chunks per thread: loads of a half first, then
        // conversion and stores (one 8-byte e4m3 group + its scale per chunk)
        for (int half = 0; half < 2 && ok; ++half) {
          uint2 raw[18];
          float scl[18];
#pragma unroll
          for (int i = 0; i < 18; ++i) {
            const int q = dq + 128 * (18 * half + i);
            raw[i] = make_uint2(0, 0);
            scl[i] = 0.f;
            if (q < chunks) {
              const int tok = q / per_tok, rem = q - tok * per_tok;
              if (tok < valid) {
                const int ch = rem * 8;
                const size_t row = static_cast<size_t>(pid) * kPage + tok;
                raw[i] = __ldg(reinterpret_cast<const uint2*>(kv8 + row * kDqk + ch));
                scl[i] = __ldg(a.kv_scales + row * kGroups + (ch < 512 ? (ch >> 7) : 4));
              }
            }
          }
          if (half == 0 && !mbar_wait(smem_u32(&bars->kv_empty[stage]), ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int i = 0; i < 18; ++i) {
            const int q = dq + 128 * (18 * half + i);
            if (q >= chunks) break;
            const int tok = q / per_tok, rem = q - tok * per_tok;
            const int box = rem >> 3, c8 = rem & 7;
            const float sv = scl[i];
            out_of_range |= !(fabsf(sv) * 448.f <= 65504.f);
            float f[8];
            e4m3x2_to_f32(static_cast<uint16_t>(raw[i].x & 0xFFFFu), f[0], f[1]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw[i].x >> 16), f[2], f[3]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw[i].y & 0xFFFFu), f[4], f[5]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw[i].y >> 16), f[6], f[7]);
            uint4 w;
            w.x = pack_f16x2(f[0] * sv, f[1] * sv);
            w.y = pack_f16x2(f[2] * sv, f[3] * sv);
            w.z = pack_f16x2(f[4] * sv, f[5] * sv);
            w.w = pack_f16x2(f[6] * sv, f[7] * sv);
            *reinterpret_cast<uint4*>(dst + box * kBox + tok * 128 + ((c8 ^ (tok & 7)) << 4)) = w;
          }
        }
        if (!ok) break;
        if (out_of_range) atomicOr(a.err, kErrRange);
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars->kv_full[stage]));
        if (++stage == kStages) {
          stage = 0;
          ph ^= 1u;
        }
      }
    }
    if (!ok && !*abort_flag) signal_abort(bars, a.err, peer);
  }

  __syncwarp();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace

int decode_smem_bytes(bool) { return kSmem; }

static cudaLaunchConfig_t make_cfg(bool fp8, int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(fp8 ? Cfg<true>::kThreads : Cfg<false>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

static cudaError_t set_smem_attr(bool fp8) {
  if (fp8) return cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  return cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t decode_max_active_clusters(bool fp8, int* clusters) {
  cudaError_t e = set_smem_attr(fp8);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(fp8, 1, nullptr, attr);
  if (fp8) return cudaOccupancyMaxActiveClusters(clusters, mla_decode_kernel<true>, &cfg);
  return cudaOccupancyMaxActiveClusters(clusters, mla_decode_kernel<false>, &cfg);
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kv_map, int clusters, bool fp8,
                          cudaStream_t stream) {
  cudaError_t e = set_smem_attr(fp8);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = make_cfg(fp8, clusters, stream, attr);
  if (fp8) return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true>, kv_map, a);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false>, kv_map, a);
}

}  // namespace mla_gb300
