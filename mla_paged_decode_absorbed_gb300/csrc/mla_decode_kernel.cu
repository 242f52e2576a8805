// MLA paged decode, absorbed form: the attention kernel for sm_103a.
//
// What it computes (PaddleNLP issue #10157, "Multi-head Latent Attention (MLA)
// 算子 / 总体概述"): per 64-token KV page, Data Load -> QK GEMM -> Softmax Update
// (+ P written where the next MMA reads it) -> PV GEMM, with num_token > 1 per
// request (the MTP verify step of the same page, causal within the new tokens).
//
// Design for GB300 (the pages' three Hopper warp-group schemes are prior art):
//
// * One work unit is 128 query rows (token-major (i, h) rows of one request)
//   times a contiguous range of that request's pages.  It runs on a cluster of
//   two CTAs that split the channels: rank 0 owns latent channels [0,256),
//   rank 1 owns [256,512) plus the 64 RoPE channels.  Each CTA loads only its
//   channel slice of every page (every cache byte crosses HBM once), computes
//   a partial S = Q_slice K_slice^T, and the two partials are exchanged through
//   distributed shared memory (st.async) so both CTAs hold the same fp32 S.
//   Both then run the identical online softmax and each accumulates its own 256
//   output channels O += P V_slice.
// * Why the split: the 128 x 512 fp32 output accumulator alone fills a CTA's
//   512 TMEM columns; with 256 columns per CTA, Q (A operand, from TMEM so the
//   tensor core reads only K/V from shared memory), S and P fit beside it.
//   TMEM columns: O [0,256), Q [256,416), S [416,480), P [480,512).
// * Warp roles per CTA: warp 0 issues TMA loads of page slices into a 4-stage
//   shared-memory ring (page ids read from the block table); warp 1 issues
//   tcgen05 MMAs (one elected lane) and zeroes cache slots past seqlen in the
//   last page; warps 2-5 (one TMEM lane quarter each, one query row per thread)
//   run the exchange, the fp32 online softmax and the epilogue.  The fp8 cache
//   variant adds warps 6-9 that dequantise e4m3 x scale into the bf16 ring.
// * Online softmax in base 2 with a lazy rescale: the running max only moves
//   (and O is only rescaled in TMEM) when a tile's max exceeds it by more than
//   8 (a factor 256); the final division by the row sum is exact either way.
//   This trick is from FlashAttention-4 (Dao et al., 2025), not the pages.
// * Every barrier wait is bounded (about one second); a timeout sets an error
//   bit, tells the peer CTA to stop, and the kernel tears down normally.
#include <cuda_bf16.h>
#include <cstdint>

#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla_gb300 {
namespace {

using namespace mla_sm103;

constexpr int kBoxBf16 = 64 * 64 * 2;       // one 64-token x 64-channel bf16 box
constexpr int kBoxFp8 = 64 * 64;            // the same box in e4m3
constexpr int kMaxBoxes = 5;                // rank 1: channels 256..575
constexpr int kStageBytes = kMaxBoxes * kBoxBf16;
constexpr int kXBytes = kRowsPerBlock * 64 * 4;   // one fp32 partial-S tile
constexpr int kScaleBytes = kPage * kGroups * 4;  // 1280

constexpr uint32_t kColO = 0, kColQ = 256, kColS = 416, kColP = 480;
constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;

template <bool kFp8>
struct Cfg {
  static constexpr int kStages = kFp8 ? 2 : 4;         // bf16 ring
  static constexpr int kF8Stages = kFp8 ? 3 : 0;       // e4m3 staging ring
  static constexpr int kF8StageBytes = kMaxBoxes * kBoxFp8 + kScaleBytes;
  static constexpr int kThreads = kFp8 ? 320 : 192;
  static constexpr int kOffStages = 0;
  static constexpr int kOffX = kStages * kStageBytes;
  static constexpr int kOffF8 = kOffX + 2 * kXBytes;
  static constexpr int kOffBars = kOffF8 + kF8Stages * kF8StageBytes;
  static constexpr int kBarBytes = 512;
  static constexpr int kSmem = 1024 + kOffBars + kBarBytes;
};

template <bool kFp8>
struct Bars {
  uint64_t kv_full[Cfg<kFp8>::kStages];
  uint64_t kv_empty[Cfg<kFp8>::kStages];
  uint64_t f8_full[kFp8 ? Cfg<kFp8>::kF8Stages : 1];
  uint64_t f8_empty[kFp8 ? Cfg<kFp8>::kF8Stages : 1];
  uint64_t q_full, s_full, s_free, p_full, p_free, o_full, o_free, drain;
  uint64_t x_full[2];
  int abort_flag;
  uint32_t tmem_base;
};
static_assert(sizeof(Bars<true>) <= Cfg<true>::kBarBytes, "barrier block too large");
static_assert(Cfg<false>::kSmem <= 232448, "bf16 kernel exceeds shared memory");
static_assert(Cfg<true>::kSmem <= 232448, "fp8 kernel exceeds shared memory");

// One segment of a cluster's cost range: unit u (row block rb of request b),
// pages [page_lo, page_hi) of it.  `empty` units have no visible keys.
struct Seg {
  int u, b, rb, page_lo, page_hi, split, slot, empty;
};

// Walks the units of cluster c in order (the plan's partition rule: see mla_plan).
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

template <bool kFp8>
__device__ __forceinline__ void signal_abort(Bars<kFp8>* bars, int32_t* err, uint32_t peer) {
  atomicOr(err, kErrTimeout);
  bars->abort_flag = 1;
  st_cluster_u32(mapa_shared(smem_u32(&bars->abort_flag), peer), 1u);
}

// Zero key rows [valid, 64) of every box of a bf16 stage (cache slots past
// seqlen may hold anything, including NaN; a masked weight of 0 times NaN would
// still poison the PV product).  Whole 128-byte rows, so the swizzle is moot.
__device__ __forceinline__ void zero_tail_rows(uint8_t* stage, int valid, int nbox, int lane) {
  const int per_box = (kPage - valid) * 8;
  const int total = per_box * nbox;
  for (int i = lane; i < total; i += 32) {
    const int box = i / per_box, rem = i - box * per_box;
    const int row = valid + (rem >> 3), ch = rem & 7;
    *reinterpret_cast<uint4*>(stage + box * kBoxBf16 + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
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

template <bool kFp8>
__global__ void __launch_bounds__(Cfg<kFp8>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map, const DecodeArgs a) {
  using C = Cfg<kFp8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem + C::kOffStages;
  float* xbuf = reinterpret_cast<float*>(smem + C::kOffX);
  uint8_t* f8st = smem + C::kOffF8;
  Bars<kFp8>* bars = reinterpret_cast<Bars<kFp8>*>(smem + C::kOffBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int nbox = rank ? 5 : 4;            // 64-channel boxes of this CTA's slice
  const int ch0 = rank ? 256 : 0;           // first channel of the slice
  const int nk = nbox * 4;                  // K=16 steps of the QK MMA

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&bars->kv_full[s]), kFp8 ? 128 : 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), 1);
    }
    if (kFp8) {
      for (int s = 0; s < C::kF8Stages; ++s) {
        mbar_init(smem_u32(&bars->f8_full[s]), 1);
        mbar_init(smem_u32(&bars->f8_empty[s]), 128);
      }
    }
    mbar_init(smem_u32(&bars->q_full), 128);
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), 128);
    mbar_init(smem_u32(&bars->p_full), 128);
    mbar_init(smem_u32(&bars->p_free), 1);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->o_free), 128);
    mbar_init(smem_u32(&bars->drain), 1);
    mbar_init(smem_u32(&bars->x_full[0]), 1);
    mbar_init(smem_u32(&bars->x_full[1]), 1);
    bars->abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 0 && lane == 0) tma_prefetch_desc(&kv_map);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp walks the segments; lane 0 waits and issues the copies.
    // Page ids are read 32 at a time (one per lane) and shuffled out, so the
    // block-table read is off the per-page critical path.
    SegIter it = it0;
    Seg s;
    int stage = 0;
    uint32_t ph = 0;
    int last_par[kFp8 ? C::kF8Stages : C::kStages];
    for (int i = 0; i < (kFp8 ? C::kF8Stages : C::kStages); ++i) last_par[i] = -1;
    bool ok = true;
    const uint32_t bytes = kFp8 ? (uint32_t)(nbox * kBoxFp8 + kScaleBytes) : (uint32_t)(nbox * kBoxBf16);
    // L2 prefetch of a segment's Q rows (one request's block of <= 128 rows is
    // contiguous), so the softmax warps' Q loads at the segment start hit L2.
    auto prefetch_q = [&](const Seg& sg) {
      if (lane != 0 || sg.empty) return;
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
      const int32_t* bt = a.block_table + static_cast<size_t>(s.b) * a.max_pages;
      for (int p0 = s.page_lo; ok && p0 < s.page_hi; p0 += 32) {
        const int my_p = p0 + lane;
        const int my_pid = my_p < s.page_hi ? __ldg(bt + my_p) : 0;
        const int cnt = min(32, s.page_hi - p0);
        for (int k = 0; k < cnt; ++k) {
          int pid = __shfl_sync(0xffffffffu, my_pid, k);
          if (lane == 0) {
            uint64_t* empty_bar = kFp8 ? &bars->f8_empty[stage] : &bars->kv_empty[stage];
            uint64_t* full_bar = kFp8 ? &bars->f8_full[stage] : &bars->kv_full[stage];
            if (!mbar_wait(smem_u32(empty_bar), ph ^ 1u, abort_flag)) {
              ok = false;
              if (!*abort_flag) signal_abort(bars, a.err, peer);
            } else {
              int scale_pid = pid;
              if (pid < 0 || pid >= a.num_pages) {
                atomicOr(a.err, kErrBounds);
                pid = a.num_pages;  // outside the tensor map: TMA fills zeros, no fault
                scale_pid = 0;
              }
              mbar_arrive_expect_tx(smem_u32(full_bar), bytes);
              if (kFp8) {
                uint8_t* dst = f8st + stage * C::kF8StageBytes;
                for (int x = 0; x < nbox; ++x)
                  tma_load_3d(smem_u32(dst + x * kBoxFp8), &kv_map, ch0 + 64 * x, 0, pid, smem_u32(full_bar));
                bulk_load(smem_u32(dst + kMaxBoxes * kBoxFp8),
                          a.kv_scales + static_cast<size_t>(scale_pid) * kPage * kGroups, kScaleBytes,
                          smem_u32(full_bar));
              } else {
                uint8_t* dst = stages + stage * kStageBytes;
                for (int x = 0; x < nbox; ++x)
                  tma_load_3d(smem_u32(dst + x * kBoxBf16), &kv_map, ch0 + 64 * x, 0, pid, smem_u32(full_bar));
              }
              last_par[stage] = static_cast<int>(ph);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (++stage == (kFp8 ? C::kF8Stages : C::kStages)) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // wait (time-bounded only) for the loads already in flight
      for (int i = 0; i < (kFp8 ? C::kF8Stages : C::kStages); ++i)
        if (last_par[i] >= 0)
          mbar_wait(smem_u32(kFp8 ? &bars->f8_full[i] : &bars->kv_full[i]), (uint32_t)last_par[i], nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    SegIter it = it0;
    Seg s;
    int stage = 0;
    uint32_t ph = 0, sfree_ph = 0, pfull_ph = 0, q_ph = 0, ofree_ph = 0;
    const uint32_t idesc_qk = idesc_f16_f32(128, 64, false, false, !kFp8);
    const uint32_t idesc_pv = idesc_f16_f32(128, 256, false, true, !kFp8);
    bool ok = true;
    while (ok && it.next(s)) {
      if (s.empty) continue;
      const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
      if (!mbar_wait(smem_u32(&bars->q_full), q_ph, abort_flag)) { ok = false; break; }
      q_ph ^= 1u;
      const int n = s.page_hi - s.page_lo;
      int prev_stage = 0;
      // Step j issues QK(j) (j < n) and PV(j-1) (j > 0), whichever becomes
      // ready first (QK first when both are): PV(j-1) never waits behind the
      // arrival of page j.  Lane 0 probes the barriers without suspending and
      // broadcasts, so the warp stays converged for the tail zeroing.
      for (int j = 0; j <= n && ok; ++j) {
        bool need_qk = j < n, need_pv = j > 0;
        bool kv_ok = false, sf_ok = false, pf_ok = false, of_ok = (j != 1);
        const uint64_t t0 = globaltimer_ns();
        uint32_t spins = 0;
        auto probe = [&](uint64_t* bar, uint32_t parity) -> bool {
          int r = 0;
          if (lane == 0) r = mbar_test_wait(smem_u32(bar), parity) ? 1 : 0;
          return __shfl_sync(0xffffffffu, r, 0) != 0;
        };
        while (need_qk || need_pv) {
          bool did = false;
          if (need_qk) {
            if (!kv_ok) kv_ok = probe(&bars->kv_full[stage], ph);
            if (kv_ok && !sf_ok) sf_ok = probe(&bars->s_free, sfree_ph ^ 1u);
            if (kv_ok && sf_ok) {
              sfree_ph ^= 1u;
              uint8_t* st = stages + stage * kStageBytes;
              if (!kFp8) {
                const int valid = seqlen - (s.page_lo + j) * kPage;
                if (valid < kPage) zero_tail_rows(st, valid > 0 ? valid : 0, nbox, lane);
                __syncwarp();
              }
              tc_fence_after();
              if (lane == 0) {
                const uint32_t sbase = smem_u32(st);
                for (int k = 0; k < nk; ++k) {
                  const uint64_t bd = smem_desc_sw128(sbase + (k >> 2) * kBoxBf16 + (k & 3) * 32, 16, 1024);
                  mma_ts(tbase + kColS, tbase + kColQ + 8 * k, bd, idesc_qk, k > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars->s_full));
              }
              __syncwarp();
              need_qk = false;
              did = true;
            }
          }
          if (need_pv) {
            if (!pf_ok) pf_ok = probe(&bars->p_full, pfull_ph);
            if (pf_ok && !of_ok) of_ok = probe(&bars->o_free, ofree_ph ^ 1u);
            if (pf_ok && of_ok) {
              pfull_ph ^= 1u;
              if (j == 1) ofree_ph ^= 1u;
              tc_fence_after();
              if (lane == 0) {
                const uint32_t vbase = smem_u32(stages + prev_stage * kStageBytes);
                for (int k = 0; k < 4; ++k) {
                  const uint64_t bd = smem_desc_sw128(vbase + k * 2048, 8192, 1024);
                  mma_ts(tbase + kColO, tbase + kColP + 8 * k, bd, idesc_pv, (j > 1 || k > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars->p_free));
                mma_commit(smem_u32(&bars->kv_empty[prev_stage]));
                if (j == n) mma_commit(smem_u32(&bars->o_full));
              }
              __syncwarp();
              need_pv = false;
              did = true;
            }
          }
          if (!did && ((++spins & 15u) == 0u)) {
            if (*abort_flag || globaltimer_ns() - t0 > kWaitNs) {
              ok = false;
              break;
            }
          }
        }
        if (!ok) break;
        if (j < n) {
          prev_stage = stage;
          if (++stage == C::kStages) {
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
    // ------------------------------------------------------------ softmax / epilogue
    const int wq = warp & 3;
    const int L = wq * 32 + lane;                  // query row within the block == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int sm_tid = tid - 64;
    const uint32_t x_remote = mapa_shared(smem_u32(xbuf), peer);
    const uint32_t xbar_remote0 = mapa_shared(smem_u32(&bars->x_full[0]), peer);
    const uint32_t xbar_remote1 = mapa_shared(smem_u32(&bars->x_full[1]), peer);
    SegIter it = it0;
    Seg s;
    uint32_t sfull_ph = 0, pfree_ph = 0, ofull_ph = 0;
    uint32_t tile_ctr = 0;
    bool q_loaded = false;
    bool ok = true;

    // Q slice of this thread's row -> TMEM (A operand of QK).  The fp8-cache
    // variant computes in fp16: the row is scaled by a power of two so that
    // |q| <= 16384 (no fp16 overflow; both CTAs see the whole row and pick the
    // same factor), and the returned multiplier undoes it on the scores.
    auto load_q = [&](const Seg& sg) -> float {
      const int r = sg.rb * kRowsPerBlock + L;
      const bool valid = r < a.R;
      const uint4* row = reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(sg.b) * a.R + (valid ? r : 0)) * kDqk);
      float qs = 1.f, qmul = 1.f;
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
        qmul = ldexpf(1.f, k);
      }
      const uint4* src = row + ch0 / 8;
      for (int c2 = 0; c2 < nbox; c2 += 2) {  // two 64-channel chunks of loads in flight
        uint4 x[16];
#pragma unroll
        for (int v = 0; v < 16; ++v)
          x[v] = (valid && (c2 + (v >> 3)) < nbox) ? __ldg(src + c2 * 8 + v) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (c2 + h >= nbox) break;
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
      return qmul;
    };
    float qmul = 1.f, qmul_next = 1.f;

    while (ok && it.next(s)) {
      const int r = s.rb * kRowsPerBlock + L;
      const bool row_valid = r < a.R;
      const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
      int n_vis = 0;
      if (row_valid) {
        n_vis = seqlen - a.s_q + r / a.H + 1;
        n_vis = n_vis < 0 ? 0 : (n_vis > seqlen ? seqlen : n_vis);
      }
      const size_t out_row = static_cast<size_t>(s.b) * a.R + r;
      if (s.empty) {
        if (row_valid) {
          uint4* o = reinterpret_cast<uint4*>(a.out + out_row * kDv + rank * 256);
          for (int v = 0; v < 32; ++v) o[v] = make_uint4(0, 0, 0, 0);
          if (rank == 0) a.lse[out_row] = -INFINITY;
        }
        continue;
      }
      qmul = q_loaded ? qmul_next : load_q(s);
      q_loaded = false;
      const float row_scale = a.scale_log2 * qmul;

      float m_ref = -INFINITY, l = 0.f;
      const int n = s.page_hi - s.page_lo;
      for (int j = 0; j < n; ++j) {
        if (!mbar_wait(smem_u32(&bars->s_full), sfull_ph, abort_flag)) { ok = false; break; }
        sfull_ph ^= 1u;
        tc_fence_after();
        uint32_t sa[32], sb[32];
        tmem_ld32(tbase + lane_off + kColS, sa);
        tmem_ld32(tbase + lane_off + kColS + 32, sb);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->s_free));

        // exchange partial S with the peer CTA
        const int xi = static_cast<int>(tile_ctr & 1u);
        const uint32_t xph = (tile_ctr >> 1) & 1u;
        if (sm_tid == 0) mbar_arrive_expect_tx(smem_u32(&bars->x_full[xi]), kXBytes);
        const uint32_t rrow = x_remote + xi * kXBytes + L * 256;
        const uint32_t rbar = xi ? xbar_remote1 : xbar_remote0;
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int pos = cc ^ (L & 15);
          const uint32_t* src = cc < 8 ? &sa[4 * cc] : &sb[4 * (cc - 8)];
          st_async_v4(rrow + pos * 16, __uint_as_float(src[0]), __uint_as_float(src[1]), __uint_as_float(src[2]),
                      __uint_as_float(src[3]), rbar);
        }
        if (!mbar_wait<true>(smem_u32(&bars->x_full[xi]), xph, abort_flag)) { ok = false; break; }
        const float4* lrow = reinterpret_cast<const float4*>(xbuf + xi * (kXBytes / 4) + L * 64);
        float sc[64];
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const float4 v = lrow[cc ^ (L & 15)];
          const uint32_t* own = cc < 8 ? &sa[4 * cc] : &sb[4 * (cc - 8)];
          sc[4 * cc + 0] = __uint_as_float(own[0]) + v.x;
          sc[4 * cc + 1] = __uint_as_float(own[1]) + v.y;
          sc[4 * cc + 2] = __uint_as_float(own[2]) + v.z;
          sc[4 * cc + 3] = __uint_as_float(own[3]) + v.w;
        }

        // mask, scale (base 2), running max with lazy rescale
        const int key0 = (s.page_lo + j) * kPage;
        const int nv = n_vis - key0;  // keys of this tile visible to the row
        float mt = -INFINITY;
#pragma unroll
        for (int cidx = 0; cidx < 64; ++cidx) {
          const float x = cidx < nv ? sc[cidx] * row_scale : -INFINITY;
          sc[cidx] = x;
          mt = fmaxf(mt, x);
        }
        float alpha = 1.f;
        bool rescale = false;
        if (mt > m_ref + kRescaleLog2) {
          if (m_ref != -INFINITY) {
            alpha = ex2_approx(m_ref - mt);
            l *= alpha;
            rescale = j > 0;
          }
          m_ref = mt;
        }
        uint32_t pk[32];
        float psum = 0.f;
        if (m_ref == -INFINITY) {
#pragma unroll
          for (int v = 0; v < 32; ++v) pk[v] = 0u;
        } else {
#pragma unroll
          for (int v = 0; v < 32; ++v) {
            const float p0 = ex2_approx(sc[2 * v] - m_ref);
            const float p1 = ex2_approx(sc[2 * v + 1] - m_ref);
            psum += p0 + p1;
            pk[v] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
          }
        }
        l += psum;

        if (!mbar_wait(smem_u32(&bars->p_free), pfree_ph ^ 1u, abort_flag)) { ok = false; break; }
        pfree_ph ^= 1u;
        tc_fence_after();
        if (__any_sync(0xffffffffu, rescale)) {
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t o[32];
            tmem_ld32(tbase + lane_off + kColO + 32 * ch, o);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 32; ++v) o[v] = __float_as_uint(__uint_as_float(o[v]) * alpha);
            tmem_st32(tbase + lane_off + kColO + 32 * ch, o);
          }
        }
        tmem_st32(tbase + lane_off + kColP, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->p_full));
        ++tile_ctr;
      }
      if (!ok) break;

      // Q of the next segment with pages can go in now: its QK runs while this
      // segment's last PV and epilogue finish.
      {
        SegIter look = it;
        Seg nx;
        while (look.next(nx)) {
          if (!nx.empty) {
            qmul_next = load_q(nx);
            q_loaded = true;
            break;
          }
        }
      }

      // epilogue: O / l -> out (bf16) or the fp32 partial slot
      if (!mbar_wait(smem_u32(&bars->o_full), ofull_ph, abort_flag)) { ok = false; break; }
      ofull_ph ^= 1u;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const float lse_v = l > 0.f ? (m_ref + lg2_approx(l)) * kLn2 : -INFINITY;
      for (int ch = 0; ch < 8; ++ch) {
        uint32_t o[32];
        tmem_ld32(tbase + lane_off + kColO + 32 * ch, o);
        tmem_wait_ld();
        if (row_valid) {
          if (s.split) {
            float4* dst = reinterpret_cast<float4*>(a.o_part + (static_cast<size_t>(s.slot) * kRowsPerBlock + L) * kDv +
                                                    rank * 256 + 32 * ch);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                   __uint_as_float(o[4 * v + 2]) * inv_l, __uint_as_float(o[4 * v + 3]) * inv_l);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(a.out + out_row * kDv + rank * 256 + 32 * ch);
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
      if (row_valid && rank == 0) {
        if (s.split)
          a.lse_part[static_cast<size_t>(s.slot) * kRowsPerBlock + L] = lse_v;
        else
          a.lse[out_row] = lse_v;
      }
    }
    if (!ok && !*abort_flag) signal_abort(bars, a.err, peer);
  } else if (kFp8) {
    // ------------------------------------------------------------ fp8 dequant (warps 6-9)
    const int dq = tid - 192;  // 0..127
    SegIter it = it0;
    Seg s;
    int fstage = 0, stage = 0;
    uint32_t fph = 0, ph = 0;
    bool ok = true;
    while (ok && it.next(s)) {
      if (s.empty) continue;
      const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
      for (int p = s.page_lo; p < s.page_hi; ++p) {
        if (!mbar_wait(smem_u32(&bars->f8_full[fstage]), fph, abort_flag)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&bars->kv_empty[stage]), ph ^ 1u, abort_flag)) { ok = false; break; }
        const uint8_t* src = f8st + fstage * C::kF8StageBytes;
        const float* scl = reinterpret_cast<const float*>(src + kMaxBoxes * kBoxFp8);
        uint8_t* dst = stages + stage * kStageBytes;
        const int valid = seqlen - p * kPage;
        const int chunks = kPage * nbox * 8;  // 16-byte fp16 output chunks
        bool out_of_range = false;
        for (int q = dq; q < chunks; q += 128) {
          const int tok = q / (nbox * 8);
          const int rem = q - tok * (nbox * 8);
          const int box = rem >> 3, c8 = rem & 7;
          uint4 w = make_uint4(0, 0, 0, 0);
          if (tok < valid) {
            const uint2 raw = *reinterpret_cast<const uint2*>(src + box * kBoxFp8 + tok * 64 + c8 * 8);
            const int ch = ch0 + box * 64 + c8 * 8;
            const float sv = scl[tok * kGroups + (ch < 512 ? (ch >> 7) : 4)];
            out_of_range |= !(fabsf(sv) * 448.f <= 65504.f);
            float f[8];
            e4m3x2_to_f32(static_cast<uint16_t>(raw.x & 0xFFFFu), f[0], f[1]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw.x >> 16), f[2], f[3]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw.y & 0xFFFFu), f[4], f[5]);
            e4m3x2_to_f32(static_cast<uint16_t>(raw.y >> 16), f[6], f[7]);
            w.x = pack_f16x2(f[0] * sv, f[1] * sv);
            w.y = pack_f16x2(f[2] * sv, f[3] * sv);
            w.z = pack_f16x2(f[4] * sv, f[5] * sv);
            w.w = pack_f16x2(f[6] * sv, f[7] * sv);
          }
          *reinterpret_cast<uint4*>(dst + box * kBoxBf16 + tok * 128 + ((c8 ^ (tok & 7)) << 4)) = w;
        }
        if (out_of_range) atomicOr(a.err, kErrRange);
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars->kv_full[stage]));
        mbar_arrive(smem_u32(&bars->f8_empty[fstage]));
        if (++fstage == C::kF8Stages) {
          fstage = 0;
          fph ^= 1u;
        }
        if (++stage == C::kStages) {
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

int decode_smem_bytes(bool fp8) { return fp8 ? Cfg<true>::kSmem : Cfg<false>::kSmem; }

static cudaLaunchConfig_t make_cfg(bool fp8, int clusters, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(fp8 ? Cfg<true>::kThreads : Cfg<false>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = decode_smem_bytes(fp8);
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
  if (fp8)
    return cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<true>::kSmem);
  return cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<false>::kSmem);
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
