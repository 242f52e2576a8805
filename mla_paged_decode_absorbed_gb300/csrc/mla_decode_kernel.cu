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
//       TMEM, computes S = Q K^T over each page with tcgen05 into one of three
//       TMEM score slots (bf16: two pages per MMA chain where they sit in
//       adjacent ring stages), runs the fp32 online softmax, and streams the
//       16-bit P tile plus a per-row rescale factor into the accumulator's
//       shared memory (st.async, 16.5 KB per page, one direction);
//     - the accumulator (rank 1) holds the 128 x 512 fp32 output in all 512 of
//       its TMEM columns and runs O += P V with P read from shared memory, the
//       (rare) O rescales and the epilogue.
//   Each CTA TMA-loads each page it needs with one copy into its own ring
//   (scorer: 576 channels, three stages, each segment's Q block passing
//   through the same ring; accumulator: 512 channels, two stages for bf16);
//   the second read of a page comes from L2.
// * Why this split: a 128 x 512 fp32 accumulator fills a whole SM's TMEM, and
//   distributed shared memory moves only ~21 bytes per clock per SM pair (as
//   measured on GB300), so exchanging fp32 partial scores (32 KB per page each
//   way) costs more than the page itself; forwarding 16-bit P costs half and
//   goes one way.
// * Roles per CTA: warp 0 loads pages (TMA, 32 block-table entries per read);
//   warp 1 allocates TMEM and issues the MMAs from one lane; warps 2-5 (one
//   TMEM lane quarter each, one query row per thread) run the softmax
//   (scorer) or the rescale and epilogue (accumulator).  The bf16 scorer
//   splits each row's softmax with warps 6-9 (keys 32..63 of a page), and
//   keeps arithmetic out of the MMA warp's SM sub-partition: warps 5 and 9
//   only copy rows 32..63's scores to shared memory, where warps 10 and 11
//   run their softmax.  The accumulator's PV commit multicasts the P-buffer
//   credit straight to the scorer's barrier.  The fp8-cache variant has the
//   loader bulk-copy each page's e4m3 bytes into the top of its ring stage,
//   and warps 6, 7, 8 and 10 (variant B: 9) of both CTAs rewrite the stage in
//   place as fp16 (the MMAs then run in fp16).
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
static_assert(kStageS == 64 * kDqk * 2, "half a Q row block fills one scorer stage");
// fp8 cache: each CTA TMA-loads the raw e4m3 chunks of every block it needs
// (64 tokens x 64 bytes each, 64-byte swizzled) into the top of its ring
// stage and rewrites the stage in place as fp16: the scorer as the exact
// codes (scales are applied to the scores in fp32), the accumulator as code x
// scale (its V).  Raw chunk c of a stage sits at kRaw*Off + c * kRawSlot.
constexpr int kRawSlot = 64 * 64;                  // one raw chunk: 64 tokens x 64 bytes
constexpr int kRawBytesS = 9 * kRawSlot;           // scorer, variant A: chunks 0..8
constexpr int kRawBytesSB = 10 * kRawSlot;         // scorer, variant B: 8 latent chunks + 2 bf16 RoPE chunks
constexpr int kRawBytesA = 8 * kRawSlot;           // accumulator: latent chunks 0..7
constexpr int kRawOffS = 9 * kBox - kRawBytesS;    // top of the scorer's 72 KB stage
constexpr int kRawOffSB = 9 * kBox - kRawBytesSB;
constexpr int kRawOffA = 8 * kBox - kRawBytesA;    // top of the accumulator's 64 KB stage
static_assert(kRawOffS % 1024 == 0 && kRawOffSB % 1024 == 0 && kRawOffA % 1024 == 0, "raw chunks 1024-aligned");
// fp8 scorer: QK runs per scale group g (channels [128g, 128g+128), the RoPE
// group 4 = [512, 576)) into a ring of kGroupSlots TMEM score buffers; the
// softmax adds scale[token][g] * S_g in fp32.
constexpr int kGroupSlots = 3;
constexpr int kScaleSlotBytes = kGroups * 64 * 4;  // [group][token] fp32, one slot per ring stage
constexpr int kPBytes = kRowsPerBlock * 64 * 2;    // P tile: 128 rows x 64 keys, SW128 K-major
constexpr int kVecBytes = kRowsPerBlock * 4;       // one fp32 per row
constexpr int kPartBytes = kPartChunks * kRowsPerBlock * 16;  // one fp16 partial slot (128 KB)
// The accumulator's V ring and its P tiles in flight.  bf16: its V reads
// hit L2 (the scorer read the page shortly before), so two stages cover
// their latency, and the freed 64 KB hold four P tiles: the scorer may run
// up to four tiles ahead of PV.  fp8: three stages (each also holds the raw
// chunks being converted), two P tiles.
template <bool kFp8>
struct AccLayout {
  static constexpr int kStagesA = kFp8 ? 3 : 2;
  static constexpr int kPBufs = kFp8 ? 2 : 4;
  static constexpr int kOffP = kStagesA * kStageO;           // P tiles [kPBufs]
  static constexpr int kOffAlpha = kOffP + kPBufs * kPBytes;  // rescale factors [kPBufs][128]
  static constexpr int kOffL = kOffAlpha + kPBufs * kVecBytes;  // (row sum, lse) [128]
  static constexpr int kEnd = kOffL + kRowsPerBlock * 8;
  static_assert(kPartBytes <= kStagesA * kStageO, "a partial slot must fit in the page ring");
};
constexpr int kMaxPBufs = 4;

// Shared-memory layout (byte offsets from the 1024-aligned base; the same in
// both CTAs, each uses its part).  Both CTAs keep their page ring at offset 0.
constexpr int kQStageBytes = 32 * 64;              // scorer: 2 KB per lane quarter after the ring
constexpr int kOffQStage = kStages * kStageS;      // (fp8: the Q staging below; bf16: kOffFwd)
constexpr int kScorerEnd = kOffQStage + 4 * kQStageBytes;
// bf16 scorer: the page scores of rows 32..63, forwarded from the warps that
// can read those TMEM lanes to the warps that run their softmax:
// [half][4-key group][row] float4 (8 KB, in the otherwise unused Q staging)
constexpr int kOffFwd = kOffQStage;
static_assert(kOffFwd + 2 * 8 * 32 * 16 <= kScorerEnd, "forwarding buffer overlaps");
// fp8 scorer: a smaller Q staging (32 rows x 16 channels per warp), then the
// per-stage scale slots the softmax reads
constexpr int kQStageBytesF8 = 32 * 32;
constexpr int kOffScale = kOffQStage + 4 * kQStageBytesF8;
constexpr int kScorerEndF8 = kOffScale + kStages * kScaleSlotBytes;
constexpr int kAccEnd = AccLayout<true>::kEnd > AccLayout<false>::kEnd ? AccLayout<true>::kEnd : AccLayout<false>::kEnd;
// bf16 scorer: each row's softmax runs on two threads (keys 0..31 and 32..63
// of a page) that add their row sums at a segment's end through
// [parity][half][row] floats here
constexpr int kOffXchg = kScorerEnd;
constexpr int kXchgBytes = 2 * 2 * kRowsPerBlock * 4;
constexpr int kOffBars = kScorerEnd > kAccEnd ? kScorerEnd : kAccEnd;
static_assert(kOffXchg + kXchgBytes <= kOffBars, "softmax exchange area overlaps the barriers");
static_assert(kScorerEndF8 <= kOffBars, "fp8 scorer layout overlaps the barriers");
constexpr int kBarBytes = 416;
constexpr int kSmemMax = 232448;
constexpr int kSmem = kSmemMax;                    // layout + slack for aligning the base
constexpr int kAlignSlack = kSmem - kOffBars - kBarBytes;
static_assert(kAlignSlack >= 0, "shared memory layout too large");

// TMEM columns.  Scorer: Q (576 16-bit channels) then three 64-column score
// slots: one per ring stage (bf16 cache; two adjacent slots hold the scores of
// a page pair) or the per-group score ring (fp8 cache).
constexpr uint32_t kColQ = 0, kColG = 288;
static_assert(kColG + 64 * kGroupSlots <= 512 && kGroupSlots == kStages, "score slots exceed TMEM");
// bf16 scorer stage layout (5-D page map): token group g (8 tokens), chunk c
// (64 channels) is the 1 KB 128-byte-swizzled atom at (9g + c) KB, so the
// 8-row groups of a page are kTokGroupStride apart and the next stage's first
// group follows the last one: two adjacent stages form one 128-token operand.
constexpr int kTokGroupStride = 9 * 1024;
static_assert(kStageS == 8 * kTokGroupStride, "a stage is 8 token groups");

constexpr float kRescaleLog2 = 8.0f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

// Warps: loader, MMA issuer, four row warps (softmax of the scorer, rescale +
// epilogue of the accumulator), then more:
// - bf16: warps 6-9, the second half of each row's softmax (scorer), and
//   warps 10 and 11, which run the softmax of rows 32..63 (below);
// - fp8: the dequantisation on warps 6, 7, 8 and one more.  For variant A
//   that is warp 10: warp 9 would share the MMA warp's SM sub-partition
//   (warp % 4 == 1), where arithmetic slows every MMA issue 2-4x, so it stays
//   idle (12% faster).  Variant B (heavier conversion: bf16 RoPE, scales read
//   from the token records) measured 12-20% slower with warp 10 and with an
//   idle eleventh warp than with ten warps and warp 9, so it keeps those.
template <bool kFp8, bool kRopeB = false>
struct Cfg {
  static constexpr int kThreads = !kFp8 ? 384 : (kRopeB ? 320 : 352);
  static constexpr int kSoftmaxCols = kFp8 ? 64 : 32;  // keys of a page one softmax thread scores
};

struct Bars {
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t q_full;        // scorer: Q written to TMEM (softmax threads: bf16 256, fp8 128)
  uint64_t pbuf_free[kMaxPBufs];  // scorer: accumulator finished with P tile b (remote, 1)
  uint64_t l_free;        // scorer: accumulator read the row sums (remote, 4)
  uint64_t p_full[kMaxPBufs];     // accumulator: P tile + factors arrived (1 + tx)
  uint64_t corr_done[kMaxPBufs];  // accumulator: O rescaled if needed for P buffer b (128).  One
                                  // per P buffer: the rescale warps may run as many tiles ahead
                                  // of the MMA warp as there are P buffers.
  uint64_t pv_done[kMaxPBufs];    // accumulator: PV of the tile in P buffer b done (commit)
  uint64_t o_full;        // accumulator: last PV of a segment done (commit)
  uint64_t o_free;        // accumulator: epilogue read O (128)
  uint64_t l_full;        // accumulator: row sums + lse arrived (1 + tx)
  uint64_t mrg_bar;       // accumulator: a partial of another piece arrived in the ring (1 + tx)
  uint64_t epi_bar;       // accumulator: barrier of the four epilogue warps (128), bounded
                          // unlike bar.sync, so a warp that gives up cannot strand the others
  uint64_t drain;
  uint64_t raw_full[kStages];    // fp8: this CTA's raw e4m3 chunks arrived (1 + tx)
  uint64_t dq_sync;              // fp8: the dequant threads read their raw chunks (128), bounded
  uint64_t sg_full[kGroupSlots]; // scorer: scores of a slot written (commit); bf16: slot = stage,
                                 // fp8: one scale group of the group-score ring
  uint64_t sg_free[kGroupSlots]; // scorer: that slot read by the softmax (fp8: 128; bf16: 256, both halves)
  uint64_t mx_bar[4];            // bf16 scorer: the two softmax halves of a row quarter added their
                                 // row sums (64)
  uint64_t fwd_full[2];          // bf16 scorer: half h of rows 32..63's scores forwarded (32)
  uint64_t fwd_empty[2];         // bf16 scorer: ... and read by both softmax warps of those rows (64)
  uint64_t stall;                // never signalled: the wait a test's stall request runs out on
  int abort_flag;
  uint32_t tmem_base;
  int ticket;             // accumulator: finish order of this piece among its unit's pieces
};
static_assert(sizeof(Bars) <= kBarBytes, "barrier block too large");

// One segment of a cluster's cost range: unit u (row block rb of request b),
// pages [page_lo, page_hi) of it.  `empty` units have no visible keys.
struct Seg {
  int u, b, rb, page_lo, page_hi, split, slot, empty;
};

// End of unit u's cost range: the next unit's start, except for the last
// unit of a row block (its row block's stretch may be followed by idle cost;
// the planner stores each row block's end after pre[U]).
__device__ __forceinline__ int unit_end(const int32_t* pre, int u, int U, int B) {
  return (u % B == B - 1) ? __ldg(pre + U + 1 + u / B) : __ldg(pre + u + 1);
}

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
      const int p1 = unit_end(pre, u, U, B);
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

// Writes output channels [64*cc, 64*cc + 64) of a warp's 32 rows (rows
// row0.. of request b): thread `lane` holds row `lane` (64 final values).  The
// rows are staged in `est` (4 KB, 1024-aligned) in the 128-byte-swizzled
// layout of one out_map box, and one lane hands the box to the TMA unit (rows
// past the request are clipped by the tensor map).  The staging area is free
// again when the call returns.
__device__ __forceinline__ void store_rows_tma(uint8_t* est, const float (&v)[64], const CUtensorMap* out_map,
                                               int cc, int row0, int b, int R, int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(est + lane * 128 + ((q ^ (lane & 7)) << 4)) = w;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < R) {  // a warp whose rows all lie past the request stores nothing
    tma_store_3d(out_map, 64 * cc, row0, b, smem_u32(est));
    bulk_commit_group();
    bulk_wait_read_all();
  }
  __syncwarp();
}

// Stages output channels [64*cc, 64*cc + 64) of a warp's 32 rows, cc = 4*half
// + k, into `half_buf` (16 KB, 1024-aligned) in the layout of one out_map4
// box: 32 rows x 4 chunks of 64 channels, row r of chunk k at line 32k + r,
// 128-byte swizzled (no bank conflicts: the line index mod 8 is the row).
__device__ __forceinline__ void stage_half(uint8_t* half_buf, const float (&v)[64], int k, int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4*>(half_buf + (k * 32 + lane) * 128 + ((q ^ (lane & 7)) << 4)) = w;
  }
}

// One TMA store of a staged half (256 channels x 32 rows); the caller waits
// for its reads before reusing the buffer.
__device__ __forceinline__ void store_half(uint8_t* half_buf, const CUtensorMap* out_map4, int half, int row0,
                                           int b, int R, int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0 && row0 < R) {
    tma_store_4d(out_map4, 0, row0, 4 * half, b, smem_u32(half_buf));
    bulk_commit_group();
  }
  __syncwarp();
}

// e4m3 x2 times a scale given as hi + lo halves (hi = fp16(scale), lo =
// fp16(scale - hi)) -> f16x2.  x*lo is small, so the fused x*hi + x*lo is
// rounded once: within a tiny error of fp16(x * scale) for scales >= 2^-14.
__device__ __forceinline__ uint32_t e4m3x2_scaled_f16x2(uint16_t v, __half2 hi, __half2 lo) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  const __half2 x = *reinterpret_cast<const __half2*>(&h2);
  const __half2 y = __hfma2(x, hi, __hmul2(x, lo));
  return *reinterpret_cast<const uint32_t*>(&y);
}

// e4m3 x2 -> f16x2, exact (every e4m3 value is an fp16 value).
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return h2;
}

// Tree reductions over 64 values (independent chains for ILP).
// Maximum of n floats: two independent chains of three-input maxima.
template <int n>
__device__ __forceinline__ float max_n(const float (&x)[n]) {
  static_assert(n >= 8 && n % 4 == 0, "max_n expects a multiple of four");
  float m0 = fmax3(x[0], x[1], x[2]), m1 = fmax3(x[3], x[4], x[5]);
#pragma unroll
  for (int i = 6; i + 3 < n; i += 4) {
    m0 = fmax3(m0, x[i], x[i + 1]);
    m1 = fmax3(m1, x[i + 2], x[i + 3]);
  }
  return fmax3(m0, m1, fmax3(x[n - 2], x[n - 1], x[n - 2]));
}

// Bounded barrier wait, its waiting loop inlined or out of line (kOut).  The
// fp8 variant A kernel ran 9% faster with every loop out of line (less code
// for its warps to fetch); the bf16 kernel ran 6% slower on the MTP workload
// that way, so it keeps the loops of its per-page waits inline; variant B was
// not measured and keeps all of them inline.
template <bool kOut, bool kClusterAcquire = false>
__device__ __forceinline__ bool kwait(uint32_t bar, uint32_t parity, const volatile int* abort_flag) {
  if constexpr (kOut) {
    return mbar_wait_ool<kClusterAcquire>(bar, parity, abort_flag);
  } else {
    return mbar_wait<kClusterAcquire>(bar, parity, abort_flag);
  }
}

// kRopeB (with kFp8): fp8 variant B, 656-byte token records (scales inside,
// RoPE in bf16).
template <bool kFp8, bool kRopeB = false>
__global__ void __launch_bounds__(Cfg<kFp8, kRopeB>::kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap kv_map_s, const __grid_constant__ CUtensorMap kv_map_a,
                      const __grid_constant__ CUtensorMap kv_map_r,
                      const __grid_constant__ CUtensorMap q_map, const __grid_constant__ CUtensorMap out_map,
                      const __grid_constant__ CUtensorMap out_map4, const DecodeArgs a) {
  // see kwait: fp8 variant A takes every waiting loop out of line; bf16 the
  // loops of waits outside the per-page loops (segment ends, epilogue, merge)
  constexpr bool kOutWait = kFp8 && !kRopeB;
  constexpr bool kOutCold = !(kFp8 && kRopeB);
  constexpr int kStagesA = AccLayout<kFp8>::kStagesA, kPBufs = AccLayout<kFp8>::kPBufs;
  constexpr int kOffP = AccLayout<kFp8>::kOffP, kOffAlpha = AccLayout<kFp8>::kOffAlpha, kOffL = AccLayout<kFp8>::kOffL;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBars);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const bool scorer = rank == 0;
  if (pad > static_cast<uint32_t>(kAlignSlack)) {  // never expected: report, do nothing
    griddep_wait();  // the planner clears the error word first
    if (tid == 0) atomicOr(a.err, kErrTimeout);
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // fp8: the 128 dequant threads complete a stage; the fp8 scorer's stage
      // is freed by its 128 softmax threads once they have read the stage's
      // scales (the group commits they waited on imply its MMAs are done)
      mbar_init(smem_u32(&bars->kv_full[s]), kFp8 ? 128 : 1);
      mbar_init(smem_u32(&bars->kv_empty[s]), (kFp8 && scorer) ? 128 : 1);
    }
    // bf16: both softmax halves write Q; fp8: the four softmax warps
    mbar_init(smem_u32(&bars->q_full), kFp8 ? 128 : 256);
    for (int i = 0; i < kMaxPBufs; ++i) {
      mbar_init(smem_u32(&bars->pbuf_free[i]), 1);
      mbar_init(smem_u32(&bars->p_full[i]), 1);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
      mbar_init(smem_u32(&bars->corr_done[i]), 128);
    }
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->o_free), 128);
    mbar_init(smem_u32(&bars->l_free), 4);
    mbar_init(smem_u32(&bars->l_full), 1);
    mbar_init(smem_u32(&bars->mrg_bar), 1);
    mbar_init(smem_u32(&bars->epi_bar), 128);
    mbar_init(smem_u32(&bars->drain), 1);
    for (int s = 0; s < kStages; ++s) mbar_init(smem_u32(&bars->raw_full[s]), 1);
    for (int s = 0; s < kGroupSlots; ++s) {
      mbar_init(smem_u32(&bars->sg_full[s]), 1);
      mbar_init(smem_u32(&bars->sg_free[s]), kFp8 ? 128 : 256);
    }
    for (int s = 0; s < 4; ++s) mbar_init(smem_u32(&bars->mx_bar[s]), 64);
    for (int h = 0; h < 2; ++h) {
      mbar_init(smem_u32(&bars->fwd_full[h]), 32);
      mbar_init(smem_u32(&bars->fwd_empty[h]), 64);
    }
    mbar_init(smem_u32(&bars->stall), 1);
    mbar_init(smem_u32(&bars->dq_sync), 128);
    bars->abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(scorer ? &kv_map_s : &kv_map_a);
    if (kFp8 && scorer) tma_prefetch_desc(&kv_map_r);
    if (!kFp8 && scorer) tma_prefetch_desc(&q_map);
    if (!scorer) {
      tma_prefetch_desc(&out_map);
      tma_prefetch_desc(&out_map4);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem_base), 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  cluster_sync_all();
  tc_fence_after();
  // Everything above overlaps the planner kernel (programmatic dependent
  // launch); the plan, the error word and the outputs are touched only after
  // the planner has finished.
  griddep_wait();
  griddep_launch_dependents();
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
  const int nst = scorer ? kStages : kStagesA;     // ring stages of this CTA

  if (warp == 0) {
    // ---------------------------------------------------------------- loader
    // The whole warp walks the segments; lane 0 waits and issues the copies.
    // Page ids are read 32 at a time (one per lane) and shuffled out.  Each
    // page is ONE 4-D copy (the TMA unit spends a fixed time per copy, so few
    // large copies keep it fastest); the accumulator's read of a page is its
    // last use (the scorer read it a little earlier), so it is marked to be
    // evicted from L2 first.  Nothing else is issued to the TMA unit here.
    SegIter it = it0;
    Seg s;
    const uint64_t policy = l2_policy_evict_first();
    // bf16 scorer: each segment's Q block (128 rows x 576 channels, exactly
    // two ring stages) goes through the ring ahead of the segment's pages, as
    // two 64-row copies; the softmax warps move it to TMEM, and the MMA warp
    // frees the two stages once Q is there.  So the next segment's Q arrives
    // while the current segment still runs.
    const bool q_ring = scorer && !kFp8;
    // At kernel start every CTA wants its first data at once (DRAM-bound).  The
    // accumulator needs V only for its first PV, after the first P tile has
    // arrived; waiting for that keeps its (second) reads of the first pages
    // out of the start-up burst, so the scorer's Q and first page land sooner.
    bool wait_first_p = !scorer && !kFp8;
    int stage = 0;
    uint32_t ph = 0;
    int last_par[kStages];
    for (int i = 0; i < kStages; ++i) last_par[i] = -1;
    bool ok = true;
    const uint32_t bytes = static_cast<uint32_t>(nbox * kBox);
    while (ok && it.next(s)) {
      if (s.empty) continue;
      for (int h = 0; q_ring && h < 2; ++h) {
        if (lane == 0) {
          if (!kwait<kOutWait>(smem_u32(&bars->kv_empty[stage]), ph ^ 1u, abort_flag)) {
            ok = false;
            if (!*abort_flag) signal_abort(bars, a.err, peer);
          } else {
            const uint32_t qb = smem_u32(&bars->kv_full[stage]);
            mbar_arrive_expect_tx(qb, static_cast<uint32_t>(kStageS));
            tma_load_4d(smem_u32(smem + stage * kStageS), &q_map, 0, 0, s.rb * kRowsPerBlock + 64 * h, s.b, qb);
            last_par[stage] = ph == 0u ? 0 : 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (++stage == nst) {
          stage = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      const int32_t* bt = a.block_table + static_cast<size_t>(s.b) * a.max_pages;
      for (int p0 = s.page_lo; ok && p0 < s.page_hi; p0 += 32) {
        const int my_p = p0 + lane;
        const int my_pid = my_p < s.page_hi ? __ldg(bt + my_p) : 0;
        const int cnt = min(32, s.page_hi - p0);
        for (int k = 0; k < cnt; ++k) {
          int pid = __shfl_sync(0xffffffffu, my_pid, k);
          if (lane == 0 && wait_first_p) {
            wait_first_p = false;
            if (!kwait<kOutCold, true>(smem_u32(&bars->p_full[0]), 0u, abort_flag)) {
              ok = false;
              if (!*abort_flag) signal_abort(bars, a.err, peer);
            }
          }
          if (lane == 0 && ok) {
            if (!kwait<kOutWait>(smem_u32(&bars->kv_empty[stage]), ph ^ 1u, abort_flag)) {
              ok = false;
              if (!*abort_flag) signal_abort(bars, a.err, peer);
            } else {
              if (pid < 0 || pid >= a.num_pages) {
                atomicOr(a.err, kErrBounds);
                pid = a.num_pages;  // outside the tensor map: TMA fills zeros, no fault
              }
              const uint32_t fb = smem_u32(kFp8 ? &bars->raw_full[stage] : &bars->kv_full[stage]);
              uint8_t* dst = smem + stage * stage_bytes;
              if (kFp8) {
                // every raw chunk this CTA converts, into the top of its stage
                mbar_arrive_expect_tx(
                    fb, static_cast<uint32_t>(scorer ? (kRopeB ? kRawBytesSB : kRawBytesS) : kRawBytesA));
                if (scorer) {
                  const int off = kRopeB ? kRawOffSB : kRawOffS;
                  // variant A: chunks 0..8 of the e4m3 row; variant B: the 8 latent chunks
                  tma_load_4d(smem_u32(dst + off), &kv_map_s, 0, 0, 0, pid, fb);
                  // variant B: the two bf16 RoPE chunks of the record
                  if (kRopeB) tma_load_4d(smem_u32(dst + off + 8 * kRawSlot), &kv_map_r, 0, 0, 0, pid, fb);
                } else {
                  tma_load_4d(smem_u32(dst + kRawOffA), &kv_map_a, 0, 0, 0, pid, fb);
                }
              } else if (scorer) {
                // token-group-major: (64 channels, 8 tokens, 9 chunks, 8 token groups, page)
                mbar_arrive_expect_tx(fb, bytes);
                tma_load_5d(smem_u32(dst), &kv_map_s, 0, 0, 0, 0, pid, fb);
              } else {
                mbar_arrive_expect_tx(fb, bytes);
                tma_load_4d_hint(smem_u32(dst), &kv_map_a, 0, 0, 0, pid, fb, policy);
              }
              last_par[stage] = static_cast<int>(ph);
            }
          }
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!ok) break;
          if (++stage == nst) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && lane == 0) {
      // wait (time-bounded only) for the loads already in flight
      for (int i = 0; i < nst; ++i)
        if (last_par[i] >= 0)
          kwait<kOutCold>(smem_u32(kFp8 ? &bars->raw_full[i] : &bars->kv_full[i]), static_cast<uint32_t>(last_par[i]), nullptr);
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
    if (scorer && __ldg(a.hdr + kHdrStall) != 0) {
      // a test's stall request: wait on a barrier nothing signals, so the
      // bounded wait runs out and the whole cluster takes its abort path
      if (!kwait<kOutCold>(smem_u32(&bars->stall), 0u, abort_flag)) ok = false;
    }
    if (scorer) {
      // S = Q K^T: 36 steps of K=16 over the 576 channels, A = Q in TMEM.
      // bf16 cache: a page in ring stage 0 or 1 is paired with the next page of
      // the segment (which sits in the next stage) and both are scored by one
      // N=128 chain into two adjacent slots; an N=64 MMA re-reads its slice of
      // Q from TMEM as an N=128 one does, so the pair costs about what one page
      // did.  A page in the last stage goes alone (N=64).
      // fp8 cache: the same steps over the exact e4m3 codes, one MMA chain per
      // scale group (8 steps per latent group of 128 channels, 4 for the RoPE)
      // into the next slot of the group-score ring; the softmax applies the
      // tokens' scales and frees the stage.
      const uint32_t idesc = idesc_f16_f32(128, 64, false, false, !kFp8);
      const uint32_t idesc2 = idesc_f16_f32(128, 128, false, false, !kFp8);
      uint32_t gj = 0;  // fp8: group-score ring counter over the whole kernel
      // bf16: score slot s is used by the pages that sit in stage s; bit s of
      // sgp is the parity of its next use (the Q block's stages score nothing)
      uint32_t sgp = 0;
      while (ok && it.next(s)) {
        if (s.empty) continue;
        if (!kwait<kOutCold>(smem_u32(&bars->q_full), q_ph, abort_flag)) { ok = false; break; }
        q_ph ^= 1u;
        if (!kFp8) {
          // Q is in TMEM, so the two stages that brought it are free
          for (int h = 0; h < 2; ++h) {
            if (lane == 0) mbar_arrive(smem_u32(&bars->kv_empty[stage]));
            if (++stage == kStages) {
              stage = 0;
              ph ^= 1u;
            }
          }
        }
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          if (!kwait<kOutWait>(smem_u32(&bars->kv_full[stage]), ph, abort_flag)) { ok = false; break; }
          const uint64_t b0 = smem_desc_sw128(smem_u32(smem + stage * kStageS), 16, kFp8 ? 1024 : kTokGroupStride);
          if (kFp8) {
            for (int g = 0; g < kGroups && ok; ++g, ++gj) {
              const uint32_t slot = gj % kGroupSlots, gph = (gj / kGroupSlots) & 1u;
              // warp-uniform outcome: the issue below ends in __syncwarp
              if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->sg_free[slot]), gph ^ 1u, abort_flag))) {
                ok = false;
                break;
              }
              tc_fence_after();
              if (lane == 0) {
                const uint32_t dcol = tbase + kColG + 64 * slot;
                const int k0 = 8 * g, k1 = g < 4 ? 8 * g + 8 : 36;
                for (int k = k0; k < k1; ++k)
                  mma_ts(dcol, tbase + kColQ + 8 * k, b0 + static_cast<uint64_t>(((k >> 2) * kBox + (k & 3) * 32) >> 4),
                         idesc, k > k0 ? 1u : 0u);
                mma_commit(smem_u32(&bars->sg_full[slot]));
              }
              __syncwarp();
            }
            if (!ok) break;
          } else {
            // slot = stage (a pair: stage and stage + 1, no wrap)
            // (not a segment's first page: the page after it goes to a stage the
            // segment's Q block frees only once Q is in TMEM)
            const bool pair = stage < kStages - 1 && j > s.page_lo && j + 1 < s.page_hi;
            bool ready = kwait<kOutWait>(smem_u32(&bars->sg_free[stage]), ((sgp >> stage) & 1u) ^ 1u, abort_flag);
            if (pair) {
              ready = ready && kwait<kOutWait>(smem_u32(&bars->kv_full[stage + 1]), ph, abort_flag) &&
                      kwait<kOutWait>(smem_u32(&bars->sg_free[stage + 1]), ((sgp >> (stage + 1)) & 1u) ^ 1u, abort_flag);
            }
            sgp ^= (pair ? 3u : 1u) << stage;
            if (!__all_sync(0xffffffffu, ready)) { ok = false; break; }  // uniform: the issue ends in __syncwarp
            tc_fence_after();
            if (lane == 0) {
              const uint32_t dcol = tbase + kColG + 64 * stage;
              const uint32_t id = pair ? idesc2 : idesc;
              // chunk 0, then the other eight 64-channel chunks two per
              // iteration: a fully unrolled chain of 36 made the kernel 2-3%
              // slower (more code for the issuing warp to fetch)
              mma_ts(dcol, tbase + kColQ, b0, id, 0u);
#pragma unroll
              for (int k = 1; k < 4; ++k)
                mma_ts(dcol, tbase + kColQ + 8 * k, b0 + static_cast<uint64_t>((k * 32) >> 4), id, 1u);
#pragma unroll 1
              for (int c = 1; c < 9; c += 2) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  mma_ts(dcol, tbase + kColQ + 32 * c + 8 * k, b0 + static_cast<uint64_t>((c * 1024 + (k >> 2) * 1024 + (k & 3) * 32) >> 4), id, 1u);
              }
              mma_commit(smem_u32(&bars->sg_full[stage]));
              mma_commit(smem_u32(&bars->kv_empty[stage]));
              if (pair) {
                mma_commit(smem_u32(&bars->sg_full[stage + 1]));
                mma_commit(smem_u32(&bars->kv_empty[stage + 1]));
              }
            }
            __syncwarp();
            if (pair) {  // the second page of the pair is done too (stage + 1 < kStages: no wrap)
              ++j;
              ++t;
              ++stage;
            }
          }
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
          const uint32_t sb = t % kPBufs;
          if (!kwait<kOutWait>(smem_u32(&bars->kv_full[stage]), ph, abort_flag)) { ok = false; break; }
          uint8_t* st = smem + stage * kStageO;
          if (!kFp8) {
            const int valid = seqlen - j * kPage;
            if (valid < kPage) zero_tail_rows(st, valid > 0 ? valid : 0, 8, lane);
            __syncwarp();
          }
          if (!kwait<kOutWait>(smem_u32(&bars->corr_done[sb]), (t / kPBufs) & 1u, abort_flag)) { ok = false; break; }
          if (j == s.page_lo) {
            if (!kwait<kOutCold>(smem_u32(&bars->o_free), ofree_ph ^ 1u, abort_flag)) { ok = false; break; }
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
            // P buffer sb may be refilled by the scorer once this PV is done; the
            // buffer of a segment's last tile is returned by the epilogue instead,
            // which stages its stores there.
            if (j + 1 < s.page_hi) mma_commit_multicast(smem_u32(&bars->pbuf_free[sb]), static_cast<uint16_t>(1u << peer));
            if (j + 1 == s.page_hi) mma_commit(smem_u32(&bars->o_full));
          }
          __syncwarp();
          if (++stage == kStagesA) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
    }
    if (!ok && !*abort_flag && lane == 0) signal_abort(bars, a.err, peer);
    if (lane == 0) {
      mma_commit(smem_u32(&bars->drain));
      kwait<kOutCold>(smem_u32(&bars->drain), 0u, nullptr);
    }
    __syncwarp();
  } else if (warp < 6 || (!kFp8 && scorer)) {
    // bf16 scorer: a warp can reach only the TMEM lanes of its SM sub-partition
    // (warp % 4), and the MMA warp (warp 1) shares sub-partition 1 with warps
    // 5 and 9.  Arithmetic in that sub-partition slows every MMA issue 2-4x
    // (arithmetic in the other three costs it nothing), so warps 5 and 9 only
    // move data for rows 32..63: Q into TMEM, and each page's scores from TMEM
    // to shared memory (`fwd`).  Warps 10 and 11 (sub-partitions 2 and 3) run
    // the softmax of those rows from there (`xq`).
    const bool fwd = !kFp8 && scorer && (warp == 5 || warp == 9);
    const bool xq = !kFp8 && warp >= 10;
    const int wq = xq ? 1 : (warp & 3);
    const int L = wq * 32 + lane;  // query row within the block (== TMEM lane, xq: not read)
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int ctid = tid - 64;     // 0..127 (rows of warps 2-5)
    // bf16 scorer: half hh of the row's keys (warps 2-5 and 10: keys 0..31 of
    // a page, warps 6-9 and 11: keys 32..63); the fp8 softmax runs whole rows
    // on warps 2-5
    constexpr int kSC = Cfg<kFp8>::kSoftmaxCols;
    const int hh = kFp8 ? 0 : (xq ? warp - 10 : (warp >= 6 ? 1 : 0));
    const int c0 = kSC * hh;
    SegIter it = it0;
    Seg s;
    uint32_t t = 0, seg_n = 0;
    bool ok = true;
    if (scorer) {
      // ------------------------------------------------------------ softmax (scorer)
      const uint32_t rP = mapa_shared(smem_u32(smem + kOffP), peer);
      const uint32_t rAlpha = mapa_shared(smem_u32(smem + kOffAlpha), peer);
      const uint32_t rL = mapa_shared(smem_u32(smem + kOffL), peer);
      const uint32_t rPfull0 = mapa_shared(smem_u32(&bars->p_full[0]), peer);  // + 8 b: P buffer b's
      const uint32_t rLfull = mapa_shared(smem_u32(&bars->l_full), peer);
      uint32_t q_loaded = 0;
      float qmul = 1.f, qmul_next = 1.f;
      uint32_t gj = 0;  // fp8: group-score ring counter (advances like the MMA warp's)

      // bf16: Q rows -> TMEM (the A operand of QK) from the segment's two Q
      // stages of the ring (rows 0..63 in the first, 64..127 in the second;
      // row r, chunk c at line 9r + c of the 128-byte-swizzled box).  The two
      // softmax halves split the chunks (0..4, 5..8); the MMA warp frees the
      // stages after q_full.
      auto load_q_ring = [&](uint32_t r0) -> bool {
        const uint32_t rq = r0 + (L >= 64 ? 1u : 0u);
        const uint32_t st = rq % kStages;
        if (!kwait<kOutCold>(smem_u32(&bars->kv_full[st]), (rq / kStages) & 1u, abort_flag)) return false;
        const uint8_t* qs_base = smem + st * kStageS;
        const int row = L & 63;
        for (int c = hh ? 5 : 0; c < (hh ? 9 : 5); ++c) {
          uint32_t w[32];
          const int n = 9 * row + c;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 y = *reinterpret_cast<const uint4*>(qs_base + n * 128 + ((k ^ (n & 7)) << 4));
            w[4 * k + 0] = y.x;
            w[4 * k + 1] = y.y;
            w[4 * k + 2] = y.z;
            w[4 * k + 3] = y.w;
          }
          tmem_st32(tbase + lane_off + kColQ + 32 * c, w);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->q_full));
        return true;
      };
      // fp8 cache: the MMAs run in fp16, so each row is first scaled by a power
      // of two that puts |q| <= 16384 (no overflow; undone on the scores).
      // Same coalesced scheme with 16-channel half-steps through a 1 KB
      // staging area per warp (the rest of the space holds the scale slots).
      uint8_t* const qst8 = smem + kOffQStage + wq * kQStageBytesF8;
      auto load_q_f16 = [&](const Seg& sg) -> float {
        const int r0 = sg.rb * kRowsPerBlock + wq * 32;
        const int rsub = lane >> 1, csub = lane & 1;     // load view: rows rsub + 16i, 16-byte chunk csub of 32
        const uint8_t* qb = reinterpret_cast<const uint8_t*>(a.q) + static_cast<size_t>(sg.b) * a.R * (kDqk * 2);
        bool rv[2];
        const uint8_t* rp[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int r = r0 + rsub + 16 * i;
          rv[i] = r < a.R;
          rp[i] = qb + static_cast<size_t>(rv[i] ? r : 0) * (kDqk * 2) + csub * 16;
        }
        float am[2] = {0.f, 0.f};
        for (int h0 = 0; h0 < 36; h0 += 12) {
          uint4 x[24];
#pragma unroll
          for (int u = 0; u < 12; ++u)
#pragma unroll
            for (int i = 0; i < 2; ++i)
              x[2 * u + i] = rv[i] ? __ldg(reinterpret_cast<const uint4*>(rp[i] + (h0 + u) * 32)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int v = 0; v < 24; ++v) {
            const uint4 y = x[v];
            const float m = fmaxf(fmaxf(fmaxf(fabsf(bf16_lo(y.x)), fabsf(bf16_hi(y.x))),
                                        fmaxf(fabsf(bf16_lo(y.y)), fabsf(bf16_hi(y.y)))),
                                  fmaxf(fmaxf(fabsf(bf16_lo(y.z)), fabsf(bf16_hi(y.z))),
                                        fmaxf(fabsf(bf16_lo(y.w)), fabsf(bf16_hi(y.w)))));
            am[v & 1] = fmaxf(am[v & 1], m);
          }
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) am[i] = fmaxf(am[i], __shfl_xor_sync(0xffffffffu, am[i], 1));
        // row `lane` of the warp was read by lanes 2 * (lane & 15) + 0..1, as its (lane >> 4)-th row
        const float v0 = __shfl_sync(0xffffffffu, am[0], 2 * (lane & 15));
        const float v1 = __shfl_sync(0xffffffffu, am[1], 2 * (lane & 15));
        const float amax = (lane >> 4) ? v1 : v0;
        int k = 0;
        while (k < 126 && amax * ldexpf(1.f, -k) > 16384.f) ++k;
        const float qs = ldexpf(1.f, -k);
        for (int h0 = 0; h0 < 36; h0 += 12) {
          uint4 x[24];
#pragma unroll
          for (int u = 0; u < 12; ++u)
#pragma unroll
            for (int i = 0; i < 2; ++i)
              x[2 * u + i] = rv[i] ? __ldg(reinterpret_cast<const uint4*>(rp[i] + (h0 + u) * 32)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 12; ++u) {
            // staging row rr at rr * 32, its 16-byte chunk c at (c ^ ((rr >> 2) & 1)) (no bank conflicts)
#pragma unroll
            for (int i = 0; i < 2; ++i) {
              const int rr = rsub + 16 * i;
              *reinterpret_cast<uint4*>(qst8 + rr * 32 + ((csub ^ ((rr >> 2) & 1)) << 4)) = x[2 * u + i];
            }
            __syncwarp();
            uint32_t w[8];
#pragma unroll
            for (int c2 = 0; c2 < 2; ++c2) {
              const uint4 y = *reinterpret_cast<const uint4*>(qst8 + lane * 32 + ((c2 ^ ((lane >> 2) & 1)) << 4));
              w[4 * c2 + 0] = pack_f16x2(bf16_lo(y.x) * qs, bf16_hi(y.x) * qs);
              w[4 * c2 + 1] = pack_f16x2(bf16_lo(y.y) * qs, bf16_hi(y.y) * qs);
              w[4 * c2 + 2] = pack_f16x2(bf16_lo(y.z) * qs, bf16_hi(y.z) * qs);
              w[4 * c2 + 3] = pack_f16x2(bf16_lo(y.w) * qs, bf16_hi(y.w) * qs);
            }
            __syncwarp();
            tmem_st8(tbase + lane_off + kColQ + 8 * (h0 + u), w);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->q_full));
        return ldexpf(1.f, k);
      };
      uint32_t rr = 0, sgp = 0;  // bf16: ring index of the next stage, parities of the score slots
      uint32_t fph = 0;          // bf16, rows 32..63: parity of the forwarding barriers' next use
      // bf16: the two halves of a row meet at a segment's end to add their
      // row sums; bounded waits
      float* const xchg = reinterpret_cast<float*>(smem + kOffXchg);
      uint32_t xph = 0;
      auto exchange = [&](float v, float& other) -> bool {
        xchg[((xph & 1u) * 2 + hh) * kRowsPerBlock + L] = v;
        mbar_arrive(smem_u32(&bars->mx_bar[wq]));
        const bool done = kwait<kOutCold>(smem_u32(&bars->mx_bar[wq]), xph & 1u, abort_flag);
        other = xchg[((xph & 1u) * 2 + (hh ^ 1)) * kRowsPerBlock + L];
        ++xph;
        return done;
      };

      while (ok && it.next(s)) {
        if (s.empty) continue;  // the accumulator writes its zero output and lse
        const int r = s.rb * kRowsPerBlock + L;
        const bool row_valid = r < a.R;
        const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
        int n_vis = 0;
        if (row_valid) {
          n_vis = seqlen - a.s_q + r / a.H + 1;
          n_vis = n_vis < 0 ? 0 : (n_vis > seqlen ? seqlen : n_vis);
        }
        if (kFp8) {
          qmul = q_loaded ? qmul_next : load_q_f16(s);
        } else {
          if (!xq && !q_loaded && !load_q_ring(rr)) { ok = false; break; }
          rr += 2;  // the Q block's two stages
          qmul = 1.f;
        }
        q_loaded = 0;
        const float row_scale = a.scale_log2 * qmul;
        float m_ref = -INFINITY, l = 0.f;
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t, ++rr) {
          const uint32_t sb = t % kPBufs, sph = (t / kPBufs) & 1u;
          if (kFp8 && j == max(s.page_lo, s.page_hi - 3)) {
            // the next segment's Q row of this thread into L2 (plain prefetches,
            // so the TMA unit stays free for pages)
            SegIter look = it;
            Seg nx;
            while (look.next(nx))
              if (!nx.empty) {
                const int rn = nx.rb * kRowsPerBlock + L;
                if (rn < a.R) {
                  const uint8_t* row = reinterpret_cast<const uint8_t*>(a.q + (static_cast<size_t>(nx.b) * a.R + rn) * kDqk);
#pragma unroll
                  for (int v = 0; v < 9; ++v) prefetch_line_l2(row + 128 * v);
                }
                break;
              }
          }
          float x[kSC];
          float mt_page = 0.f;  // bf16: the page maximum over the row's 64 keys, scaled
          if constexpr (kFp8) {
            // S = sum_g scale[token][g] * S_g, in fp32 from the group-score ring;
            // the tokens' scales are in the scale slot of the tile's stage
            const int stg = static_cast<int>(t % kStages);
            const float* scl = reinterpret_cast<const float*>(smem + kOffScale + stg * kScaleSlotBytes);
#pragma unroll
            for (int i = 0; i < kSC; ++i) x[i] = 0.f;
            for (int g = 0; g < kGroups; ++g, ++gj) {
              const uint32_t slot = gj % kGroupSlots, gph = (gj / kGroupSlots) & 1u;
              // warp-uniform outcome: tcgen05.ld below is a warp-wide instruction
              if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->sg_full[slot]), gph, abort_flag))) {
                ok = false;
                break;
              }
              // the dequant threads wrote the scales before completing the stage
              if (g == 0 &&
                  !__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->kv_full[stg]), (t / kStages) & 1u, abort_flag))) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint32_t col = tbase + lane_off + kColG + 64 * slot;
              const float4* sc4 = reinterpret_cast<const float4*>(scl + g * 64);
              // the group's 64 scores in two halves of 32 (fewer live registers)
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {
                uint32_t v0[32];
                tmem_ld32(col + 32 * hf, v0);
                tmem_wait_ld();
                if (hf == 1) {
                  tc_fence_before();
                  mbar_arrive(smem_u32(&bars->sg_free[slot]));
                }
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4) {
                  const float4 sc = sc4[8 * hf + i4];
                  float* xa = x + 32 * hf + 4 * i4;
                  ffma2(xa[0], xa[1], __uint_as_float(v0[4 * i4 + 0]), __uint_as_float(v0[4 * i4 + 1]), sc.x, sc.y, xa[0], xa[1]);
                  ffma2(xa[2], xa[3], __uint_as_float(v0[4 * i4 + 2]), __uint_as_float(v0[4 * i4 + 3]), sc.z, sc.w, xa[2], xa[3]);
                }
              }
            }
            if (!ok) break;
            // scales read and every QK MMA of the page done: the stage may be refilled
            mbar_arrive(smem_u32(&bars->kv_empty[stg]));
            const int nv = n_vis - j * kPage;  // keys of this page visible to the row
#pragma unroll
            for (int i = 0; i < kSC; ++i) x[i] = i < nv ? x[i] * row_scale : -INFINITY;
          } else {
            // Both threads of a row read all 64 scores of the page: each takes
            // the page maximum over all of them (so the two agree on it without
            // exchanging anything) and exponentiates its own half (v0).
            uint32_t v0[32], v1[32];
            float4* const fwd_row = reinterpret_cast<float4*>(smem + kOffFwd) + hh * 256 + lane;
            if (xq) {
              // rows 32..63: the scores forwarded by warps 5 and 9 (one half each)
              const bool got = kwait<kOutWait>(smem_u32(&bars->fwd_full[0]), fph, abort_flag) &&
                               kwait<kOutWait>(smem_u32(&bars->fwd_full[1]), fph, abort_flag);
              if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
              }
              const float4* const oth_row = reinterpret_cast<const float4*>(smem + kOffFwd) + (hh ^ 1) * 256 + lane;
#pragma unroll
              for (int k4 = 0; k4 < 8; ++k4) {
                const float4 y = fwd_row[32 * k4], z = oth_row[32 * k4];
                v0[4 * k4 + 0] = __float_as_uint(y.x);
                v0[4 * k4 + 1] = __float_as_uint(y.y);
                v0[4 * k4 + 2] = __float_as_uint(y.z);
                v0[4 * k4 + 3] = __float_as_uint(y.w);
                v1[4 * k4 + 0] = __float_as_uint(z.x);
                v1[4 * k4 + 1] = __float_as_uint(z.y);
                v1[4 * k4 + 2] = __float_as_uint(z.z);
                v1[4 * k4 + 3] = __float_as_uint(z.w);
              }
              mbar_arrive(smem_u32(&bars->fwd_empty[0]));
              mbar_arrive(smem_u32(&bars->fwd_empty[1]));
              fph ^= 1u;
            } else {
              const uint32_t slot = rr % kStages, sph3 = (sgp >> slot) & 1u;  // the page's stage and its use
              sgp ^= 1u << slot;
              if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->sg_full[slot]), sph3, abort_flag))) {
                ok = false;
                break;
              }
              tc_fence_after();
              tmem_ld32(tbase + lane_off + kColG + 64 * slot + c0, v0);         // this half's 32 keys
              if (!fwd) tmem_ld32(tbase + lane_off + kColG + 64 * slot + (c0 ^ 32), v1);  // the other half's
              tmem_wait_ld();
              tc_fence_before();
              mbar_arrive(smem_u32(&bars->sg_free[slot]));
              if (fwd) {
                // rows 32..63: hand the scores on (the previous page's were read)
                if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->fwd_empty[hh]), fph ^ 1u, abort_flag))) {
                  ok = false;
                  break;
                }
#pragma unroll
                for (int k4 = 0; k4 < 8; ++k4)
                  fwd_row[32 * k4] = make_float4(__uint_as_float(v0[4 * k4 + 0]), __uint_as_float(v0[4 * k4 + 1]),
                                                 __uint_as_float(v0[4 * k4 + 2]), __uint_as_float(v0[4 * k4 + 3]));
                mbar_arrive(smem_u32(&bars->fwd_full[hh]));
                fph ^= 1u;
                continue;
              }
            }
            // raw scores (the scale is applied in the exponent's FMA below);
            // keys the row does not see (only on a request's last pages) -> -inf
            const int nv = n_vis - j * kPage - c0;         // keys of this half visible to the row
            const int nvo = n_vis - j * kPage - (c0 ^ 32);  // ... of the other half
            float xo[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              x[i] = __uint_as_float(v0[i]);
              xo[i] = __uint_as_float(v1[i]);
            }
            if (__any_sync(0xffffffffu, nv < 32 || nvo < 32)) {
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                x[i] = i < nv ? x[i] : -INFINITY;
                xo[i] = i < nvo ? xo[i] : -INFINITY;
              }
            }
            // the page's maximum over the whole row (the same value in both
            // threads: max is exact), then scaled (softmax_scale > 0 commutes with it)
            mt_page = fmaxf(max_n(x), max_n(xo)) * row_scale;
          }
          float mt = kFp8 ? max_n(x) : mt_page;
          const float xs = kFp8 ? 1.f : row_scale;  // fp8: x is already scaled
          float alpha = 1.f;
          if (mt > m_ref + kRescaleLog2) {
            if (m_ref != -INFINITY) {
              alpha = ex2_approx(m_ref - mt);
              l *= alpha;
            }
            m_ref = mt;
          }
          uint32_t pk[kSC / 2];
          float ps[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) ps[i] = 0.f;
          if (m_ref == -INFINITY) {
#pragma unroll
            for (int v = 0; v < kSC / 2; ++v) pk[v] = 0u;
          } else {
            const float nm = -m_ref;
#pragma unroll
            for (int v = 0; v < kSC / 2; ++v) {
              float t0, t1;
              ffma2(t0, t1, x[2 * v], x[2 * v + 1], xs, xs, nm, nm);
              const float p0 = ex2_approx(t0), p1 = ex2_approx(t1);
              float* acc = ps + 2 * (v & 3);
              fadd2(acc[0], acc[1], acc[0], acc[1], p0, p1);
              pk[v] = kFp8 ? pack_f16x2(p0, p1) : pack_bf16x2(p0, p1);
            }
          }
          l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));

          // this thread's part of P tile t (16-byte granules c0/8 ..) and, from
          // the first half, the row's factor to the accumulator (its buffer sb must be free)
          if (!kwait<kOutWait>(smem_u32(&bars->pbuf_free[sb]), sph ^ 1u, abort_flag)) { ok = false; break; }
          const uint32_t pbar = rPfull0 + 8u * sb;
          const uint32_t prow = rP + sb * kPBytes + L * 128;
#pragma unroll
          for (int cc = 0; cc < kSC / 8; ++cc)
            st_async_v4_u32(prow + (((c0 / 8 + cc) ^ (L & 7)) << 4), pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2],
                            pk[4 * cc + 3], pbar);
          if (hh == 0) st_async_f32(rAlpha + sb * kVecBytes + L * 4, alpha, pbar);
        }
        if (!ok) break;

        if (!kFp8 && !fwd) {  // the row sum over both halves
          float other;
          if (!exchange(l, other)) { ok = false; break; }
          l += other;
        }
        if (hh == 0 && !fwd) {
          // the row sum and lse go to the accumulator, which writes the outputs
          const float lse_v = l > 0.f ? (m_ref + lg2_approx(l)) * kLn2 : -INFINITY;
          if (!kwait<kOutCold>(smem_u32(&bars->l_free), (seg_n & 1u) ^ 1u, abort_flag)) { ok = false; break; }
          st_async_v2_f32(rL + L * 8, l, lse_v, rLfull);
          ++seg_n;
        }
        // Q of the next segment with pages can go in now: the QK of this
        // segment's last page is done (its scores were read), and the next
        // QK overlaps the accumulator's last PV and epilogue of this one
        if (!xq) {
          SegIter look = it;
          Seg nx;
          while (look.next(nx)) {
            if (!nx.empty) {
              if (kFp8) {
                qmul_next = load_q_f16(nx);
              } else if (!load_q_ring(rr)) {
                ok = false;
              }
              q_loaded = 1;
              break;
            }
          }
        }
      }
    } else {
      // ------------------------------------------------------------ rescale + epilogue (accumulator)
      const float* alpha_s = reinterpret_cast<const float*>(smem + kOffAlpha);
      const float2* l_s = reinterpret_cast<const float2*>(smem + kOffL);
      const uint32_t rLfree = mapa_shared(smem_u32(&bars->l_free), peer);
      const uint32_t rPfree0 = mapa_shared(smem_u32(&bars->pbuf_free[0]), peer);  // + 8 b: P buffer b's
      uint32_t ofull_ph = 0, epi_ph = 0, mrg_n = 0;
      auto epi_sync = [&]() -> bool {
        mbar_arrive(smem_u32(&bars->epi_bar));
        const bool done = kwait<kOutCold>(smem_u32(&bars->epi_bar), epi_ph, abort_flag);
        epi_ph ^= 1u;
        return done;
      };
      while (ok && it.next(s)) {
        const int r = s.rb * kRowsPerBlock + L;
        const bool row_valid = r < a.R;
        const size_t out_row = static_cast<size_t>(s.b) * a.R + r;
        if (s.empty) {  // no visible keys: zero output, lse -inf
          if (row_valid) {
            uint4* o = reinterpret_cast<uint4*>(a.out + out_row * kDv);
            for (int v = 0; v < kDv / 8; ++v) o[v] = make_uint4(0, 0, 0, 0);
            a.lse[out_row] = -INFINITY;
          }
          continue;
        }
        // A piece of a split unit with at most kFuseMax pieces takes its ticket
        // when its last P tile arrives (the order in which the unit's pieces
        // near their end); the atomic's result is first needed in the
        // epilogue, so nothing waits on it.  The piece with the last ticket
        // merges, after the others have written their partials (it waits on
        // their flags; they are on their last tile and wait on nothing).
        int split_first = 0, split_c0 = 0, split_k = 1, ticket = 0;
        if (s.split) {
          const int p0 = __ldg(a.pre + s.u), p1 = unit_end(a.pre, s.u, a.U, a.B);
          split_first = p0 + a.overhead;
          split_c0 = split_first / W;
          split_k = (p1 - 1) / W - split_c0 + 1;
        }
        for (int j = s.page_lo; j < s.page_hi; ++j, ++t) {
          const uint32_t sb = t % kPBufs, sph = (t / kPBufs) & 1u;
          if (ctid == 0) mbar_arrive_expect_tx(smem_u32(&bars->p_full[sb]), kPBytes + kVecBytes);
          if (!kwait<kOutWait, true>(smem_u32(&bars->p_full[sb]), sph, abort_flag)) { ok = false; break; }
          if (j + 1 == s.page_hi && s.split && split_k <= kFuseMax && ctid == 0)
            ticket = atomicAdd(a.unit_cnt + split_c0, 1);
          const float alpha = alpha_s[sb * kRowsPerBlock + L];
          if (__any_sync(0xffffffffu, alpha != 1.f) && j > s.page_lo) {
            // O must hold PV of the previous tile before it is rescaled
            const uint32_t pb = (t - 1u) % kPBufs, pph = ((t - 1u) / kPBufs) & 1u;
            if (!kwait<kOutWait>(smem_u32(&bars->pv_done[pb]), pph, abort_flag)) { ok = false; break; }
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

        // ---- epilogue.  Three cases:
        //  0  the unit is not split: O / l -> out (bf16), lse -> lse;
        //  1  a piece of a split unit: O / l (fp16, row-scaled) and lse -> its
        //     partial slot; when the unit has at most kFuseMax pieces, a ready
        //     flag follows;
        //  2  the last piece to finish of a unit with at most kFuseMax pieces:
        //     merges the other pieces' partials with its own O (the LSE merge)
        //     and writes out and lse itself.
        if (!kwait<kOutCold>(smem_u32(&bars->o_full), ofull_ph, abort_flag)) { ok = false; break; }
        ofull_ph ^= 1u;
        if (ctid == 0) mbar_arrive_expect_tx(smem_u32(&bars->l_full), kRowsPerBlock * 8);
        if (!kwait<kOutCold, true>(smem_u32(&bars->l_full), seg_n & 1u, abort_flag)) { ok = false; break; }
        const float2 lrow = l_s[L];  // (row sum, lse) of this piece
        ++seg_n;
        const float l = lrow.x, lse_own = lrow.y;
        int mode = 0;
        const int c0 = split_c0, k = split_k, first = split_first;
        if (s.split) {
          mode = 1;
          if (k <= kFuseMax) {
            if (ctid == 0) bars->ticket = ticket;
            if (!epi_sync()) { ok = false; break; }
            if (*reinterpret_cast<volatile int*>(&bars->ticket) == k - 1) mode = 2;
          }
        }
        // partial slot of piece i (cluster c0 + i) of this unit
        auto piece_slot = [&](int i) { return (i == 0 && first != c0 * W) ? 2 * c0 + 1 : 2 * (c0 + i); };
        // At the cluster's last segment the page ring is idle (all its pages
        // were consumed by the last PV and nothing more is loaded).
        bool ring_free = true;
        {
          SegIter look = it;
          Seg nx;
          while (look.next(nx))
            if (!nx.empty) {
              ring_free = false;
              break;
            }
        }
        const int row0 = s.rb * kRowsPerBlock + wq * 32;
        tc_fence_after();
        // Final rows go through the P buffer of the segment's last tile (its PV
        // is done; its credit goes back to the scorer only after this).
        const uint32_t last_sb = (t - 1u) % kPBufs;
        uint8_t* const est = smem + kOffP + last_sb * kPBytes + wq * (kPBytes / 4);
        if (mode == 1) {
          // fp16 partial O / l, scaled by a power of two that puts the row's
          // largest magnitude in [2^14, 2^15) (lse_part holds the scale): every
          // bf16-representable value within 2^-29 of the row maximum is stored
          // exactly, and nothing can overflow.  Chunk-interleaved slot: thread
          // L writes 8-channel chunk j of its row at [j][L], so each store
          // instruction covers 512 contiguous bytes.
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
          float amax = 0.f;
          for (int ch = 0; ch < 16; ++ch) {
            uint32_t o[32];
            tmem_ld32(tbase + lane_off + 32 * ch, o);
            tmem_wait_ld();
#pragma unroll
            for (int v = 0; v < 32; ++v) amax = fmaxf(amax, fabsf(__uint_as_float(o[v])));
          }
          float sc = 1.f;
          if (amax * inv_l > 0.f) {
            int e2;
            frexpf(amax * inv_l, &e2);  // amax / l < 2^e2
            sc = ldexpf(1.f, max(-120, min(120, e2 - 15)));
          }
          const float f = inv_l / sc;
          uint4* part = reinterpret_cast<uint4*>(a.o_part) + static_cast<size_t>(s.slot) * kPartChunks * kRowsPerBlock + L;
          for (int ch = 0; ch < 16; ++ch) {
            uint32_t o[32];
            tmem_ld32(tbase + lane_off + 32 * ch, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 4; ++q)
              part[static_cast<size_t>(4 * ch + q) * kRowsPerBlock] =
                  make_uint4(pack_f16x2(__uint_as_float(o[8 * q + 0]) * f, __uint_as_float(o[8 * q + 1]) * f),
                             pack_f16x2(__uint_as_float(o[8 * q + 2]) * f, __uint_as_float(o[8 * q + 3]) * f),
                             pack_f16x2(__uint_as_float(o[8 * q + 4]) * f, __uint_as_float(o[8 * q + 5]) * f),
                             pack_f16x2(__uint_as_float(o[8 * q + 6]) * f, __uint_as_float(o[8 * q + 7]) * f));
          }
          // O has been read and the last tile's P buffer is not used here: the
          // next segment's PV may start while the stores drain
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->o_free));
          if (ctid == 0) mbar_arrive_remote(rPfree0 + 8u * last_sb);
          reinterpret_cast<float2*>(a.lse_part)[static_cast<size_t>(s.slot) * kRowsPerBlock + L] = make_float2(lse_own, sc);
          __threadfence();  // the partial is visible GPU-wide before its ready flag
        } else if (mode == 0) {
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
          for (int cc = 0; cc < 8; ++cc) {
            float v[64];
            {
              uint32_t o0[32], o1[32];
              tmem_ld32(tbase + lane_off + 64 * cc, o0);
              tmem_ld32(tbase + lane_off + 64 * cc + 32, o1);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                v[i] = __uint_as_float(o0[i]) * inv_l;
                v[32 + i] = __uint_as_float(o1[i]) * inv_l;
              }
            }
            if (ring_free) {  // two 16 KB half boxes per warp, staged in the idle ring
              uint8_t* hb = smem + (cc >> 2) * 65536 + wq * 16384;
              stage_half(hb, v, cc & 3, lane);
              if ((cc & 3) == 3) store_half(hb, &out_map4, cc >> 2, row0, s.b, a.R, lane);
            } else {
              store_rows_tma(est, v, &out_map, cc, row0, s.b, a.R, lane);
            }
          }
          if (row_valid) a.lse[out_row] = lse_own;
        } else {
          // Incremental LSE merge: one other piece per pass, each pass as soon
          // as that piece's partial is ready, the unit's pieces taken from its
          // tail (later pieces start their clusters, so they finish first).
          // Running result out_run (O times a factor, in TMEM between passes)
          // and lse_run, starting from the own piece: O / l and lse_own.  With
          // partial j (lse_j, stored values times sc_j):
          //   m = max(lse_run, lse_j), e_r = exp(lse_run - m), e_j = exp(lse_j - m),
          //   out_run <- (e_r out_run + e_j sc_j stored_j) / (e_r + e_j),
          //   lse_run <- m + ln(e_r + e_j).
          // (The other pieces hold tickets: they are on their last tile or in
          // their epilogues and wait on nothing outside their cluster.)
          float lse_run = lse_own;
          float o_scale = l > 0.f ? 1.f / l : 0.f;  // O / l is the own piece's result
          const int own = c - c0;
          for (int pi = 0; pi < k - 1 && ok; ++pi) {
            const int cand = k - 1 - pi;
            const int i = cand > own ? cand : cand - 1;  // k-1, ..., 0 without own
            if (ctid == 0 && !wait_flag_gpu(a.slot_ready + piece_slot(i))) atomicOr(a.err, kErrTimeout);
            if (!epi_sync()) { ok = false; break; }  // partial i is complete and visible
            const float2 ls = __ldcg(reinterpret_cast<const float2*>(a.lse_part) +
                                     static_cast<size_t>(piece_slot(i)) * kRowsPerBlock + L);
            const float mm = fmaxf(lse_run, ls.x);
            float a_run = 0.f, cf = 0.f;  // factors on the running result and on the stored partial
            if (mm != -INFINITY) {
              const float er = ex2_approx((lse_run - mm) * kLog2e), ej = ex2_approx((ls.x - mm) * kLog2e);
              const float inv = 1.f / (er + ej);
              a_run = er * inv * o_scale;
              cf = ej * inv * ls.y;
              lse_run = mm + lg2_approx(er + ej) * kLn2;
            }
            o_scale = 1.f;
            const uint4* gsrc = reinterpret_cast<const uint4*>(a.o_part) +
                                static_cast<size_t>(piece_slot(i)) * kPartChunks * kRowsPerBlock;
            const uint4* src = gsrc + L;
            if (ring_free) {
              if (ctid == 0) {
                const uint32_t mb = smem_u32(&bars->mrg_bar);
                mbar_arrive_expect_tx(mb, kPartBytes);
                for (int off = 0; off < kPartBytes; off += 32768)
                  bulk_load(smem_u32(smem + off), reinterpret_cast<const uint8_t*>(gsrc) + off, 32768, mb);
              }
              if (!kwait<kOutCold>(smem_u32(&bars->mrg_bar), mrg_n & 1u, abort_flag)) { ok = false; break; }
              ++mrg_n;
              src = reinterpret_cast<const uint4*>(smem) + L;
            }
            const bool last_pass = pi == k - 2;
            for (int cc = 0; cc < 8; ++cc) {
              float v[64];
              {
                uint32_t o0[32], o1[32];
                tmem_ld32(tbase + lane_off + 64 * cc, o0);
                tmem_ld32(tbase + lane_off + 64 * cc + 32, o1);
                tmem_wait_ld();
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                  v[x] = __uint_as_float(o0[x]) * a_run;
                  v[32 + x] = __uint_as_float(o1[x]) * a_run;
                }
              }
              uint4 w[8];
#pragma unroll
              for (int q = 0; q < 8; ++q)
                w[q] = ring_free ? src[static_cast<size_t>(8 * cc + q) * kRowsPerBlock]
                                 : __ldcg(src + static_cast<size_t>(8 * cc + q) * kRowsPerBlock);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const uint32_t ww[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                  const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&ww[h]));
                  v[8 * q + 2 * h] += cf * f2.x;
                  v[8 * q + 2 * h + 1] += cf * f2.y;
                }
              }
              if (last_pass && ring_free) {
                // half 0 staged in the ring's free top 64 KB; half 1 where the
                // partial's chunks 0..31 were (read by every warp before it)
                uint8_t* hb = (cc < 4 ? smem + 2 * 65536 : smem) + wq * 16384;
                stage_half(hb, v, cc & 3, lane);
                if ((cc & 3) == 3) store_half(hb, &out_map4, cc >> 2, row0, s.b, a.R, lane);
                if (cc == 3 && !epi_sync()) { ok = false; break; }
              } else if (last_pass) {
                store_rows_tma(est, v, &out_map, cc, row0, s.b, a.R, lane);
              } else {
                uint32_t o0[32], o1[32];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                  o0[x] = __float_as_uint(v[x]);
                  o1[x] = __float_as_uint(v[32 + x]);
                }
                tmem_st32(tbase + lane_off + 64 * cc, o0);
                tmem_st32(tbase + lane_off + 64 * cc + 32, o1);
              }
            }
            if (!last_pass) tmem_wait_st();
            if (ring_free && !last_pass && !epi_sync()) { ok = false; break; }  // ring read before the next copy
          }
          if (!ok) break;
          if (row_valid) a.lse[out_row] = lse_run;
          if (ctid == 0) {  // leave the flags and the counter clear for the next call
            for (int i = 0; i < k; ++i)
              if (c0 + i != c) a.slot_ready[piece_slot(i)] = 0;
            a.unit_cnt[c0] = 0;
          }
        }
        tc_fence_before();
        // mode 1: every thread's partial is fenced before the flag; otherwise
        // all four warps are done with the staging buffer and with O
        if (!epi_sync()) { ok = false; break; }
        if (mode == 1) {
          if (ctid == 0 && k <= kFuseMax) st_release_gpu(a.slot_ready + s.slot, 1);
        } else {
          mbar_arrive(smem_u32(&bars->o_free));
          if (ctid == 0) mbar_arrive_remote(rPfree0 + 8u * last_sb);
        }
        // the row sums were read long ago (a remote arrive stalls its thread
        // for about a microsecond, so it comes last)
        if (lane == 0) mbar_arrive_remote(rLfree);
      }
    }
    if (!ok && !*abort_flag) signal_abort(bars, a.err, peer);
    if (!scorer && lane == 0) bulk_wait_all();  // output stores complete before the CTA ends
  } else if (kFp8 && (kRopeB || warp != 9)) {
    // ---------------------------------------------------------------- fp8 dequant (warps 6-8, and 10 or 9)
    // This CTA's raw e4m3 chunks (64-byte swizzled, in the top of its stage)
    // -> fp16 blocks of the same stage, 128-byte swizzled as the MMA
    // descriptors expect.  The scorer writes the exact codes of its 9 blocks
    // (variant B: the 8 latent blocks, and the RoPE block from bf16) and the
    // tokens' group scales into the stage's scale slot; the accumulator writes
    // code x scale for the 8 latent blocks.  Thread = (token t, half h): it
    // reads all its raw pieces into registers, the 128 threads meet (the fp16
    // blocks overwrite the raw chunks in place), then it converts and writes.
    // Rows past seqlen and pages with a bad id (read as zeros by TMA) are
    // written as zeros, with scale 0.
    const int dq = kRopeB ? tid - 192 : (warp == 10 ? 3 : warp - 6) * 32 + lane;  // 0..127
    const int t = dq & 63, h = dq >> 6;
    constexpr int kPieces = 18;                     // 16-channel pieces per thread (the scorer's count)
    const int n = scorer ? 18 : 16;                 // scorer: 36 pieces per token; accumulator: 32
    const int f0 = n * h;
    const uint32_t raw_off = static_cast<uint32_t>(scorer ? (kRopeB ? kRawOffSB : kRawOffS) : kRawOffA);
    const uint8_t* kv8 = reinterpret_cast<const uint8_t*>(a.kv);
    SegIter it = it0;
    Seg s;
    int stage = 0;
    uint32_t ph = 0, sync_ph = 0;
    bool ok = true;
    while (ok && it.next(s)) {
      if (s.empty) continue;
      const int seqlen = clamp_seqlen(__ldg(a.seqlens + s.b), a.max_pages);
      const int32_t* bt = a.block_table + static_cast<size_t>(s.b) * a.max_pages;
      const int dl = dq & 31;
      int ids = 0;  // page ids 32 at a time, one per lane
      for (int p = s.page_lo; p < s.page_hi; ++p) {
        const int slot = (p - s.page_lo) & 31;
        if (slot == 0) ids = p + dl < s.page_hi ? __ldg(bt + p + dl) : 0;
        const int pid = __shfl_sync(0xffffffffu, ids, slot);
        const bool bad = pid < 0 || pid >= a.num_pages;  // the loader reports it
        const bool live = !bad && t < seqlen - p * kPage;
        const size_t row = static_cast<size_t>(live ? pid : 0) * kPage + t;
        // scales of this thread's groups: the accumulator's two latent groups
        // (2h, 2h + 1); the scorer's half-0 threads fetch all five for the softmax
        float sg[kGroups] = {0.f, 0.f, 0.f, 0.f, 0.f};
        if (live && (!scorer || h == 0)) {
          if (kRopeB) {
            const float4 s4 = __ldg(reinterpret_cast<const float4*>(kv8 + row * kFp8bRecord + kFp8bScaleOffset));
            sg[0] = s4.x;
            sg[1] = s4.y;
            sg[2] = s4.z;
            sg[3] = s4.w;
            sg[4] = 1.f;  // the bf16 RoPE carries no scale
          } else {
            const float* sp = a.kv_scales + row * kGroups;
#pragma unroll
            for (int g = 0; g < kGroups; ++g) sg[g] = __ldg(sp + g);
          }
        }
        // warp-uniform outcomes (the page-id shuffle above is warp-wide)
        if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->raw_full[stage]), ph, abort_flag))) {
          ok = false;
          break;
        }
        uint8_t* const dst = smem + stage * (scorer ? kStageS : kStageO);
        const uint8_t* const raw = dst + raw_off + t * 64;
        const int sw = t & 7, rsw = (t >> 1) & 3;
        // raw pieces -> registers (variant B RoPE pieces, f >= 32, are 32 bytes of bf16)
        uint4 ra[kPieces], rb[4];
#pragma unroll
        for (int i = 0; i < kPieces; ++i) {
          ra[i] = make_uint4(0, 0, 0, 0);
          const int f = f0 + i;
          if (i < n && live) {
            if (kRopeB && f >= 32) {
              const int qr = f - 32;
              const uint8_t* rr = raw + (8 + (qr >> 1)) * kRawSlot;
              ra[i] = *reinterpret_cast<const uint4*>(rr + (((2 * (qr & 1)) ^ rsw) << 4));
              if (i >= kPieces - 4) rb[i - (kPieces - 4)] = *reinterpret_cast<const uint4*>(rr + (((2 * (qr & 1) + 1) ^ rsw) << 4));
            } else {
              ra[i] = *reinterpret_cast<const uint4*>(raw + (f >> 2) * kRawSlot + (((f & 3) ^ rsw) << 4));
            }
          }
        }
        // every thread has its raw pieces: the fp16 blocks may now overwrite them
        mbar_arrive(smem_u32(&bars->dq_sync));
        if (!__all_sync(0xffffffffu, kwait<kOutWait>(smem_u32(&bars->dq_sync), sync_ph, abort_flag))) {
          ok = false;
          break;
        }
        sync_ph ^= 1u;
        bool out_of_range = false;
        __half2 shi[2], slo[2];
        if (!scorer) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const float sv = sg[2 * h + q];
            out_of_range |= live && !(fabsf(sv) * 448.f <= 65504.f);
            const __half hs = __float2half_rn(sv);
            shi[q] = __half2half2(hs);
            slo[q] = __half2half2(__float2half_rn(sv - __half2float(hs)));
          }
        }
#pragma unroll
        for (int i = 0; i < kPieces; ++i) {
          if (i < n) {
            const int f = f0 + i;
            const int c = 64 * (f >> 2) + 16 * (f & 3);  // first channel of the piece (variant B RoPE: 512 + 16 qr)
            uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
            if (live) {
              const uint4 r = ra[i];
              if (kRopeB && f >= 32) {
                // 16 bf16 RoPE channels -> fp16, exact inside the fp16 range
                const uint4 r1 = i >= kPieces - 4 ? rb[i - (kPieces - 4)] : make_uint4(0, 0, 0, 0);
                const uint32_t w[8] = {r.x, r.y, r.z, r.w, r1.x, r1.y, r1.z, r1.w};
                uint32_t hw[8];
                float amax = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  const float lo = bf16_lo(w[k]), hi = bf16_hi(w[k]);
                  amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
                  hw[k] = pack_f16x2(lo, hi);
                }
                out_of_range |= !(amax <= 65504.f);
                o0 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                o1 = make_uint4(hw[4], hw[5], hw[6], hw[7]);
              } else if (scorer) {
                // the exact codes (every e4m3 value is an fp16 value)
                o0.x = e4m3x2_f16x2(static_cast<uint16_t>(r.x & 0xFFFFu));
                o0.y = e4m3x2_f16x2(static_cast<uint16_t>(r.x >> 16));
                o0.z = e4m3x2_f16x2(static_cast<uint16_t>(r.y & 0xFFFFu));
                o0.w = e4m3x2_f16x2(static_cast<uint16_t>(r.y >> 16));
                o1.x = e4m3x2_f16x2(static_cast<uint16_t>(r.z & 0xFFFFu));
                o1.y = e4m3x2_f16x2(static_cast<uint16_t>(r.z >> 16));
                o1.z = e4m3x2_f16x2(static_cast<uint16_t>(r.w & 0xFFFFu));
                o1.w = e4m3x2_f16x2(static_cast<uint16_t>(r.w >> 16));
              } else {
                const int q = (c >> 7) - 2 * h;           // which of the thread's two groups
                const __half2 hh = q ? shi[1] : shi[0], ll = q ? slo[1] : slo[0];
                o0.x = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.x & 0xFFFFu), hh, ll);
                o0.y = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.x >> 16), hh, ll);
                o0.z = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.y & 0xFFFFu), hh, ll);
                o0.w = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.y >> 16), hh, ll);
                o1.x = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.z & 0xFFFFu), hh, ll);
                o1.y = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.z >> 16), hh, ll);
                o1.z = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.w & 0xFFFFu), hh, ll);
                o1.w = e4m3x2_scaled_f16x2(static_cast<uint16_t>(r.w >> 16), hh, ll);
              }
            }
            const int c8 = (c & 63) >> 3;
            uint8_t* const rowp = dst + (c >> 6) * kBox + t * 128;
            *reinterpret_cast<uint4*>(rowp + ((c8 ^ sw) << 4)) = o0;
            *reinterpret_cast<uint4*>(rowp + (((c8 + 1) ^ sw) << 4)) = o1;
          }
        }
        if (scorer && h == 0) {  // the tokens' scales for the softmax, [group][token]
          float* slot_sc = reinterpret_cast<float*>(smem + kOffScale + stage * kScaleSlotBytes);
#pragma unroll
          for (int g = 0; g < kGroups; ++g) slot_sc[g * 64 + t] = sg[g];
        }
        if (out_of_range) atomicOr(a.err, kErrRange);
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&bars->kv_full[stage]));
        if (++stage == nst) {
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

static cudaLaunchConfig_t make_cfg(bool fp8, bool rope_b, int clusters, cudaStream_t stream, cudaLaunchAttribute* attr,
                                   bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  cfg.blockDim = dim3(!fp8 ? Cfg<false>::kThreads : (rope_b ? Cfg<true, true>::kThreads : Cfg<true, false>::kThreads), 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the prologue may overlap the planner
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

static cudaError_t set_smem_attr(bool fp8) {
  if (fp8) {
    cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(mla_decode_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  }
  return cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t decode_max_active_clusters(bool fp8, int* clusters) {
  cudaError_t e = set_smem_attr(fp8);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_cfg(fp8, false, 1, nullptr, attr);
  // both fp8 variants have the same shared memory (one CTA per SM)
  if (fp8) return cudaOccupancyMaxActiveClusters(clusters, mla_decode_kernel<true, false>, &cfg);
  return cudaOccupancyMaxActiveClusters(clusters, mla_decode_kernel<false>, &cfg);
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kv_map_s, const CUtensorMap& kv_map_a,
                          const CUtensorMap& kv_map_r, const CUtensorMap& q_map, const CUtensorMap& out_map, const CUtensorMap& out_map4,
                          int clusters, bool fp8, cudaStream_t stream) {
  cudaError_t e = set_smem_attr(fp8);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = make_cfg(fp8, fp8 && a.rope_bf16, clusters, stream, attr, true);
  if (fp8 && a.rope_bf16)
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, true>, kv_map_s, kv_map_a, kv_map_r, q_map, out_map,
                              out_map4, a);
  if (fp8)
    return cudaLaunchKernelEx(&cfg, mla_decode_kernel<true, false>, kv_map_s, kv_map_a, kv_map_r, q_map, out_map,
                              out_map4, a);
  return cudaLaunchKernelEx(&cfg, mla_decode_kernel<false>, kv_map_s, kv_map_a, kv_map_r, q_map, out_map, out_map4, a);
}

}  // namespace mla_gb300
