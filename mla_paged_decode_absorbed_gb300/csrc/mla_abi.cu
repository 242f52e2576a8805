// C ABI of the MLA paged-decode library (declared in include/mla.h): argument
// validation, workspace layout, the split planner kernel, the LSE combine
// kernel, tensor-map encoding and the launch sequence on the caller's stream.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "mla.h"
#include "mla_internal.h"

namespace mla_gb300 {

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kCombineSplit = 4;          // threads per (row, chunk): each merges every 4th piece
constexpr int kCombineThreads = 128 * kCombineSplit;
constexpr int kCombineBatch = 8;         // partial pieces whose loads a combine thread keeps in flight
constexpr int kCombineJobColumns = 3;    // CTA columns of the combine grid; column x takes jobs x, x + 3, ...

// ------------------------------------------------------------------ planner
// Cost of unit u (row block rb = u / B of request b = u % B): the pages the
// block's last row can see, plus a fixed overhead for the unit's prologue and
// epilogue.  seqlen outside [0, 64*max_pages] is clamped and flagged.
__device__ __forceinline__ int unit_cost(const int32_t* seqlens, int u, int B, int s_q, int H, int R,
                                         int max_pages, int ovh, int32_t* err) {
  const int b = u % B, rb = u / B;
  int seqlen = seqlens[b];
  if (seqlen < 0 || seqlen > max_pages * kPage) {
    atomicOr(err, kErrBounds);
    seqlen = seqlen < 0 ? 0 : max_pages * kPage;
  }
  const int r_last = min(R, (rb + 1) * kRowsPerBlock) - 1;
  int n = seqlen - s_q + r_last / H + 1;
  n = n < 0 ? 0 : (n > seqlen ? seqlen : n);
  return (n + kPage - 1) / kPage + ovh;
}

// One CTA: per-unit costs laid out on the cost axis (`pre`: unit starts,
// then the end of the last unit, then the end of each row block's stretch),
// the per-cluster budget W, the first unit each cluster touches, and the
// units with more than kFuseMax pieces.  Also clears the merge counters and
// partial-slot flags the attention kernel uses.
//
// Layout: the units of a row block (rb-major order u = rb * B + b) lie back
// to back.  With several row blocks and at least as many clusters, row
// block r gets its own Gl = G / n_rb clusters and starts at r * Gl * W, with
// W = max_r ceil(total_r / Gl): cluster r * Gl + g then covers the same
// stretch of every request's pages for each r, so the row blocks of a
// request read each page at about the same time and the second read comes
// from L2.  Otherwise the row blocks follow each other and W = ceil(total / G).
constexpr int kMaxRowBlocks = 128;  // s_q <= 16, H <= 1024

__global__ void __launch_bounds__(kPlanThreads) mla_plan_kernel(const int32_t* seqlens, int B, int s_q, int H,
                                                                int R, int U, int max_pages, int G, int ovh,
                                                                int32_t* hdr, int32_t* cl_first, int32_t* pre,
                                                                int32_t* sync) {
  __shared__ int warp_sum[32];
  __shared__ int s_total, s_njobs, s_W;
  __shared__ int s_rb[kMaxRowBlocks + 1];   // prefix of costs at each row block's first unit
  __shared__ int s_base[kMaxRowBlocks];     // each row block's start on the cost axis
  // the attention kernel may start its prologue now; it reads the plan only
  // after this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" :::);
  const int tid = threadIdx.x, T = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int n_rb = U / B;
  if (tid == 0) {
    hdr[kHdrErr] = 0;
    hdr[kHdrStall] = 0;
    s_njobs = 0;
  }
  for (int i = tid; i < 4 * G; i += T) sync[i] = 0;
  for (int c = tid; c < G; c += T) cl_first[c] = U;
  __syncthreads();
  int32_t* err = hdr + kHdrErr;
  const int chunk = (U + T - 1) / T;
  const int u0 = min(U, tid * chunk), u1 = min(U, u0 + chunk);
  int local = 0;
  for (int u = u0; u < u1; ++u) local += unit_cost(seqlens, u, B, s_q, H, R, max_pages, ovh, err);
  // block-wide exclusive scan of `local` (everything after it stays on chip
  // except the writes of the plan itself)
  int incl = local;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int nw = T / 32;
    int v = lane < nw ? warp_sum[lane] : 0;
    int vi = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, vi, d);
      if (lane >= d) vi += x;
    }
    if (lane < nw) warp_sum[lane] = vi - v;  // exclusive warp offsets
    if (lane == nw - 1) s_total = vi;
  }
  __syncthreads();
  const int total = s_total;
  const int start = warp_sum[warp] + incl - local;  // prefix of costs at u0
  {
    int run = start;
    for (int u = u0; u < u1; ++u) {
      if (u % B == 0) s_rb[u / B] = run;
      run += unit_cost(seqlens, u, B, s_q, H, R, max_pages, ovh, err);
    }
    if (tid == 0) s_rb[n_rb] = total;
  }
  __syncthreads();
  if (tid == 0) {
    const bool lockstep = n_rb > 1 && G >= n_rb;
    int W = 1;
    if (lockstep) {
      const int gl = G / n_rb;
      for (int r = 0; r < n_rb; ++r) W = max(W, (s_rb[r + 1] - s_rb[r] + gl - 1) / gl);
      for (int r = 0; r < n_rb; ++r) s_base[r] = r * gl * W;
    } else {
      W = max(1, (total + G - 1) / G);
      for (int r = 0; r < n_rb; ++r) s_base[r] = s_rb[r];
    }
    s_W = W;
    for (int r = 0; r < n_rb; ++r) pre[U + 1 + r] = s_base[r] + s_rb[r + 1] - s_rb[r];
    pre[U] = s_base[n_rb - 1] + s_rb[n_rb] - s_rb[n_rb - 1];
    hdr[kHdrW] = W;
    hdr[kHdrTotal] = pre[U];
    hdr[kHdrUnits] = U;
    hdr[kHdrClusters] = G;
    hdr[kHdrOvh] = ovh;
  }
  __syncthreads();
  const int W = s_W;
  // combine jobs: units of more than kFuseMax pieces, as (unit, first cluster,
  // last cluster, slot of the first piece); at most one per first cluster
  int4* jobs = reinterpret_cast<int4*>(sync + 4 * G);
  int run = start;
  for (int u = u0; u < u1; ++u) {
    const int cost = unit_cost(seqlens, u, B, s_q, H, R, max_pages, ovh, err);
    const int r = u / B;
    const int p0 = s_base[r] + run - s_rb[r], p1 = p0 + cost;
    run += cost;
    pre[u] = p0;
    const int cf = (p0 + W - 1) / W, cl = (p1 + W - 1) / W - 1;
    for (int c = cf; c <= cl && c < G; ++c) cl_first[c] = u;
    if (p1 - p0 > ovh) {
      const int first = p0 + ovh, c0 = first / W, c1 = (p1 - 1) / W;
      if (c1 - c0 + 1 > kFuseMax) {
        const int j = atomicAdd(&s_njobs, 1);
        jobs[j] = make_int4(u, c0, c1, first != c0 * W ? 2 * c0 + 1 : 2 * c0);
      }
    }
  }
  __syncthreads();
  const int njobs = s_njobs;
  if (tid == 0) hdr[kHdrCombine] = njobs;
  for (int j = njobs + tid; j < G; j += T) jobs[j] = make_int4(-1, 0, 0, 0);  // no job
}

// ------------------------------------------------------------------ combine
// Part q of one combine job's merge for 8-channel chunk j of row L of the
// unit's row block: pieces c + q, c + q + kCombineSplit, ... in batches of
// kCombineBatch (all loads of a batch issued together), with a running
// maximum: returns (max lse, sum of exp(lse_k - max), sum of
// exp(lse_k - max) * out_k over 8 channels), out_k = stored_k * scale_k.
__device__ __forceinline__ void combine_part(const float2* lp, const uint4* op, int4 job, int L, int j, int q,
                                             float& mx, float& wsum, float (&acc)[8]) {
  const int c = job.y, last = job.z, slot0 = job.w;
  mx = -INFINITY;
  wsum = 0.f;
#pragma unroll
  for (int h = 0; h < 8; ++h) acc[h] = 0.f;
  for (int cb = c + q; cb <= last; cb += kCombineSplit * kCombineBatch) {
    float2 ls[kCombineBatch];
    uint4 o[kCombineBatch];
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const int cc = cb + kCombineSplit * i;
      ls[i] = make_float2(-INFINITY, 0.f);
      o[i] = make_uint4(0, 0, 0, 0);
      if (cc <= last) {
        const size_t slot = static_cast<size_t>(cc == c ? slot0 : 2 * cc);
        ls[i] = lp[slot * kRowsPerBlock + L];
        o[i] = op[(slot * kPartChunks + j) * kRowsPerBlock + L];
      }
    }
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) bm = fmaxf(bm, ls[i].x);
    const float m_new = fmaxf(mx, bm);
    if (m_new == -INFINITY) continue;  // no piece saw a key of this row yet
    const float keep = mx == -INFINITY ? 0.f : expf(mx - m_new);
    wsum *= keep;
#pragma unroll
    for (int h = 0; h < 8; ++h) acc[h] *= keep;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const float w = expf(ls[i].x - m_new);  // 0 for a piece that saw no key of this row
      wsum += w;
      const float ws = w * ls[i].y;
      const uint32_t ow[4] = {o[i].x, o[i].y, o[i].z, o[i].w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ow[h]));
        acc[2 * h] += ws * f.x;
        acc[2 * h + 1] += ws * f.y;
      }
    }
    mx = m_new;
  }
}

// Units with at most kFuseMax pieces are merged inside the attention kernel;
// this kernel merges the others (the planner's job list: unit, first and last
// cluster, slot of the first piece).  CTA (j, x) takes the 8-channel chunk j
// of every row (64 chunks, so a single job already keeps 64 SMs busy) of jobs
// x, x + kCombineJobColumns, ... (the jobs' rounds of dependent loads then
// overlap instead of adding up); thread (q, L) takes
// row L and every kCombineSplit-th piece from q, so the chunk-interleaved
// fp16 partial slots are read with coalesced loads.  The kCombineSplit part
// merges meet in shared memory, and thread (0, L) finishes the row:
//   lse = ln sum_k exp(lse_k),  out = sum_k exp(lse_k - lse) * out_k.
__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(const CombineArgs a) {
  __shared__ float s_m[kCombineSplit][kRowsPerBlock], s_w[kCombineSplit][kRowsPerBlock];
  __shared__ float s_acc[kCombineSplit][8][kRowsPerBlock];
  // launched as a programmatic dependent of the attention kernel: wait for it
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int L = threadIdx.x & (kRowsPerBlock - 1);  // row within the block
  const int q = threadIdx.x >> 7;                   // which pieces
  const int j = blockIdx.x;                         // 8-channel chunk
  const float2* lp = reinterpret_cast<const float2*>(a.lse_part);
  const uint4* op = reinterpret_cast<const uint4*>(a.o_part);
  // the planner packs the jobs in front of the unused slots, which hold unit -1
  const int4* jobs = reinterpret_cast<const int4*>(a.sync + 4 * a.clusters);
  for (int jb = blockIdx.y; jb < a.clusters; jb += gridDim.y) {
    const int4 job = jobs[jb];
    if (job.x < 0) break;  // the same job for every thread of the CTA
    const int b = job.x % a.B, rb = job.x / a.B;
    const int r = rb * kRowsPerBlock + L;
    float mx, wsum, acc[8];
    if (r < a.R) {
      combine_part(lp, op, job, L, j, q, mx, wsum, acc);
    } else {
      mx = -INFINITY;
      wsum = 0.f;
#pragma unroll
      for (int h = 0; h < 8; ++h) acc[h] = 0.f;
    }
    s_m[q][L] = mx;
    s_w[q][L] = wsum;
#pragma unroll
    for (int h = 0; h < 8; ++h) s_acc[q][h][L] = acc[h];
    __syncthreads();
    if (q == 0 && r < a.R) {
      float m = -INFINITY;
#pragma unroll
      for (int k = 0; k < kCombineSplit; ++k) m = fmaxf(m, s_m[k][L]);
      float w = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (m != -INFINITY) {
#pragma unroll
        for (int k = 0; k < kCombineSplit; ++k) {
          const float mk = s_m[k][L];
          if (mk == -INFINITY) continue;  // that part saw no key of this row
          const float e = expf(mk - m);
          w += e * s_w[k][L];
#pragma unroll
          for (int h = 0; h < 8; ++h) o[h] += e * s_acc[k][h][L];
        }
      }
      const float inv = w > 0.f ? 1.f / w : 0.f;
      const size_t orow = static_cast<size_t>(b) * a.R + r;
      uint32_t packed[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        __nv_bfloat162 v = __floats2bfloat162_rn(o[2 * h] * inv, o[2 * h + 1] * inv);
        packed[h] = *reinterpret_cast<uint32_t*>(&v);
      }
      reinterpret_cast<uint4*>(a.out + orow * kDv)[j] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
      if (j == 0) a.lse[orow] = w > 0.f ? m + logf(w) : -INFINITY;
    }
    __syncthreads();  // the shared arrays are rewritten by the next job
  }
}


// ------------------------------------------------------------------ combine of caller partials
// mla_combine(): the LSE merge of fp32 partials a caller computed.  One warp
// per (request b, row r): the lanes first reduce the partials' lse maximum,
// then walk the partials four at a time; lane l owns output channels
// [8l, 8l + 8) and [256 + 8l, 256 + 8l + 8), so every load instruction of the
// warp reads 1 KB of one partial row in 16-byte pieces and every store writes
// 512 contiguous bytes of bf16.  A partial whose lse is -inf is skipped (its
// row is never read: it may hold anything).
constexpr int kCpWarps = 8;

__device__ __forceinline__ void fma4(float (&acc)[4], float w, const float4 v) {
  acc[0] += w * v.x;
  acc[1] += w * v.y;
  acc[2] += w * v.z;
  acc[3] += w * v.w;
}

__global__ void __launch_bounds__(32 * kCpWarps) mla_combine_partials_kernel(
    const float* __restrict__ o_part, const float* __restrict__ lse_part, const int32_t* __restrict__ indptr,
    int num_partials, int R, uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.y * kCpWarps + (threadIdx.x >> 5);
  const int b = blockIdx.x;
  if (r >= R) return;
  const int k0 = max(0, __ldg(indptr + b)), k1 = min(num_partials, __ldg(indptr + b + 1));
  float m = -INFINITY;
  for (int k = k0 + lane; k < k1; k += 32) m = fmaxf(m, __ldg(lse_part + static_cast<size_t>(k) * R + r));
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, d));
  float acc[4][4] = {};  // [lo chunk 0, lo chunk 1, hi chunk 0, hi chunk 1][4]
  float wsum = 0.f;
  if (m != -INFINITY) {
    for (int kb = k0; kb < k1; kb += 4) {
      float w[4];
      float4 v[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int k = kb + i;
        const float l = k < k1 ? __ldg(lse_part + static_cast<size_t>(k) * R + r) : -INFINITY;
        w[i] = l == -INFINITY ? 0.f : expf(l - m);
        if (w[i] > 0.f) {
          const float4* src = reinterpret_cast<const float4*>(o_part + (static_cast<size_t>(k) * R + r) * kDv);
          v[i][0] = __ldg(src + 2 * lane);
          v[i][1] = __ldg(src + 2 * lane + 1);
          v[i][2] = __ldg(src + 64 + 2 * lane);
          v[i][3] = __ldg(src + 64 + 2 * lane + 1);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) v[i][j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        wsum += w[i];
#pragma unroll
        for (int j = 0; j < 4; ++j) fma4(acc[j], w[i], v[i][j]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  const size_t orow = static_cast<size_t>(b) * R + r;
  uint4* dst = reinterpret_cast<uint4*>(out + orow * kDv);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t pk[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float* a2 = acc[2 * h + (q >> 1)];
      __nv_bfloat162 x = __floats2bfloat162_rn(a2[2 * (q & 1)] * inv, a2[2 * (q & 1) + 1] * inv);
      pk[q] = *reinterpret_cast<uint32_t*>(&x);
    }
    dst[32 * h + lane] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  }
  if (lane == 0) lse[orow] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
}


// ------------------------------------------------------------------ host helpers
size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Dims {
  int B, s_q, H, R, n_rb, U, P, maxp, ovh;
  bool fp8;        // an fp8 cache (variant A or B)
  bool rope_bf16;  // fp8 variant B: 656-byte token records with the RoPE in bf16
};

mla_status check_desc(const mla_desc* d, Dims* out) {
  if (!d) return MLA_ERR_INVALID_ARG;
  if (d->page_size != kPage || d->d_qk != kDqk || d->d_v != kDv) return MLA_ERR_UNSUPPORTED;
  if (d->kv_dtype != MLA_KV_BF16 && d->kv_dtype != MLA_KV_FP8_E4M3 && d->kv_dtype != MLA_KV_FP8_E4M3_ROPE_BF16)
    return MLA_ERR_UNSUPPORTED;
  if (d->batch < 1 || d->s_q < 1 || d->s_q > 16 || d->num_heads < 1 || d->num_heads > 1024) return MLA_ERR_INVALID_ARG;
  if (d->num_pages < 1 || d->max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if (d->max_clusters < 0 || d->plan_overhead < 0) return MLA_ERR_INVALID_ARG;
  for (int i = 0; i < 5; ++i)
    if (d->reserved[i] != 0) return MLA_ERR_INVALID_ARG;
  Dims x;
  x.B = d->batch;
  x.s_q = d->s_q;
  x.H = d->num_heads;
  x.R = d->s_q * d->num_heads;
  x.n_rb = (x.R + kRowsPerBlock - 1) / kRowsPerBlock;
  x.P = d->num_pages;
  x.maxp = d->max_pages_per_seq;
  x.ovh = d->plan_overhead > 0 ? d->plan_overhead : kDefaultOverhead;
  x.fp8 = d->kv_dtype == MLA_KV_FP8_E4M3 || d->kv_dtype == MLA_KV_FP8_E4M3_ROPE_BF16;
  x.rope_bf16 = d->kv_dtype == MLA_KV_FP8_E4M3_ROPE_BF16;
  const int64_t U = static_cast<int64_t>(x.B) * x.n_rb;
  // the plan's int32 cost prefix and page*64 token indices must not overflow
  if (U * (static_cast<int64_t>(x.maxp) + x.ovh) >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(x.maxp) * kPage >= (int64_t(1) << 31)) return MLA_ERR_INVALID_ARG;
  x.U = static_cast<int>(U);
  if (out) *out = x;
  return MLA_OK;
}

mla_workspace_layout layout_for(const Dims& x, int G) {
  mla_workspace_layout l;
  size_t off = 0;
  l.header = off;
  off += 256;
  l.cl_first = off;
  off += align256(sizeof(int32_t) * static_cast<size_t>(G));
  l.pre = off;
  off += align256(sizeof(int32_t) * (static_cast<size_t>(x.U) + 1 + x.n_rb));
  l.sync = off;
  off += align256(sizeof(int32_t) * 8 * static_cast<size_t>(G));
  l.lse_part = off;
  off += align256(sizeof(float) * 2 * 2 * static_cast<size_t>(G) * kRowsPerBlock);
  l.o_part = off;
  off += sizeof(uint16_t) * 2 * static_cast<size_t>(G) * kRowsPerBlock * kDv;
  l.total = align256(off);
  return l;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct DeviceInfo {
  bool ready = false;
  int sms = 0;
  int clusters_bf16 = 0, clusters_fp8 = 0;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

mla_status device_info(DeviceInfo* info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return MLA_ERR_LAUNCH;  // built for sm_103a only
    di.sms = prop.multiProcessorCount;
    if (decode_max_active_clusters(false, &di.clusters_bf16) != cudaSuccess) return MLA_ERR_LAUNCH;
    if (decode_max_active_clusters(true, &di.clusters_fp8) != cudaSuccess) return MLA_ERR_LAUNCH;
    di.ready = true;
  }
  *info = di;
  return MLA_OK;
}

int clusters_for(const mla_desc* d, const Dims& x, const DeviceInfo& di) {
  int G = x.fp8 ? di.clusters_fp8 : di.clusters_bf16;
  G = G < di.sms / 2 ? G : di.sms / 2;
  if (d->max_clusters > 0 && d->max_clusters < G) G = d->max_clusters;
  return G < 1 ? 1 : G;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return tensor_map_encoder(); }

// The bf16 [num_pages, 64, 576] cache as a 4-D tensor (64 channels, 64
// tokens, 9 channel chunks, pages) whose chunk stride is 128 bytes: one box of
// 64 x 64 x `chunks` x 1 brings channel blocks 0..chunks-1 of a page in a
// single copy, laid out in shared memory as consecutive 64-token x 64-channel
// blocks with the 128-byte swizzle the MMA descriptors expect.
mla_status make_kv_map4(const void* kv, int num_pages, int chunks, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(kPage), 9, static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {kDqk * 2, 128, kDqk * 2 * kPage};
  cuuint32_t box[4] = {64, 64, static_cast<cuuint32_t>(chunks), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(kv), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// The bf16 cache as a 5-D tensor (64 channels, 8 tokens, 9 channel chunks, 8
// token groups, pages) for the scorer: one box (64, 8, 9, 8, 1) is a whole
// page, landing as token-group-major 1 KB atoms (group g, chunk c at
// (9g + c) KB, 128-byte swizzled), so the 8-row groups of a page are 9 KB
// apart and a page in the next 72 KB stage continues the same stride: two
// adjacent stages are one 128-token MMA operand.
mla_status make_kv_map5(const void* kv, int num_pages, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[5] = {64, 8, 9, 8, static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[4] = {kDqk * 2, 128, 8 * kDqk * 2, kDqk * 2 * kPage};
  cuuint32_t box[5] = {64, 8, 9, 8, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(kv), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// fp8 cache as a 4-D byte tensor (64 bytes, 64 tokens, `nchunks` chunks of
// 64 channels, pages) starting at `base`, with `token_bytes` per token:
// variant A [P, 64, 576] e4m3 (9 chunks); variant B [P, 64, 656] records
// (8 latent chunks at the record start; the RoPE, 2 chunks of bf16 at byte
// 528, as its own map).  Box (64, 64, `chunks`, 1) brings `chunks`
// consecutive chunks of a page as 64-token x 64-byte slots, 64-byte swizzled
// (so that both the dequant reads and its swizzled 16-byte fp16 writes are
// free of bank conflicts).
mla_status make_kv_map_fp8(const void* base, int num_pages, int token_bytes, int nchunks, int chunks,
                           CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(kPage), static_cast<cuuint64_t>(nchunks),
                        static_cast<cuuint64_t>(num_pages)};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(token_bytes), 64, static_cast<cuuint64_t>(token_bytes) * kPage};
  cuuint32_t box[4] = {64, 64, static_cast<cuuint32_t>(chunks), 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// q [B, R, 576] bf16 as a 4-D tensor (64 channels, 9 chunks, R rows, B): one
// box (64, 9, 64, 1) is half a 128-row block (72 KB), 128-byte swizzled; rows
// past R read as zeros.
mla_status make_q_map(const void* q, int B, int R, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[4] = {64, 9, static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {128, kDqk * 2, static_cast<cuuint64_t>(R) * kDqk * 2};
  cuuint32_t box[4] = {64, 9, kRowsPerBlock / 2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// out [B, R, 512] bf16 as a 3-D tensor: one box (64, 32, 1) is 32 rows x 64
// channels, 128-byte swizzled; rows past R are not written.
mla_status make_out_map(void* out, int B, int R, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDv), static_cast<cuuint64_t>(R), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {kDv * 2, static_cast<cuuint64_t>(R) * kDv * 2};
  cuuint32_t box[3] = {64, 32, 1};
  cuuint32_t es[3] = {1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, out, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

// out as a 4-D tensor (64 channels, R rows, 8 channel chunks, B): one box
// (64, 32, 4, 1) is 32 rows x 256 channels, stored from shared memory as 4
// chunk-major blocks of 32 x 128-byte swizzled rows.
mla_status make_out_map4(void* out, int B, int R, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return MLA_ERR_CUDA;
  cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(R), 8, static_cast<cuuint64_t>(B)};
  cuuint64_t strides[3] = {kDv * 2, 128, static_cast<cuuint64_t>(R) * kDv * 2};
  cuuint32_t box[4] = {64, 32, 4, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

struct Prepared {
  Dims x;
  DeviceInfo di;
  int G;
  mla_workspace_layout lay;
  uint8_t* ws;
};

mla_status prepare(const mla_desc* d, void* workspace, size_t workspace_bytes, Prepared* p) {
  mla_status st = check_desc(d, &p->x);
  if (st != MLA_OK) return st;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  st = device_info(&p->di);
  if (st != MLA_OK) return st;
  p->G = clusters_for(d, p->x, p->di);
  p->lay = layout_for(p->x, p->G);
  if (workspace_bytes < p->lay.total) return MLA_ERR_WORKSPACE;
  p->ws = static_cast<uint8_t*>(workspace);
  return MLA_OK;
}

mla_status check_tensors(const Dims& x, const void* q, const void* kv, const float* kv_scales, const int32_t* bt,
                         const int32_t* seqlens, const void* out, const float* lse) {
  if (!q || !kv || !bt || !seqlens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(bt, 4) ||
      !aligned(seqlens, 4))
    return MLA_ERR_INVALID_ARG;
  if (x.rope_bf16) {
    if (kv_scales) return MLA_ERR_INVALID_ARG;  // the scales are inside the token records
  } else if (x.fp8) {
    if (!kv_scales || !aligned(kv_scales, 16)) return MLA_ERR_INVALID_ARG;
  } else if (kv_scales) {
    return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

mla_status launch_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH; }

mla_status run_plan(const Prepared& p, const int32_t* seqlens, cudaStream_t stream) {
  int32_t* hdr = reinterpret_cast<int32_t*>(p.ws + p.lay.header);
  mla_plan_kernel<<<1, kPlanThreads, 0, stream>>>(seqlens, p.x.B, p.x.s_q, p.x.H, p.x.R, p.x.U, p.x.maxp, p.G,
                                                  p.x.ovh, hdr, reinterpret_cast<int32_t*>(p.ws + p.lay.cl_first),
                                                  reinterpret_cast<int32_t*>(p.ws + p.lay.pre),
                                                  reinterpret_cast<int32_t*>(p.ws + p.lay.sync));
  return launch_status(cudaGetLastError());
}

mla_status run_attention(const Prepared& p, const void* q, const void* kv, const float* kv_scales,
                         const int32_t* bt, const int32_t* seqlens, float scale, void* out, float* lse,
                         cudaStream_t stream) {
  // page maps of the scorer and the accumulator: bf16, the whole page
  // token-group-major (scorer) and 8 chunk-major 64-channel blocks
  // (accumulator); fp8, every raw e4m3 chunk of the row for the scorer
  // (variant B: the 8 latent chunks, plus the two bf16 RoPE chunks by their
  // own map) and the 8 latent chunks for the accumulator
  CUtensorMap map_s, map_a, map_r;
  std::memset(&map_r, 0, sizeof(map_r));
  {
    mla_status st;
    if (p.x.fp8) {
      const int tb = p.x.rope_bf16 ? kFp8bRecord : kDqk;
      const int nch = p.x.rope_bf16 ? 8 : 9;
      st = make_kv_map_fp8(kv, p.x.P, tb, nch, nch, &map_s);
      if (st == MLA_OK) st = make_kv_map_fp8(kv, p.x.P, tb, nch, 8, &map_a);
      if (st == MLA_OK) {
        if (p.x.rope_bf16)  // the RoPE bf16 bytes [528, 656) of each record: 2 chunks
          st = make_kv_map_fp8(static_cast<const uint8_t*>(kv) + kFp8bRopeOffset, p.x.P, tb, 2, 2, &map_r);
        else                // not read by variant A (its RoPE chunk is chunk 8 of map_s); a valid map all the same
          st = make_kv_map_fp8(kv, p.x.P, tb, nch, 1, &map_r);
      }
    } else {
      st = make_kv_map5(kv, p.x.P, &map_s);
      if (st == MLA_OK) st = make_kv_map4(kv, p.x.P, 8, &map_a);
    }
    if (st != MLA_OK) return st;
  }
  CUtensorMap qmap, omap, omap4;
  mla_status st = make_q_map(q, p.x.B, p.x.R, &qmap);
  if (st == MLA_OK) st = make_out_map(out, p.x.B, p.x.R, &omap);
  if (st == MLA_OK) st = make_out_map4(out, p.x.B, p.x.R, &omap4);
  if (st != MLA_OK) return st;
  DecodeArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.kv = kv;
  a.kv_scales = kv_scales;
  a.rope_bf16 = p.x.rope_bf16 ? 1 : 0;
  a.block_table = bt;
  a.seqlens = seqlens;
  a.hdr = reinterpret_cast<const int32_t*>(p.ws + p.lay.header);
  a.cl_first = reinterpret_cast<const int32_t*>(p.ws + p.lay.cl_first);
  a.pre = reinterpret_cast<const int32_t*>(p.ws + p.lay.pre);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.o_part = p.ws + p.lay.o_part;
  a.lse_part = reinterpret_cast<float*>(p.ws + p.lay.lse_part);
  a.unit_cnt = reinterpret_cast<int32_t*>(p.ws + p.lay.sync);
  a.slot_ready = a.unit_cnt + p.G;
  a.err = reinterpret_cast<int32_t*>(p.ws + p.lay.header);
  a.B = p.x.B;
  a.s_q = p.x.s_q;
  a.H = p.x.H;
  a.R = p.x.R;
  a.n_rb = p.x.n_rb;
  a.U = p.x.U;
  a.num_pages = p.x.P;
  a.max_pages = p.x.maxp;
  a.overhead = p.x.ovh;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_status(launch_decode(a, map_s, map_a, map_r, qmap, omap, omap4, p.G, p.x.fp8, stream));
}

mla_status run_combine(const Prepared& p, void* out, float* lse, cudaStream_t stream) {
  CombineArgs a;
  a.hdr = reinterpret_cast<const int32_t*>(p.ws + p.lay.header);
  a.cl_first = reinterpret_cast<const int32_t*>(p.ws + p.lay.cl_first);
  a.pre = reinterpret_cast<const int32_t*>(p.ws + p.lay.pre);
  a.o_part = p.ws + p.lay.o_part;
  a.lse_part = reinterpret_cast<const float*>(p.ws + p.lay.lse_part);
  a.sync = reinterpret_cast<const int32_t*>(p.ws + p.lay.sync);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.B = p.x.B;
  a.R = p.x.R;
  a.U = p.x.U;
  a.clusters = p.G;
  a.overhead = p.x.ovh;
  // programmatic dependent of the attention kernel (it waits on the device)
  cudaLaunchConfig_t cfg = {};
  // one CTA per 8-channel chunk and job column, each column looping over its
  // jobs: a grid sized for the worst-case job count cost several microseconds
  // per step to schedule even when there is no job
  cfg.gridDim = dim3(kPartChunks, kCombineJobColumns, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_status(cudaLaunchKernelEx(&cfg, mla_combine_kernel, a));
}

}  // namespace
}  // namespace mla_gb300

using namespace mla_gb300;

extern "C" {

size_t mla_workspace_size(const mla_desc* desc, int num_sms) {
  Dims x;
  if (check_desc(desc, &x) != MLA_OK) return 0;
  if (num_sms <= 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  }
  int G = num_sms / 2;
  if (desc->max_clusters > 0 && desc->max_clusters < G) G = desc->max_clusters;
  if (G < 1) G = 1;
  return layout_for(x, G).total;
}

int mla_num_clusters(const mla_desc* desc) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  DeviceInfo di;
  st = device_info(&di);
  if (st != MLA_OK) return st;
  return clusters_for(desc, x, di);
}

mla_status mla_get_workspace_layout(const mla_desc* desc, int num_clusters, mla_workspace_layout* layout) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (num_clusters < 1 || !layout) return MLA_ERR_INVALID_ARG;
  *layout = layout_for(x, num_clusters);
  return MLA_OK;
}

mla_status mla_plan(const mla_desc* desc, const int32_t* seqlens, void* workspace, size_t workspace_bytes,
                    void* stream) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (!seqlens || !aligned(seqlens, 4)) return MLA_ERR_INVALID_ARG;
  Prepared p;
  st = prepare(desc, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  return run_plan(p, seqlens, static_cast<cudaStream_t>(stream));
}

mla_status mla_decode_attention(const mla_desc* desc, const void* q, const void* kv_pages, const float* kv_scales,
                                const int32_t* block_table, const int32_t* seqlens, int32_t s_q,
                                float softmax_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (s_q != desc->s_q || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  st = check_tensors(x, q, kv_pages, kv_scales, block_table, seqlens, out, lse);
  if (st != MLA_OK) return st;
  Prepared p;
  st = prepare(desc, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  return run_attention(p, q, kv_pages, kv_scales, block_table, seqlens, softmax_scale, out, lse,
                       static_cast<cudaStream_t>(stream));
}

mla_status mla_combine_workspace(const mla_desc* desc, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (!out || !lse || !aligned(out, 16) || !aligned(lse, 4)) return MLA_ERR_INVALID_ARG;
  Prepared p;
  st = prepare(desc, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  return run_combine(p, out, lse, static_cast<cudaStream_t>(stream));
}

mla_status mla_combine(const mla_desc* desc, const float* o_part, const float* lse_part, const int32_t* split_indptr,
                       int32_t num_partials, void* out, float* lse, void* stream) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (num_partials < 0 || !split_indptr || !out || !lse || !aligned(split_indptr, 4) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  if (num_partials > 0 && (!o_part || !lse_part || !aligned(o_part, 16) || !aligned(lse_part, 4)))
    return MLA_ERR_INVALID_ARG;
  const dim3 grid(static_cast<unsigned>(x.B), static_cast<unsigned>((x.R + kCpWarps - 1) / kCpWarps), 1);
  mla_combine_partials_kernel<<<grid, 32 * kCpWarps, 0, static_cast<cudaStream_t>(stream)>>>(
      o_part, lse_part, split_indptr, num_partials, x.R, static_cast<uint16_t*>(out), lse);
  return launch_status(cudaGetLastError());
}

mla_status mla_decode(const mla_desc* desc, const void* q, const void* kv_pages, const float* kv_scales,
                      const int32_t* block_table, const int32_t* seqlens, int32_t s_q, float softmax_scale,
                      void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream) {
  Dims x;
  mla_status st = check_desc(desc, &x);
  if (st != MLA_OK) return st;
  if (s_q != desc->s_q || !std::isfinite(softmax_scale) || !(softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  st = check_tensors(x, q, kv_pages, kv_scales, block_table, seqlens, out, lse);
  if (st != MLA_OK) return st;
  Prepared p;
  st = prepare(desc, workspace, workspace_bytes, &p);
  if (st != MLA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = run_plan(p, seqlens, s);
  if (st != MLA_OK) return st;
  st = run_attention(p, q, kv_pages, kv_scales, block_table, seqlens, softmax_scale, out, lse, s);
  if (st != MLA_OK) return st;
  return run_combine(p, out, lse, s);
}

mla_status mla_get_device_error(const void* workspace, void* stream) {
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  int32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (word & kErrTimeout) return MLA_ERR_DEVICE_TIMEOUT;
  if (word & kErrBounds) return MLA_ERR_DEVICE_BOUNDS;
  if (word & kErrRange) return MLA_ERR_DEVICE_RANGE;
  return MLA_OK;
}

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case MLA_ERR_LAUNCH: return "kernel launch failed";
    case MLA_ERR_DEVICE_BOUNDS: return "device saw a page id or seqlen out of bounds";
    case MLA_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case MLA_ERR_CUDA: return "CUDA runtime call failed";
    case MLA_ERR_DEVICE_RANGE: return "fp8 cache scale outside the fp16 compute range";
    default: return "unknown status";
  }
}

}  // extern "C"
