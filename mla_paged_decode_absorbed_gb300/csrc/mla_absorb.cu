// Matrix absorption around the attention step (best-practice digest §2.4.3,
// the `--mla_use_matrix_absorption` switch; the algebra is standard MLA):
//   mla_absorb_q:    q[t, h] = [W_UK[h] q_nope[t, h] ; q_rope[t, h]]   (128 -> 512 channels)
//   mla_project_out: o[t, h] = W_UV[h]^T out[t, h]                       (512 -> 128 channels)
// Both are per-head GEMMs with a 128-row output tile: one CTA computes
// D[128 x tt] = A[128 x K] * B[tt x K]^T with tcgen05 (fp32 accumulator in
// TMEM), where B is tt tokens of the activations (K-major) and A is a 128-row
// slice of the head's weights (absorb: W_UK rows, K-major; project: W_UV read
// MN-major).  TMA brings each operand in one or two large copies (the TMA
// unit spends a fixed time per copy, so a few 32-64 KB copies are far faster
// than many 8 KB ones): the 64-channel chunks of an operand land as
// consecutive 128-byte-swizzled blocks through a tensor map whose chunk index
// is a dimension of its own.  The epilogue stages D transposed through shared
// memory so that every (token, head) row of 128 outputs leaves as 256
// contiguous bytes.
//
// Roofline: the weights (H x 512 x 128 bf16 = 16.8 MB at H = 128) are read
// once; with few tokens the step is HBM-bound on them, with many it is
// tensor-bound.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>

#include "mla.h"
#include "mla_internal.h"
#include "sm103_ptx.cuh"

namespace mla_gb300 {
namespace {

using namespace mla_sm103;

constexpr int kGemmThreads = 128;           // thread 0 loads, warp 1 issues MMAs, all four run the epilogue
constexpr int kChunkA = 128 * 64 * 2;       // one 64-channel chunk of a 128-row A tile (16 KB)
constexpr int kNopeDim = 128, kRopeDim = 64, kLat = 512;

// Shared memory: A (absorb: 2 chunks x 128 rows = 32 KB; project: 2 halves of
// 64 output channels x 512 k rows = 128 KB), then B (tt tokens x K).
// project runs 64-token tiles (B = 64 KB) so that both fit.
__host__ __device__ constexpr int gemm_a_bytes(bool project) { return project ? 2 * kLat * 128 : 2 * kChunkA; }
__host__ __device__ constexpr int gemm_b_bytes(bool project, int tt) { return tt * (project ? kLat : kNopeDim) * 2; }

struct GemmArgs {
  const uint16_t* rope;  // absorb: q_rope [T, H, 64] (copied into q[..., 512:576]); project: unused
  uint16_t* y;           // output: absorb q [T, H, 576]; project o [T, H, 128]
  int32_t* err;          // error word of a workspace, or null
  int T, H, tt;          // tokens, heads, tokens per CTA (the MMA's N)
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, int32_t* err) {
  if (mbar_wait(bar, parity, nullptr)) return true;
  if (err) atomicOr(err, kErrTimeout);
  return false;
}

// CTA (x, h, z): head h, tokens [z*tt, z*tt + tt), output channels
// [128x, 128x + 128) (absorb; x = 0 for project).
template <bool kProject>
__global__ void __launch_bounds__(kGemmThreads, 1)
    mla_absorb_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                           const GemmArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tt = a.tt;
  constexpr int kA = gemm_a_bytes(kProject);
  const int b_bytes = gemm_b_bytes(kProject, tt);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kA + b_bytes);  // [2]: the operand copies landed
  uint64_t* done = full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int xt = blockIdx.x, h = blockIdx.y, t0 = blockIdx.z * tt;
  if (tid == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    mbar_init(smem_u32(done), 1);
    fence_mbarrier_init_cluster();
    // ------------------------------------------------------------ loads
    // issued at once (the barriers are this thread's own), so their latency
    // overlaps the TMEM allocation and the block barrier below
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_x);
    uint8_t* const sa0 = smem;
    uint8_t* const sb0 = smem + kA;
    const uint32_t f0 = smem_u32(&full[0]), f1 = smem_u32(&full[1]);
    if (kProject) {
      // B: every 64-channel chunk of the tile's tokens (chunk-major), and the
      // first 256 k rows of W_UV[h] (both 64-wide output-channel halves);
      // then the other 256 rows on their own barrier
      mbar_arrive_expect_tx(f0, static_cast<uint32_t>(b_bytes + kA / 2));
      tma_load_4d(smem_u32(sb0), &map_x, 0, t0, 0, h, f0);
      tma_load_3d(smem_u32(sa0), &map_w, 0, h * kLat, 0, f0);
      mbar_arrive_expect_tx(f1, static_cast<uint32_t>(kA / 2));
      tma_load_3d(smem_u32(sa0 + kA / 2), &map_w, 0, h * kLat + 256, 0, f1);
    } else {
      // W_UK[h] rows n = 128x.. (both 64-channel chunks) and the tokens' q_nope
      mbar_arrive_expect_tx(f0, static_cast<uint32_t>(kA + b_bytes));
      tma_load_3d(smem_u32(sa0), &map_w, 0, h * kLat + 128 * xt, 0, f0);
      tma_load_4d(smem_u32(sb0), &map_x, 0, t0, 0, h, f0);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(tt));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;
  uint8_t* const sa = smem;
  uint8_t* const sb = smem + kA;

  // absorb: the RoPE part of q passes through, q[t, h, 512:576] = q_rope[t, h].
  // The four CTAs of a token tile (x = 0..3) copy a quarter of its tokens each,
  // and the loads are issued now, so that their latency overlaps the operand
  // loads instead of lengthening one CTA's epilogue (tt / 4 tokens x 8
  // 16-byte pieces = 2 tt pieces per CTA, at most four per thread)
  uint4 rope_v[4];
  if (!kProject) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + i * kGemmThreads, t = t0 + xt * (tt / 4) + (idx >> 3);
      rope_v[i] = make_uint4(0, 0, 0, 0);
      if (idx < 2 * tt && t < a.T)
        rope_v[i] = __ldg(reinterpret_cast<const uint4*>(a.rope + (static_cast<size_t>(t) * a.H + h) * kRopeDim) + (idx & 7));
    }
  }

  bool ok = true;
  if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = idesc_bf16_f32(128, tt, kProject, false);
    // B: K-major token rows, chunk c at c * tt * 128 bytes
    const uint64_t bd = smem_desc_sw128(smem_u32(sb), 16, 1024);
    if (kProject) {
      // A: MN-major, two 64-channel halves 256 rows x 128 B = 32 KB apart (the
      // descriptor's leading offset) in each 64 KB block of 256 k rows
      for (int half = 0; half < 2 && ok; ++half) {
        if (!wait_bounded(smem_u32(&full[half]), 0u, a.err)) { ok = false; break; }
        tc_fence_after();
        const uint64_t ad = smem_desc_sw128(smem_u32(sa + half * (kA / 2)), kA / 4, 1024);
#pragma unroll 4
        for (int k = 0; k < 16; ++k) {
          const int kg = 16 * half + k;  // K step of 16 rows: chunk kg / 4 of B
          mma_ss(tbase, ad + static_cast<uint64_t>((k * 2048) >> 4),
                 bd + static_cast<uint64_t>(((kg >> 2) * tt * 128 + (kg & 3) * 32) >> 4), idesc, kg > 0 ? 1u : 0u);
        }
      }
    } else {
      if (wait_bounded(smem_u32(&full[0]), 0u, a.err)) {
        tc_fence_after();
        // A: K-major rows of 128 bytes, chunk c at c * 16 KB
        const uint64_t ad = smem_desc_sw128(smem_u32(sa), 16, 1024);
#pragma unroll
        for (int k = 0; k < 8; ++k)
          mma_ss(tbase, ad + static_cast<uint64_t>(((k >> 2) * kChunkA + (k & 3) * 32) >> 4),
                 bd + static_cast<uint64_t>(((k >> 2) * tt * 128 + (k & 3) * 32) >> 4), idesc, k > 0 ? 1u : 0u);
      } else {
        ok = false;
      }
    }
    if (ok) mma_commit(smem_u32(done));
  }
  __syncwarp();

  // -------------------------------------------------------------- epilogue
  // Thread = output channel (TMEM lane); D's columns are tokens.  Stage
  // bf16 [tt tokens][128 channels] over the (consumed) operand stages.
  const bool have = wait_bounded(smem_u32(done), 0u, a.err);
  tc_fence_after();
  uint16_t* stg = reinterpret_cast<uint16_t*>(smem);
  if (have) {
    for (int col = 0; col < tt; col += 32) {
      uint32_t r[32];
      tmem_ld32(tbase + (static_cast<uint32_t>(32 * warp) << 16) + static_cast<uint32_t>(col), r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const __nv_bfloat16 v = __float2bfloat16_rn(__uint_as_float(r[i]));
        stg[(col + i) * 128 + tid] = *reinterpret_cast<const uint16_t*>(&v);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (have) {
    const int y_row = kProject ? a.H * kNopeDim : a.H * kDqk;  // elements between tokens
    const int y_head = kProject ? kNopeDim : kDqk;
    const int y_col = kProject ? 0 : 128 * xt;
    for (int idx = tid; idx < tt * 16; idx += kGemmThreads) {
      const int row = idx >> 4, q16 = idx & 15, t = t0 + row;
      if (t < a.T) {
        uint16_t* dst = a.y + static_cast<size_t>(t) * y_row + static_cast<size_t>(h) * y_head + y_col + q16 * 8;
        *reinterpret_cast<uint4*>(dst) = reinterpret_cast<const uint4*>(stg + row * 128)[q16];
      }
    }
    if (!kProject) {  // this CTA's quarter of the tile's RoPE pieces, loaded at the start
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int idx = tid + i * kGemmThreads, t = t0 + xt * (tt / 4) + (idx >> 3);
        if (idx < 2 * tt && t < a.T)
          reinterpret_cast<uint4*>(a.y + (static_cast<size_t>(t) * a.H + h) * kDqk + kLat)[idx & 7] = rope_v[i];
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, static_cast<uint32_t>(tt));
  }
}

int token_tile(bool project, int T) { return project || T <= 64 ? 64 : (T <= 128 ? 128 : 256); }

// operands, alignment slack, barriers (3 mbarriers and the TMEM address)
int gemm_smem(bool project, int tt) { return gemm_a_bytes(project) + gemm_b_bytes(project, tt) + 1024 + 256; }

// bf16 tensor with up to 4 dims (innermost first) as a TMA map with a
// 64-element x box[1] x ... box, 128-byte swizzled.  The strides need not
// grow with the dimension: a dimension of 64-channel chunks (stride 128 B)
// after a row dimension makes one box land as consecutive swizzled blocks.
mla_status make_map(const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                    const cuuint32_t* box, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return MLA_ERR_CUDA;
  cuuint32_t es[4] = {1, 1, 1, 1};
  std::memset(map, 0, sizeof(*map));
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                   dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MLA_OK : MLA_ERR_INVALID_ARG;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

mla_status check_sizes(int32_t tokens, int32_t heads) {
  if (tokens < 1 || heads < 1 || heads > 1024) return MLA_ERR_INVALID_ARG;
  // row indices of the weight maps and token*head offsets stay in range
  if (static_cast<int64_t>(tokens) * heads * kDqk > (int64_t(1) << 40)) return MLA_ERR_INVALID_ARG;
  return MLA_OK;
}

template <bool kProject>
mla_status launch_gemm(const CUtensorMap& mw, const CUtensorMap& mx, const GemmArgs& a, cudaStream_t stream) {
  const int smem = gemm_smem(kProject, a.tt);
  if (cudaFuncSetAttribute(mla_absorb_gemm_kernel<kProject>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return MLA_ERR_CUDA;
  const dim3 grid(kProject ? 1 : kLat / 128, static_cast<unsigned>(a.H),
                  static_cast<unsigned>((a.T + a.tt - 1) / a.tt));
  mla_absorb_gemm_kernel<kProject><<<grid, kGemmThreads, smem, stream>>>(mw, mx, a);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_LAUNCH;
}

int32_t* error_word(void* workspace) { return workspace ? static_cast<int32_t*>(workspace) : nullptr; }

}  // namespace
}  // namespace mla_gb300

using namespace mla_gb300;

extern "C" mla_status mla_absorb_q(const void* q_nope, const void* q_rope, const void* w_uk, int32_t tokens,
                                   int32_t num_heads, void* q, void* workspace, void* stream) {
  mla_status st = check_sizes(tokens, num_heads);
  if (st != MLA_OK) return st;
  if (!q_nope || !q_rope || !w_uk || !q || !aligned16(q_nope) || !aligned16(q_rope) || !aligned16(w_uk) ||
      !aligned16(q) || (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return MLA_ERR_INVALID_ARG;
  const int tt = token_tile(false, tokens);
  const cuuint64_t H = static_cast<cuuint64_t>(num_heads);
  CUtensorMap mw, mx;
  {  // W_UK [H*512 rows n, 128 k] as (64 k, rows, 2 chunks): box 64 x 128 rows x 2 = 32 KB
    const cuuint64_t dims[3] = {64, H * kLat, 2};
    const cuuint64_t strides[2] = {kNopeDim * 2, 128};
    const cuuint32_t box[3] = {64, 128, 2};
    st = make_map(w_uk, 3, dims, strides, box, &mw);
  }
  if (st == MLA_OK) {  // q_nope [T, H, 128] as (64 ch, T, 2 chunks, H): box 64 x tt x 2 x 1
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(tokens), 2, H};
    const cuuint64_t strides[3] = {H * kNopeDim * 2, 128, kNopeDim * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(tt), 2, 1};
    st = make_map(q_nope, 4, dims, strides, box, &mx);
  }
  if (st != MLA_OK) return st;
  GemmArgs a;
  a.rope = static_cast<const uint16_t*>(q_rope);
  a.y = static_cast<uint16_t*>(q);
  a.err = error_word(workspace);
  a.T = tokens;
  a.H = num_heads;
  a.tt = tt;
  return launch_gemm<false>(mw, mx, a, static_cast<cudaStream_t>(stream));
}

extern "C" mla_status mla_project_out(const void* out_latent, const void* w_uv, int32_t tokens, int32_t num_heads,
                                      void* o, void* workspace, void* stream) {
  mla_status st = check_sizes(tokens, num_heads);
  if (st != MLA_OK) return st;
  if (!out_latent || !w_uv || !o || !aligned16(out_latent) || !aligned16(w_uv) || !aligned16(o) ||
      (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)))
    return MLA_ERR_INVALID_ARG;
  const int tt = token_tile(true, tokens);
  const cuuint64_t H = static_cast<cuuint64_t>(num_heads);
  CUtensorMap mw, mx;
  {  // W_UV [H*512 rows k, 128 j] as (64 j, rows, 2 halves): box 64 x 256 rows x 2 = 64 KB
    const cuuint64_t dims[3] = {64, H * kLat, 2};
    const cuuint64_t strides[2] = {kNopeDim * 2, 128};
    const cuuint32_t box[3] = {64, 256, 2};
    st = make_map(w_uv, 3, dims, strides, box, &mw);
  }
  if (st == MLA_OK) {  // out [T, H, 512] as (64 ch, T, 8 chunks, H): box 64 x 64 tokens x 8 x 1 = 64 KB
    const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(tokens), 8, H};
    const cuuint64_t strides[3] = {H * kLat * 2, 128, kLat * 2};
    const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(tt), 8, 1};
    st = make_map(out_latent, 4, dims, strides, box, &mx);
  }
  if (st != MLA_OK) return st;
  GemmArgs a;
  a.rope = nullptr;
  a.y = static_cast<uint16_t*>(o);
  a.err = error_word(workspace);
  a.T = tokens;
  a.H = num_heads;
  a.tt = tt;
  return launch_gemm<true>(mw, mx, a, static_cast<cudaStream_t>(stream));
}
