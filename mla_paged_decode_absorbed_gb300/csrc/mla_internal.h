// Declarations shared by the library's translation units (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mla_gb300 {

constexpr int kPage = 64;            // tokens per KV page
constexpr int kDqk = 576;            // channels per query head / KV token (512 latent + 64 RoPE)
constexpr int kDv = 512;             // output channels (latent part of a KV row)
constexpr int kRowsPerBlock = 128;   // query rows (token-major (i, h)) per work unit = MMA M
constexpr int kGroups = 5;           // fp8 scale groups per token
constexpr int kDefaultOverhead = 2;  // planner cost per work unit, in pages

// Device error bits in workspace word 0.
enum : int32_t { kErrBounds = 1, kErrTimeout = 2, kErrRange = 4 };

// Workspace header words (int32).
enum : int { kHdrErr = 0, kHdrW = 1, kHdrTotal = 2, kHdrUnits = 3, kHdrClusters = 4, kHdrOvh = 5 };

struct DecodeArgs {
  const uint16_t* q;          // bf16 [B, s_q, H, 576]
  const void* kv;             // the cache itself (the fp8 variant reads it with plain loads)
  const float* kv_scales;     // fp32 [P, 64, 5] (fp8 cache) or nullptr
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seqlens;     // [B]
  const int32_t* hdr;         // workspace header
  const int32_t* cl_first;    // [clusters]
  const int32_t* pre;         // [units + 1]
  uint16_t* out;              // bf16 [B, s_q, H, 512]
  float* lse;                 // [B, s_q, H]
  float* o_part;              // [2 * clusters, 128, 512]
  float* lse_part;            // [2 * clusters, 128]
  int32_t* err;               // workspace word 0
  int B, s_q, H, R, n_rb, U, num_pages, max_pages, overhead;
  float scale_log2;           // softmax_scale * log2(e)
};

struct CombineArgs {
  const int32_t* hdr;
  const int32_t* cl_first;
  const int32_t* pre;
  const float* o_part;
  const float* lse_part;
  uint16_t* out;
  float* lse;
  int B, R, U, clusters, overhead;
};

// mla_decode_kernel.cu
int decode_smem_bytes(bool fp8);
cudaError_t decode_max_active_clusters(bool fp8, int* clusters);
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kv_map, int clusters, bool fp8,
                          cudaStream_t stream);

}  // namespace mla_gb300
