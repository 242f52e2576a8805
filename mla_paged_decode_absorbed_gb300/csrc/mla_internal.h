// Declarations shared by the library's translation units (not part of the C ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cstdint>

namespace mla_gb300 {

constexpr int kPage = 64;            // tokens per KV page
constexpr int kDqk = 576;            // channels per query head / KV token (512 latent + 64 RoPE)
constexpr int kDv = 512;             // output channels (latent part of a KV row)
constexpr int kRowsPerBlock = 128;   // query rows (token-major (i, h)) per work unit = MMA M
constexpr int kGroups = 5;           // fp8 scale groups per token
constexpr int kFp8bRecord = 656;     // fp8 variant B bytes per token: e4m3 latent, 4 fp32 scales, RoPE bf16
constexpr int kFp8bScaleOffset = 512, kFp8bRopeOffset = 528;
constexpr int kDefaultOverhead = 4;  // planner cost per work unit, in pages
// A split unit with at most this many pieces is merged inside the attention
// kernel by the piece that finishes last; units with more pieces are merged by
// the combine kernel.
constexpr int kFuseMax = 3;
// Partial slots hold fp16 O / l in 8-channel chunks: [slot][kPartChunks][128 rows][8].
constexpr int kPartChunks = 512 / 8;

// Device error bits in workspace word 0.
enum : int32_t { kErrBounds = 1, kErrTimeout = 2, kErrRange = 4 };

// Workspace header words (int32).
// kHdrCombine: number of units with more than kFuseMax pieces (combine jobs).
// kHdrStall: a test writes nonzero here after the plan to make the next
// attention kernel's scorers wait on a barrier nothing signals (the plan clears it).
enum : int {
  kHdrErr = 0, kHdrW = 1, kHdrTotal = 2, kHdrUnits = 3, kHdrClusters = 4, kHdrOvh = 5, kHdrCombine = 6, kHdrStall = 7
};

struct DecodeArgs {
  const uint16_t* q;          // bf16 [B, s_q, H, 576]
  const void* kv;             // the cache (fp8 variant B: its records' scales are read with plain loads)
  const float* kv_scales;     // fp32 [P, 64, 5] (fp8 variant A) or nullptr
  const int32_t* block_table; // [B, max_pages]
  const int32_t* seqlens;     // [B]
  const int32_t* hdr;         // workspace header
  const int32_t* cl_first;    // [clusters]
  const int32_t* pre;         // [units + 1]
  uint16_t* out;              // bf16 [B, s_q, H, 512]
  float* lse;                 // [B, s_q, H]
  void* o_part;               // fp16 [2 * clusters][64 chunks of 8 channels][128 rows][8]
  float* lse_part;            // [2 * clusters, 128, 2]: (lse, power-of-two scale of the stored values)
  int32_t* unit_cnt;          // [clusters]: pieces finished of the split unit whose pages start in cluster c
  int32_t* slot_ready;        // [2 * clusters]: partial slot written (1) / consumed (0)
  int32_t* err;               // workspace word 0
  int B, s_q, H, R, n_rb, U, num_pages, max_pages, overhead;
  float scale_log2;           // softmax_scale * log2(e)
  int rope_bf16;              // fp8 variant B: 656-byte token records, scales inside, RoPE in bf16
};

struct CombineArgs {
  const int32_t* hdr;
  const int32_t* cl_first;
  const int32_t* pre;
  const void* o_part;
  const int32_t* sync;        // merge counters, slot flags, then combine jobs (int4 at [4 * clusters])
  const float* lse_part;
  uint16_t* out;
  float* lse;
  int B, R, U, clusters, overhead;
};

// mla_abi.cu: the driver's tensor-map encoder (null if it cannot be found).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// mla_decode_kernel.cu
int decode_smem_bytes(bool fp8);
cudaError_t decode_max_active_clusters(bool fp8, int* clusters);
// kv_map_s / kv_map_a: the page maps of the scorer and the accumulator.  bf16
// cache: the scorer's is a 5-D tensor (64 channels, 8 tokens, 9 channel
// chunks, 8 token groups, pages) whose box is a whole page as token-group-major
// 1 KB atoms; the accumulator's a 4-D tensor (64 channels, 64 tokens, 9
// channel chunks, pages) whose box brings chunks 0..7 as consecutive
// 64-token x 64-channel swizzled blocks.  fp8 cache: the e4m3 bytes as a 4-D tensor (64 bytes, 64
// tokens, 9 chunks (variant B: 8 latent chunks of a 656-byte record),
// pages), 64-byte swizzled; boxes of every chunk (scorer) or the 8 latent
// chunks (accumulator), and kv_map_r the two bf16 RoPE chunks of a variant B
// record.  kv_map_r is unused for the bf16 cache and fp8 variant A.
// q_map: q as a 4-D tensor (64 channels, 9 channel chunks, R rows, B) whose
// box (64, 9, 64, 1) is half a row block (rows past R read as zeros).
// out_map: out as a 3-D tensor (512 channels, R rows, B) whose box
// (64, 32, 1) is 32 rows x 64 channels (rows past R are not written).
// out_map4: out as a 4-D tensor (64 channels, R rows, 8 channel chunks, B)
// whose box (64, 32, 4, 1) is 32 rows x 256 channels.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kv_map_s, const CUtensorMap& kv_map_a,
                          const CUtensorMap& kv_map_r, const CUtensorMap& q_map, const CUtensorMap& out_map, const CUtensorMap& out_map4,
                          int clusters, bool fp8, cudaStream_t stream);

}  // namespace mla_gb300
