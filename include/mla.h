/*
 * mla.h -- C ABI of the GB300 (sm_103a) MLA paged-decode library, absorbed form.
 *
 * The operation (PaddleNLP issue #10157, section "Multi-head Latent Attention
 * (MLA) 算子 / 总体概述": Data Load -> QK GEMM -> Softmax Update + R2S -> PV
 * GEMM, with the decoder supporting num_token > 1; the verify step of
 * "MTP 高效推理实现大批次加速 / draft token 验证阶段注意力计算优化" keeps the batch
 * size and verifies every draft token in one pass; the matrix-absorption switch
 * of the PaddleNLP best-practice digest, section 2.4.3,
 * "--mla_use_matrix_absorption 1", runs the attention on the latent cache):
 *
 *   for request b, new token i < s_q, head h, with n = seqlen[b] - s_q + i + 1:
 *     s_t  = softmax_scale * <q[b,i,h,0:576], K_t[0:576]>,  t < n
 *     out[b,i,h,c] = sum_t softmax(s)_t * K_t[c],  c < 512
 *     lse[b,i,h]   = ln sum_t exp(s_t)                  (natural log)
 *   K_t is row t%64 of page block_table[b][t/64]; n <= 0 gives out 0, lse -inf.
 *
 * The split of each request's pages across SMs and the LSE merge of the pieces
 * follow the cache partitioning of the same digest, section 1.4 ("Append
 * Attention 优化", FLAGS_cascade_attention_max_partition_size).  The two
 * absorption GEMMs that put q into this form and take the output back to
 * the head dimension are mla_absorb_q() and mla_project_out().
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers must point to device memory of the
 *     current CUDA device; the caller owns every buffer, the library allocates
 *     nothing and keeps no state besides a per-device cache of launch limits
 *     (and, for mla_decode_noalloc() only, a fixed scratch array of its own).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous on that stream and never synchronise the host, except
 *     mla_get_device_error().
 *   - Problems the host can see (bad sizes, NULL or misaligned pointers, short
 *     workspace) return a negative mla_status and launch nothing.  Problems
 *     only the device can see (a page id outside the pool, a seqlen beyond the
 *     block table, an fp8 value outside the fp16 compute range, a pipeline
 *     wait that timed out) set an error word in the
 *     workspace, the kernels finish without trapping, and
 *     mla_get_device_error() reports them.  Nothing aborts the process.
 *   - The library sees pointers only: it cannot tell that a buffer is smaller
 *     than the descriptor says, and a short buffer is read or written past its
 *     end.  Sizing every buffer as documented below is the caller's part (the
 *     Python binding checks each tensor's dtype, shape and contiguity against
 *     the descriptor before the call).
 */
#ifndef MLA_GB300_H_
#define MLA_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,    /* bad size, NULL or misaligned pointer, bad scale */
  MLA_ERR_UNSUPPORTED = -2,    /* page_size != 64, d_qk != 576, d_v != 512, unknown kv dtype */
  MLA_ERR_WORKSPACE = -3,      /* workspace NULL, misaligned or smaller than mla_workspace_size() */
  MLA_ERR_LAUNCH = -4,         /* a kernel launch failed (no sm_103a device, bad configuration) */
  MLA_ERR_DEVICE_BOUNDS = -5,  /* device saw a page id outside [0, num_pages) or seqlen outside [0, 64*max_pages] */
  MLA_ERR_DEVICE_TIMEOUT = -6, /* a pipeline wait in the decode kernel exceeded its time limit */
  MLA_ERR_CUDA = -7,           /* a CUDA runtime call failed */
  MLA_ERR_DEVICE_RANGE = -8    /* fp8 cache: a scale with 448*|scale| > 65504 (outside the fp16 compute range) */
} mla_status;

typedef enum {
  MLA_KV_BF16 = 0,     /* kv_pages: bf16 [num_pages, 64, 576]; MMAs in bf16 */
  MLA_KV_FP8_E4M3 = 1, /* kv_pages: e4m3 bytes [num_pages, 64, 576] + kv_scales fp32 [num_pages, 64, 5];
                          dequantised to fp16 in the load path and MMAs in fp16 (q is converted to
                          fp16 per row with a power-of-two scale, so it cannot overflow) */
  MLA_KV_FP8_E4M3_ROPE_BF16 = 2  /* fp8 variant B: kv_pages is [num_pages, 64, 656] bytes, one record per
                          token: e4m3 latent codes [0,512), four fp32 scales [512,528) (latent
                          channel groups of 128), the 64 RoPE channels as bf16 [528,656); kv_scales
                          must be NULL.  Computed as MLA_KV_FP8_E4M3 (fp16 MMAs) */
} mla_kv_dtype;

/* Problem description.  All fields are plain sizes; unset optional fields are 0. */
typedef struct {
  int32_t batch;              /* B >= 1 requests */
  int32_t s_q;                /* new tokens per request, 1..16 (MTP verify uses > 1) */
  int32_t num_heads;          /* H, 1..1024 */
  int32_t num_pages;          /* pages in the KV pool, >= 1 */
  int32_t max_pages_per_seq;  /* row length of block_table, >= 1 */
  int32_t page_size;          /* must be 64 tokens */
  int32_t d_qk;               /* must be 576 (512 latent + 64 RoPE) */
  int32_t d_v;                /* must be 512 (the latent part of each KV row) */
  int32_t kv_dtype;           /* mla_kv_dtype */
  int32_t max_clusters;       /* optional cap on the number of 2-CTA clusters (0 = what the device holds) */
  int32_t plan_overhead;      /* optional planner cost per (row block, request) in pages (0 = default 4) */
  int32_t reserved[5];        /* must be 0 */
} mla_desc;

/*
 * Bytes of device workspace mla_decode() needs for `desc` on a device with
 * `num_sms` SMs (num_sms <= 0: query the current device).  The workspace holds
 * the error word, the split plan and the partial outputs of split
 * requests.  Returns 0 for an invalid desc.
 */
size_t mla_workspace_size(const mla_desc* desc, int num_sms);

/*
 * Number of 2-CTA clusters the decode kernel will use on the current device for
 * `desc` (>= 1), or a negative mla_status.
 */
int mla_num_clusters(const mla_desc* desc);

/*
 * The whole hot path: mla_plan(), then mla_decode_attention(), then
 * mla_combine_workspace(), in order on `stream`.
 *
 *   q            device, bf16 [B, s_q, H, 576], contiguous, 16-byte aligned
 *   kv_pages     device, [num_pages, 64, 576] bf16 or e4m3 bytes, or [num_pages, 64, 656] fp8
 *                variant B records; contiguous, 16-byte aligned
 *   kv_scales    device, fp32 [num_pages, 64, 5] for MLA_KV_FP8_E4M3 (one scale per token per
 *                channel group [0,128) [128,256) [256,384) [384,512) [512,576)); NULL for bf16 and
 *                for fp8 variant B
 *   block_table  device, int32 [B, max_pages_per_seq]; entries at or past
 *                ceil(seqlen/64) are never read
 *   seqlens      device, int32 [B]; keys already in the cache for each request,
 *                counting its s_q new tokens
 *   s_q          must equal desc->s_q
 *   softmax_scale  finite, > 0 (1/sqrt(192) for DeepSeek-style MLA)
 *   out          device, bf16 [B, s_q, H, 512], 16-byte aligned (written)
 *   lse          device, fp32 [B, s_q, H], natural log (written)
 *   workspace    device, 256-byte aligned, >= mla_workspace_size(desc, 0) bytes
 */
mla_status mla_decode(const mla_desc* desc, const void* q, const void* kv_pages, const float* kv_scales,
                      const int32_t* block_table, const int32_t* seqlens, int32_t s_q, float softmax_scale,
                      void* out, float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Step 1 (split planner, one small kernel): reads seqlens on the device and
 * writes the plan into the workspace.  Work units are (row block of 128 query
 * rows, request) pairs ordered row-block-major; each costs ceil(n_max/64) + the
 * plan overhead, where n_max is the visible-key count of the block's last row.
 * Cluster c of G owns the cost range [c*W, (c+1)*W), W = ceil(total/G), and a
 * unit whose pages cross a range boundary is split.  Also clears the error word.
 */
mla_status mla_plan(const mla_desc* desc, const int32_t* seqlens, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Step 2 (attention over the pages, one kernel of 2-CTA clusters): needs the
 * plan of mla_plan() in the same workspace.  Writes out/lse for units that
 * were not split.  Every piece of a split unit writes a partial (normalised
 * output in fp16 with a power-of-two row scale, and its lse) into the
 * workspace; for a unit of two or three pieces the piece that finishes last
 * merges the others' partials with its own result and writes out/lse itself.
 * Units of more pieces are left to mla_combine_workspace().  The kernel leaves the
 * workspace's merge counters clear, so it may run again on the same plan;
 * after a device error, run mla_plan() again first.  The kernel is launched
 * as a programmatic dependent of the previous kernel in `stream` (its prologue
 * may overlap it; it reads nothing before that kernel has finished).
 * Arguments as for mla_decode().
 */
mla_status mla_decode_attention(const mla_desc* desc, const void* q, const void* kv_pages,
                                const float* kv_scales, const int32_t* block_table, const int32_t* seqlens,
                                int32_t s_q, float softmax_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Step 3 (LSE-weighted combine, one kernel): for every split unit of more
 * than three pieces,
 *   lse = ln sum_k exp(lse_k),  out = sum_k exp(lse_k - lse) * out_k,
 * over its pieces, written to out (bf16) and lse.  Needs the plan and the
 * partials of the two previous steps in the same workspace (the library's
 * own fp16 partial layout); returns at once on the device when the plan has
 * no such unit.  To merge partials computed elsewhere, use mla_combine().
 */
mla_status mla_combine_workspace(const mla_desc* desc, void* out, float* lse, void* workspace,
                                 size_t workspace_bytes, void* stream);

/*
 * LSE-weighted merge of split-KV partials that the caller computed (the
 * cache partitioning of the best-practice digest, section 1.4 "Append
 * Attention 优化": each request's keys are cut into chunks that are attended
 * separately and merged afterwards; it is also the merge a split of one
 * request's keys across devices needs).  For request b, row r < s_q*H, and
 * its partials k in [split_indptr[b], split_indptr[b+1]):
 *
 *   lse[b, r] = ln sum_k exp(lse_part[k, r])                     (natural log)
 *   out[b, r] = sum_k exp(lse_part[k, r] - lse[b, r]) * o_part[k, r, :]
 *
 * A partial with lse_part = -inf saw no key of that row: it contributes
 * nothing and its o_part row is not read (it may hold anything).  A row with
 * no contributing partial gets out = 0 and lse = -inf (as mla_decode() does
 * for a row with no visible key).
 *
 *   o_part        device, fp32 [num_partials, s_q*H, 512], contiguous, 16-byte aligned:
 *                 each partial's normalised output (its own softmax over its keys)
 *   lse_part      device, fp32 [num_partials, s_q*H], finite or -inf
 *   split_indptr  device, int32 [B + 1], non-decreasing; indices are clamped to
 *                 [0, num_partials], so a malformed range reads nothing outside the buffers
 *   num_partials  >= 0, the first dimension of o_part and lse_part
 *   out, lse      as mla_decode() (written)
 *
 * One kernel, one warp per (request, row), 16-byte coalesced loads and
 * stores; asynchronous on `stream`; needs no workspace.  Only desc->batch,
 * s_q and num_heads are used (the rest must still form a valid descriptor).
 */
mla_status mla_combine(const mla_desc* desc, const float* o_part, const float* lse_part, const int32_t* split_indptr,
                       int32_t num_partials, void* out, float* lse, void* stream);

/*
 * Synchronises `stream`, then reads the workspace error word written by the
 * last mla_plan()/mla_decode_attention() on this workspace: MLA_OK,
 * MLA_ERR_DEVICE_TIMEOUT, MLA_ERR_DEVICE_BOUNDS or MLA_ERR_DEVICE_RANGE (in
 * that order of precedence when several happened), or MLA_ERR_CUDA if the copy
 * itself failed.
 */
mla_status mla_get_device_error(const void* workspace, void* stream);

/*
 * mla_decode() for callers that cannot allocate device memory at call time
 * (serving loops and plugin hosts that reserve all memory up front and forbid
 * allocation afterwards; C callers that own only their inputs and outputs).
 * The pages have no counterpart: this is a packaging variant of mla_decode().
 *
 * Arguments as for mla_decode(), without the workspace.  The scratch is a
 * fixed 40 MiB array inside the library, held on every GPU that loads this
 * part of the library until the process exits; the call allocates nothing.
 * The first call on a device looks up the array's device address (make it
 * before any stream capture).  The call uses at most 76 two-CTA clusters; a
 * problem whose plan and partials need more than 40 MiB (more than about
 * 5,000,000 (row block, request) units) returns MLA_ERR_WORKSPACE and launches
 * nothing.
 * All calls share the array: calls that overlap on the GPU race, so serialise
 * them.  With check_device_error != 0 the call synchronises `stream` and
 * returns the device error status (as mla_get_device_error()); otherwise it
 * returns without synchronising, and mla_noalloc_get_device_error() reads the
 * status later.
 */
mla_status mla_decode_noalloc(const mla_desc* desc, const void* q, const void* kv_pages, const float* kv_scales,
                              const int32_t* block_table, const int32_t* seqlens, int32_t s_q, float softmax_scale,
                              void* out, float* lse, int check_device_error, void* stream);

/*
 * The device error status of the last mla_decode_noalloc() on the current
 * device (same codes as mla_get_device_error()), for callers that ran it
 * without check_device_error.  Synchronises `stream` and reads the error word
 * in the library's scratch array; the next mla_decode_noalloc() clears it.
 */
mla_status mla_noalloc_get_device_error(void* stream);

/*
 * Matrix absorption around the attention step (best-practice digest §2.4.3:
 * the --mla_use_matrix_absorption switch of the DeepSeek deployment scripts;
 * the pages give only the switch, the algebra is standard MLA).  With
 * per-head up-projections W_UK[h], W_UV[h] of shape [512, 128] (latent x
 * head dim), attention over the latent cache with an absorbed query equals
 * standard MLA attention:
 *
 *   mla_absorb_q:     q[t, h, 0:512]   = W_UK[h] @ q_nope[t, h]      (128 -> 512)
 *                     q[t, h, 512:576] = q_rope[t, h]
 *   mla_project_out:  o[t, h]          = W_UV[h]^T @ out[t, h]       (512 -> 128)
 *
 * t runs over the `tokens` = B * s_q token rows in mla_decode()'s order
 * (b-major, then i), so q and out are exactly mla_decode()'s q and out.
 * Both are per-head tcgen05 GEMMs with fp32 accumulation and bf16 results.
 *
 *   q_nope     device, bf16 [tokens, H, 128], contiguous, 16-byte aligned
 *   q_rope     device, bf16 [tokens, H, 64], contiguous, 16-byte aligned
 *   w_uk, w_uv device, bf16 [H, 512, 128], contiguous, 16-byte aligned
 *   q          device, bf16 [tokens, H, 576], 16-byte aligned (written)
 *   out        device, bf16 [tokens, H, 512], 16-byte aligned
 *   o          device, bf16 [tokens, H, 128], 16-byte aligned (written)
 *   tokens     >= 1;  num_heads 1..1024
 *   workspace  an mla_decode() workspace whose error word records a pipeline
 *              timeout (MLA_ERR_DEVICE_TIMEOUT through mla_get_device_error()),
 *              or NULL; 256-byte aligned when given
 *
 * Host-visible problems return a negative status and launch nothing; the
 * call is asynchronous on `stream` and allocates nothing.
 */
mla_status mla_absorb_q(const void* q_nope, const void* q_rope, const void* w_uk, int32_t tokens,
                        int32_t num_heads, void* q, void* workspace, void* stream);
mla_status mla_project_out(const void* out, const void* w_uv, int32_t tokens, int32_t num_heads, void* o,
                           void* workspace, void* stream);

/* Static, NUL-terminated description of a status code. */
const char* mla_status_string(int status);

/* Byte offsets of the workspace regions (for tests and tools that inspect the
 * plan).  The header is int32 words: [0] error bits, [1] W, [2] total cost,
 * [3] units, [4] clusters, [5] plan overhead, [6] number of units of more
 * than three pieces (the combine jobs of mla_combine_workspace()), [7] stall request:
 * mla_plan() writes 0; a nonzero value written there afterwards makes the next
 * mla_decode_attention() wait on a barrier that nothing signals, so its
 * bounded pipeline wait runs out and it reports MLA_ERR_DEVICE_TIMEOUT (for
 * testing the timeout path without a fault).  cl_first is int32 [clusters] (first
 * unit each cluster touches), pre is int32 [units + 1] (cost prefix), sync is
 * int32 [8*clusters]: merge counters [clusters] and partial-slot ready flags
 * [2*clusters] (mla_plan() clears them and every completed attention kernel
 * leaves them clear), then at [4*clusters] the combine jobs as int32 x 4
 * (unit, first cluster, last cluster, slot of the first piece),
 * lse_part fp32 [2*clusters, 128, 2] (lse of the piece, power-of-two scale of
 * its stored output), o_part fp16 [2*clusters][64 chunks][128 rows][8] (slot
 * s, row r, channel ch at ((s*64 + ch/8)*128 + r)*8 + ch%8; the piece's
 * normalised output is the stored value times the scale). */
typedef struct {
  size_t header, cl_first, pre, lse_part, o_part, sync, total;
} mla_workspace_layout;
mla_status mla_get_workspace_layout(const mla_desc* desc, int num_clusters, mla_workspace_layout* layout);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H_ */
