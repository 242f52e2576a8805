// mla_decode_noalloc: the whole decode step without a caller-provided
// workspace and without any device allocation.
//
// Some callers cannot allocate device memory when they call the decoder:
// serving loops and plugin hosts that reserve all device memory up front and
// forbid allocation afterwards (cudaMalloc may synchronise the device and
// fragment a planned pool), and C callers that own only their input and output
// buffers and have no allocator to draw a workspace from.  For them the
// scratch this call needs (split plan, error word, the fp16 partial outputs of
// split requests) lives in a fixed array compiled into the library.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (40 MiB).  Every GPU on which this module gets loaded holds it until the
// process exits.  Host code cannot use the array's name as a device address,
// so the first call on each device (with that device current) looks the
// address up with cudaGetSymbolAddress and caches it; make that first call
// before any stream capture.
//
// All calls share the one array, which keeps what the last call wrote.  The
// plan kernel rewrites the plan and clears the error word at the start of every
// call and partials are written before they are read, so nothing needs
// clearing between calls.  Calls whose work overlaps on the GPU (different
// streams, or different host threads) race on the array: serialise them.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "mla.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(40) << 20;
constexpr int kNoAllocMaxClusters = 76;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};

// Device address of the scratch array on the current device (looked up once
// per device), or nullptr if the lookup failed.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" mla_status mla_decode_noalloc(const mla_desc* desc, const void* q, const void* kv_pages,
                                         const float* kv_scales, const int32_t* block_table, const int32_t* seqlens,
                                         int32_t s_q, float softmax_scale, void* out, float* lse,
                                         int check_device_error, void* stream) {
  if (!desc) return MLA_ERR_INVALID_ARG;
  mla_desc d = *desc;
  if (d.max_clusters <= 0 || d.max_clusters > kNoAllocMaxClusters) d.max_clusters = kNoAllocMaxClusters;
  const size_t need = mla_workspace_size(&d, 0);
  if (need == 0) return MLA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;  // problem larger than the static scratch
  void* scratch = scratch_address();
  if (!scratch) return MLA_ERR_CUDA;
  mla_status st = mla_decode(&d, q, kv_pages, kv_scales, block_table, seqlens, s_q, softmax_scale, out, lse,
                             scratch, kNoAllocScratchBytes, stream);
  if (st != MLA_OK || !check_device_error) return st;
  return mla_get_device_error(scratch, stream);
}

// The error word of the last mla_decode_noalloc() on the current device, for
// callers that ran it without check_device_error (for instance from a
// captured graph): synchronises `stream` and reads the word through the
// scratch array's cached device address.
extern "C" mla_status mla_noalloc_get_device_error(void* stream) {
  void* scratch = scratch_address();
  if (!scratch) return MLA_ERR_CUDA;
  return mla_get_device_error(scratch, stream);
}
