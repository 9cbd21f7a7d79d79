// A decode entry point that allocates nothing: the split-KV partials live in a static
// device array of this file instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand the library a device buffer of their own, e.g. a
// runtime that plans every device byte once at start-up and forbids cudaMalloc while
// serving (cudaMalloc can synchronise the device and is not allowed in a stream being
// captured), or a caller that runs inside another framework's allocator and must not
// re-enter it.  The array below is part of the loaded library: every GPU that loads it
// holds these bytes until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/inkling.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device

// Device storage for the partial (m, l, O) rows of split sequences.  In host code this
// name is only a stand-in: the address a kernel may use comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// The scratch address on the current device, resolved on the first call on that device.
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return INKLING_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return INKLING_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return INKLING_OK;
}

}  // namespace

extern "C" {

size_t inkling_rel_attn_decode_noalloc_capacity(void) { return kScratchBytes; }

int inkling_rel_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks,
                                    const int32_t* cu_q_lens, const int32_t* seq_lens,
                                    const float* bias, int32_t R, float scale, int32_t window,
                                    void* out, int32_t out_dtype, float* lse, int32_t B,
                                    int32_t T, int32_t Hq, int32_t Hkv, int64_t num_blocks,
                                    int32_t max_q_len, int32_t max_seq_len, int32_t num_splits,
                                    int32_t* dev_status, inkling_stream_t stream) {
  // Same checks and split rule as inkling_rel_attn_decode; the only difference is where
  // the partials go.
  const size_t need = inkling_rel_attn_decode_workspace_size(B, Hq, Hkv, max_q_len, max_seq_len,
                                                             window, num_splits);
  if (need > kScratchBytes) return INKLING_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = scratch_address(&scratch);
    if (rc != INKLING_OK) return rc;
  }
  return inkling_rel_attn_decode(q, k_cache, v_cache, block_table, max_blocks, cu_q_lens,
                                 seq_lens, bias, R, scale, window, out, out_dtype, lse, B, T, Hq,
                                 Hkv, num_blocks, max_q_len, max_seq_len, num_splits, scratch,
                                 need > 0 ? kScratchBytes : 0, dev_status, stream);
}

}  // extern "C"
