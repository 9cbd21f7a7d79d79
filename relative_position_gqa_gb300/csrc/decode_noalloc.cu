// A decode entry point that allocates nothing: the split-KV partials live in a static
// device array of this file instead of a caller-provided workspace.
//
// Who needs it: callers that cannot hand the library a device buffer of their own, e.g. a
// runtime that plans every device byte once at start-up and forbids cudaMalloc while
// serving (cudaMalloc can synchronise the device and is not allowed in a stream being
// captured), or a caller that runs inside another framework's allocator and must not
// re-enter it.  The array below is part of the loaded library: every GPU that loads it
// holds these bytes until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <mutex>

#include "../../include/inkling.h"
#include "kernels.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB per device

// Device storage for the partial (m, l, O) rows of split sequences.  In host code this
// name is only a stand-in: the address a kernel may use comes from
// cudaGetSymbolAddress, looked up with the device current.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// The address is looked up once per device and CUDA context.  A context has an id that
// is never reused within the process (cuCtxGetId), so after a device reset (the module
// is loaded again and the array may sit elsewhere) the next call finds a new id and looks
// the address up again instead of handing a kernel a stale pointer.
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_entry_once;

void load_entry_points() {
  std::call_once(g_entry_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
}

// Id of the calling thread's current context; false when there is none (or no way to ask).
bool current_context_id(unsigned long long* id) {
  load_entry_points();
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

constexpr int kMaxDevices = 64;
struct ScratchSlot {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;
  bool keyed = false;  // ctx_id is valid
};
std::mutex g_mutex;
ScratchSlot g_slots[kMaxDevices];

// The scratch address on the current device, looked up on the first call there (and on
// the first call after that device's context was replaced).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return INKLING_ERR_CUDA;
  unsigned long long id = 0;
  bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_mutex);
  ScratchSlot& slot = g_slots[dev];
  if (slot.ptr != nullptr && slot.keyed && have_id && slot.ctx_id == id) {
    *out = slot.ptr;
    return INKLING_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
    return INKLING_ERR_CUDA;
  // the lookup makes the device's primary context current when no context was
  if (!have_id) have_id = current_context_id(&id);
  slot.ptr = p;
  slot.ctx_id = id;
  slot.keyed = have_id;  // without an id the address is looked up again next call
  *out = p;
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
  // The scratch goes in as the workspace of inkling_rel_attn_decode, which runs all of its
  // argument checks first and only then compares the partials' size with the workspace
  // (INKLING_ERR_WORKSPACE when they would not fit the scratch): the same checks, in the
  // same order, and the same split rule.
  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != INKLING_OK) return rc;
  return inkling_rel_attn_decode(q, k_cache, v_cache, block_table, max_blocks, cu_q_lens,
                                 seq_lens, bias, R, scale, window, out, out_dtype, lse, B, T, Hq,
                                 Hkv, num_blocks, max_q_len, max_seq_len, num_splits, scratch,
                                 kScratchBytes, dev_status, stream);
}

}  // extern "C"
