// Private launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

namespace ink {

// Launch with programmatic stream serialization allowed: the kernel may begin while the
// previous kernel on the stream drains, and every kernel of the library starts with
// pdl_wait() before it touches global inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct SconvArgs {
  const void* k_raw;
  const void* v_raw;
  const float* w_k;
  const float* w_v;
  void* state;
  const int32_t* cu_q_lens;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  int B, T, Hkv;
  long long num_blocks;
  int max_q_len;
  int* dev_status;
  bool fp8 = false;  // caches hold E4M3 bytes: code = e4m3(y / scale)
  float k_scale = 1.f, v_scale = 1.f;
};

struct SconvDenseArgs {
  const void* x;
  const float* w;
  void* state;
  const int32_t* cu_q_lens;
  void* y;
  int B, T, C, max_q_len;
  int* dev_status;
};

struct SconvRollbackArgs {
  const void* state_before;
  const void* x0;
  const void* x1;  // nullptr when streams == 1
  const int32_t* cu_q_lens;
  const int32_t* accepted;
  void* state_after;
  int B, T, C, streams;
  int* dev_status;
};

struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const float* bias;
  int R;
  float scale;
  int window;
  void* out;
  int out_dtype;  // 0 = bf16, 1 = fp32
  float* lse;
  int B, T, Hq, Hkv;
  long long num_blocks;
  int max_q_len;
  int* dev_status;
  // decode only
  int max_seq_len;
  int num_splits;
  int pages_per_split;
  void* workspace;
  size_t workspace_bytes;
  // FP8 (E4M3) cache: K = code * k_scale, V = code * v_scale (decode only)
  bool kv_fp8 = false;
  float k_scale = 1.f, v_scale = 1.f;
  // prefill only: factor on the output (v_scale when the pages were widened from FP8)
  float out_scale = 1.f;
  // decode with the step's conv fused into its prologue (bf16 cache): the new tokens'
  // raw K/V rows [T][Hkv*128], the taps [Hkv*128][4], the state [B][2][3][Hkv*128]
  // (in/out); the new rows go into k_cache / v_cache at the slots the block table gives
  const void* conv_k_raw = nullptr;
  const void* conv_v_raw = nullptr;
  const float* conv_w_k = nullptr;
  const float* conv_w_v = nullptr;
  void* conv_state = nullptr;
};

// Tensor maps built by the host for the attention kernels.
struct AttnMaps {
  CUtensorMap q;  // (d=128, head=Hq, token=T), box (64, 1, 128), 128-byte swizzle
  CUtensorMap k;  // (d=128, slot=128, page*Hkv+head), box (64, 128, 1), 128-byte swizzle
  CUtensorMap v;
};

cudaError_t launch_sconv_kv(const SconvArgs& a, cudaStream_t stream);
cudaError_t launch_sconv_dense(const SconvDenseArgs& a, cudaStream_t stream);
cudaError_t launch_sconv_rollback(const SconvRollbackArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream);
cudaError_t launch_decode(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream);
// Prefill over an FP8 cache: pages a step's queries can see, widened to a bf16 pool.
size_t prefill_fp8_range_pages(int max_q_len, int max_seq_len, int window);
size_t prefill_fp8_workspace_bytes(int B, int Hkv, int max_blocks, int max_q_len,
                                   int max_seq_len, int window);
cudaError_t launch_widen_pages(const AttnArgs& a, void* k16, void* v16, int32_t* table16,
                               int range_pages, cudaStream_t stream);

// Decode split rule shared by the workspace query and the launch.
struct DecodeSplit {
  int num_splits;
  int pages_per_split;
};
DecodeSplit decode_split(int B, int Hkv, int max_q_len, int max_seq_len, int window,
                         int num_splits_req, int num_sms);
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int max_q_len, int num_splits);

}  // namespace ink
