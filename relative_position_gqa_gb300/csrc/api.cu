// C ABI of the Inkling attention-block library: host-side argument checks, tensor-map
// construction for the TMA loads, split selection, and the launches.  No device memory is
// allocated here and nothing is synchronised.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/inkling.h"
#include "kernels.h"

namespace {

using ink::AttnArgs;
using ink::AttnMaps;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// 3-D bf16 tensor map, 128-byte swizzle, box inner extent 64 elements (128 bytes).
bool make_map3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
               uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1,
               uint32_t b2, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  cuuint32_t box[3] = {b0, b1, b2};
  cuuint32_t es[3] = {1, 1, 1};
  return g_encode(m, dtype, 3, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int num_sms_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}

// Checks shared by prefill and decode.  Returns INKLING_OK or the error.
int check_attn(const AttnArgs& a) {
  if (!a.q || !a.k_cache || !a.v_cache || !a.block_table || !a.cu_q_lens || !a.seq_lens ||
      !a.bias || !a.out)
    return INKLING_ERR_INVALID_ARG;
  if (a.B < 0 || a.T < 0 || a.Hq <= 0 || a.Hkv <= 0 || a.max_blocks <= 0 || a.num_blocks <= 0 ||
      a.max_q_len < 0)
    return INKLING_ERR_INVALID_ARG;
  if (a.Hq % a.Hkv != 0) return INKLING_ERR_INVALID_ARG;
  if (a.R < 1 || a.window < 0) return INKLING_ERR_INVALID_ARG;
  if (a.out_dtype != INKLING_OUT_BF16 && a.out_dtype != INKLING_OUT_F32) return INKLING_ERR_INVALID_ARG;
  if (!(a.scale == a.scale)) return INKLING_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.k_cache) || !aligned16(a.v_cache) || !aligned16(a.out))
    return INKLING_ERR_INVALID_ARG;
  if ((long long)a.num_blocks * a.Hkv > 0x7fffffffLL) return INKLING_ERR_UNSUPPORTED;
  if ((long long)a.max_blocks * 128 > 0x7fffffffLL) return INKLING_ERR_UNSUPPORTED;
  return INKLING_OK;
}

int build_maps(const AttnArgs& a, AttnMaps* maps, bool need_q) {
  if (!get_encoder()) return INKLING_ERR_CUDA;
  if (need_q && a.T > 0 &&
      !make_map3(&maps->q, a.q, 128, (uint64_t)a.Hq, (uint64_t)a.T, 256, (uint64_t)a.Hq * 256, 64, 1,
                 128))
    return INKLING_ERR_INVALID_ARG;
  const uint64_t pages = (uint64_t)a.num_blocks * a.Hkv;
  if (a.kv_fp8) {
    // E4M3 pages: one 128-byte x 128-slot box per page-head
    if (!make_map3(&maps->k, a.k_cache, 128, 128, pages, 128, 16384, 128, 128, 1,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8) ||
        !make_map3(&maps->v, a.v_cache, 128, 128, pages, 128, 16384, 128, 128, 1,
                   CU_TENSOR_MAP_DATA_TYPE_UINT8))
      return INKLING_ERR_INVALID_ARG;
    return INKLING_OK;
  }
  if (!make_map3(&maps->k, a.k_cache, 128, 128, pages, 256, 32768, 64, 128, 1))
    return INKLING_ERR_INVALID_ARG;
  if (!make_map3(&maps->v, a.v_cache, 128, 128, pages, 256, 32768, 64, 128, 1))
    return INKLING_ERR_INVALID_ARG;
  return INKLING_OK;
}

}  // namespace

extern "C" {

const char* inkling_status_string(int status) {
  switch (status) {
    case INKLING_OK: return "ok";
    case INKLING_ERR_INVALID_ARG: return "invalid argument";
    case INKLING_ERR_UNSUPPORTED: return "unsupported shape";
    case INKLING_ERR_CUDA: return "CUDA error";
    case INKLING_ERR_TIMEOUT: return "device wait timed out";
    case INKLING_ERR_BAD_BLOCK: return "page id or slot outside the cache";
    case INKLING_ERR_BAD_INPUT: return "sequence lengths inconsistent with the limits";
    case INKLING_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
  }
}

int inkling_version(void) { return 0x000100; }

int inkling_sconv_kv(const void* k_raw, const void* v_raw, const float* w_k, const float* w_v,
                     void* sconv_state, const int32_t* cu_q_lens, const int64_t* slot_mapping,
                     void* k_cache, void* v_cache, int32_t B, int32_t T, int32_t Hkv,
                     int64_t num_blocks, int32_t max_q_len, int32_t* dev_status,
                     inkling_stream_t stream) {
  if (B < 0 || T < 0 || Hkv <= 0 || num_blocks <= 0 || max_q_len < 0) return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0 || max_q_len == 0) return INKLING_OK;
  if (!k_raw || !v_raw || !w_k || !w_v || !sconv_state || !cu_q_lens || !slot_mapping ||
      !k_cache || !v_cache)
    return INKLING_ERR_INVALID_ARG;
  if (!aligned16(k_raw) || !aligned16(v_raw) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(sconv_state) || !aligned16(k_cache) || !aligned16(v_cache))
    return INKLING_ERR_INVALID_ARG;
  if (B > 65535 || (max_q_len + 31) / 32 > 65535) return INKLING_ERR_UNSUPPORTED;
  ink::SconvArgs a{k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache,
                   v_cache, B, T, Hkv, (long long)num_blocks, max_q_len, dev_status};
  return ink::launch_sconv_kv(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

int inkling_sconv_kv_fp8(const void* k_raw, const void* v_raw, const float* w_k,
                         const float* w_v, void* sconv_state, const int32_t* cu_q_lens,
                         const int64_t* slot_mapping, void* k_cache, void* v_cache,
                         float k_scale, float v_scale, int32_t B, int32_t T, int32_t Hkv,
                         int64_t num_blocks, int32_t max_q_len, int32_t* dev_status,
                         inkling_stream_t stream) {
  if (B < 0 || T < 0 || Hkv <= 0 || num_blocks <= 0 || max_q_len < 0) return INKLING_ERR_INVALID_ARG;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0 || max_q_len == 0) return INKLING_OK;
  if (!k_raw || !v_raw || !w_k || !w_v || !sconv_state || !cu_q_lens || !slot_mapping ||
      !k_cache || !v_cache)
    return INKLING_ERR_INVALID_ARG;
  if (!aligned16(k_raw) || !aligned16(v_raw) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(sconv_state) || !aligned16(k_cache) || !aligned16(v_cache))
    return INKLING_ERR_INVALID_ARG;
  if (B > 65535 || (max_q_len + 31) / 32 > 65535) return INKLING_ERR_UNSUPPORTED;
  ink::SconvArgs a{k_raw, v_raw, w_k, w_v, sconv_state, cu_q_lens, slot_mapping, k_cache,
                   v_cache, B, T, Hkv, (long long)num_blocks, max_q_len, dev_status};
  a.fp8 = true;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return ink::launch_sconv_kv(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

int inkling_sconv(const void* x, const float* w, void* sconv_state, const int32_t* cu_q_lens,
                  void* y, int32_t B, int32_t T, int32_t C, int32_t max_q_len,
                  int32_t* dev_status, inkling_stream_t stream) {
  if (B < 0 || T < 0 || C <= 0 || C % 8 != 0 || max_q_len < 0) return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0 || max_q_len == 0) return INKLING_OK;
  if (!x || !w || !sconv_state || !cu_q_lens || !y) return INKLING_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w) || !aligned16(sconv_state) || !aligned16(y))
    return INKLING_ERR_INVALID_ARG;
  if (x == y) return INKLING_ERR_INVALID_ARG;
  if (B > 65535 || (max_q_len + 31) / 32 > 65535) return INKLING_ERR_UNSUPPORTED;
  ink::SconvDenseArgs a{x, w, sconv_state, cu_q_lens, y, B, T, C, max_q_len, dev_status};
  return ink::launch_sconv_dense(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

int inkling_sconv_state_rollback(const void* state_before, const void* x0, const void* x1,
                                 const int32_t* cu_q_lens, const int32_t* accepted,
                                 void* state_after, int32_t B, int32_t T, int32_t C,
                                 int32_t streams, int32_t* dev_status,
                                 inkling_stream_t stream) {
  if (B < 0 || T < 0 || C <= 0 || C % 8 != 0 || (streams != 1 && streams != 2))
    return INKLING_ERR_INVALID_ARG;
  if (B == 0) return INKLING_OK;
  if (!state_before || !x0 || !cu_q_lens || !accepted || !state_after) return INKLING_ERR_INVALID_ARG;
  if (streams == 2 && !x1) return INKLING_ERR_INVALID_ARG;
  if (!aligned16(state_before) || !aligned16(x0) || (streams == 2 && !aligned16(x1)) ||
      !aligned16(state_after))
    return INKLING_ERR_INVALID_ARG;
  if (B > 65535) return INKLING_ERR_UNSUPPORTED;
  ink::SconvRollbackArgs a{state_before, x0, streams == 2 ? x1 : nullptr, cu_q_lens, accepted,
                           state_after, B, T, C, streams, dev_status};
  return ink::launch_sconv_rollback(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

int inkling_rel_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                             const int32_t* block_table, int32_t max_blocks,
                             const int32_t* cu_q_lens, const int32_t* seq_lens,
                             const float* bias, int32_t R, float scale, int32_t window,
                             void* out, int32_t out_dtype, float* lse, int32_t B, int32_t T,
                             int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
                             int32_t* dev_status, inkling_stream_t stream) {
  AttnArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.block_table = block_table;
  a.max_blocks = max_blocks; a.cu_q_lens = cu_q_lens; a.seq_lens = seq_lens; a.bias = bias;
  a.R = R; a.scale = scale; a.window = window; a.out = out; a.out_dtype = out_dtype; a.lse = lse;
  a.B = B; a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.num_blocks = num_blocks; a.max_q_len = max_q_len;
  a.dev_status = dev_status;
  const int rc = check_attn(a);
  if (rc != INKLING_OK) return rc;
  if (B == 0 || T == 0 || max_q_len == 0) return INKLING_OK;
  AttnMaps maps;
  const int mrc = build_maps(a, &maps, true);
  if (mrc != INKLING_OK) return mrc;
  return ink::launch_prefill(a, maps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

size_t inkling_rel_attn_prefill_fp8_workspace_size(int32_t B, int32_t Hkv, int32_t max_blocks,
                                                   int32_t max_q_len, int32_t max_seq_len,
                                                   int32_t window) {
  if (B <= 0 || Hkv <= 0 || max_blocks <= 0 || max_q_len <= 0 || max_seq_len <= 0 || window < 0)
    return 0;
  return ink::prefill_fp8_workspace_bytes(B, Hkv, max_blocks, max_q_len, max_seq_len, window);
}

int inkling_rel_attn_prefill_fp8(const void* q, const void* k_cache, const void* v_cache,
                                 float k_scale, float v_scale, const int32_t* block_table,
                                 int32_t max_blocks, const int32_t* cu_q_lens,
                                 const int32_t* seq_lens, const float* bias, int32_t R,
                                 float scale, int32_t window, void* out, int32_t out_dtype,
                                 float* lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv,
                                 int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_status,
                                 inkling_stream_t stream) {
  AttnArgs a{};
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.block_table = block_table;
  a.max_blocks = max_blocks; a.cu_q_lens = cu_q_lens; a.seq_lens = seq_lens; a.bias = bias;
  a.R = R; a.scale = scale; a.window = window; a.out = out; a.out_dtype = out_dtype; a.lse = lse;
  a.B = B; a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.num_blocks = num_blocks; a.max_q_len = max_q_len;
  a.dev_status = dev_status; a.max_seq_len = max_seq_len;
  if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
    return INKLING_ERR_INVALID_ARG;
  const int rc = check_attn(a);
  if (rc != INKLING_OK) return rc;
  if (max_seq_len < 0) return INKLING_ERR_INVALID_ARG;
  if (B == 0 || T == 0 || max_q_len == 0 || max_seq_len == 0) return INKLING_OK;
  if (B > 65535 || Hkv > 65535) return INKLING_ERR_UNSUPPORTED;
  const size_t rp = ink::prefill_fp8_range_pages(max_q_len, max_seq_len, window);
  if (rp > 0x7fffffff || (size_t)B * rp * (size_t)Hkv > 0x7fffffff) return INKLING_ERR_UNSUPPORTED;
  const size_t need = ink::prefill_fp8_workspace_bytes(B, Hkv, max_blocks, max_q_len,
                                                       max_seq_len, window);
  if (workspace == nullptr || workspace_bytes < need || !aligned16(workspace))
    return INKLING_ERR_WORKSPACE;
  // the bf16 pool: K pages, V pages, then the pool's block table
  const size_t pool_pages = (size_t)B * rp;
  const size_t pool_bytes = pool_pages * (size_t)Hkv * 128 * 128 * 2;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* k16 = ws;
  void* v16 = ws + pool_bytes;
  int32_t* table16 = reinterpret_cast<int32_t*>(ws + 2 * pool_bytes);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (ink::launch_widen_pages(a, k16, v16, table16, (int)rp, st) != cudaSuccess)
    return INKLING_ERR_CUDA;
  AttnArgs b = a;  // the bf16 prefill on the pool
  b.k_cache = k16; b.v_cache = v16; b.block_table = table16; b.num_blocks = (long long)pool_pages;
  b.scale = scale * k_scale;
  b.out_scale = v_scale;
  AttnMaps maps;
  const int mrc = build_maps(b, &maps, true);
  if (mrc != INKLING_OK) return mrc;
  return ink::launch_prefill(b, maps, st) == cudaSuccess ? INKLING_OK : INKLING_ERR_CUDA;
}

size_t inkling_rel_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv,
                                              int32_t max_q_len, int32_t max_seq_len,
                                              int32_t window, int32_t num_splits) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_q_len <= 0 || max_seq_len <= 0)
    return 0;
  const int sms = num_splits > 0 ? 1 : num_sms_current();
  const ink::DecodeSplit sp =
      ink::decode_split(B, Hkv, max_q_len, max_seq_len, window, num_splits, sms > 0 ? sms : 1);
  return ink::decode_workspace_bytes(B, Hq, Hkv, max_q_len, sp.num_splits);
}

int inkling_rel_attn_decode_plan(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_q_len,
                                 int32_t max_seq_len, int32_t window, int32_t num_splits,
                                 int32_t* plan) {
  if (plan == nullptr || B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_q_len <= 0 ||
      max_q_len > INKLING_MAX_DECODE_Q || max_seq_len <= 0 || window < 0 || num_splits < 0)
    return INKLING_ERR_INVALID_ARG;
  const int sms = num_splits > 0 ? 1 : num_sms_current();
  if (sms <= 0) return INKLING_ERR_CUDA;
  const ink::DecodeSplit sp =
      ink::decode_split(B, Hkv, max_q_len, max_seq_len, window, num_splits, sms);
  const long long grid = (long long)sp.num_splits * Hkv * B;
  plan[0] = sp.num_splits;
  plan[1] = (int32_t)(grid < 0x7fffffffLL ? grid : 0x7fffffffLL);
  plan[2] = sp.pages_per_split;
  plan[3] = sp.num_splits > 1 ? 1 : 0;
  return INKLING_OK;
}

static int decode_entry(bool kv_fp8, float k_scale, float v_scale,
                        const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, int32_t max_blocks,
                            const int32_t* cu_q_lens, const int32_t* seq_lens,
                            const float* bias, int32_t R, float scale, int32_t window,
                            void* out, int32_t out_dtype, float* lse, int32_t B, int32_t T,
                            int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
                            int32_t max_seq_len, int32_t num_splits, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status,
                            inkling_stream_t stream, const AttnArgs* conv = nullptr) {
  AttnArgs a{};
  if (conv != nullptr) {  // the step's conv fused into the decode (bf16 cache only)
    a.conv_k_raw = conv->conv_k_raw;
    a.conv_v_raw = conv->conv_v_raw;
    a.conv_w_k = conv->conv_w_k;
    a.conv_w_v = conv->conv_w_v;
    a.conv_state = conv->conv_state;
  }
  a.q = q; a.k_cache = k_cache; a.v_cache = v_cache; a.block_table = block_table;
  a.max_blocks = max_blocks; a.cu_q_lens = cu_q_lens; a.seq_lens = seq_lens; a.bias = bias;
  a.R = R; a.scale = scale; a.window = window; a.out = out; a.out_dtype = out_dtype; a.lse = lse;
  a.B = B; a.T = T; a.Hq = Hq; a.Hkv = Hkv; a.num_blocks = num_blocks; a.max_q_len = max_q_len;
  a.dev_status = dev_status; a.max_seq_len = max_seq_len;
  a.kv_fp8 = kv_fp8; a.k_scale = k_scale; a.v_scale = v_scale;
  if (kv_fp8 && (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) ||
                 !std::isfinite(v_scale)))
    return INKLING_ERR_INVALID_ARG;
  const int rc = check_attn(a);
  if (rc != INKLING_OK) return rc;
  if (max_q_len > INKLING_MAX_DECODE_Q || max_seq_len < 0 || num_splits < 0)
    return INKLING_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (G > 16 || max_q_len * G > 128) return INKLING_ERR_UNSUPPORTED;
  if (B == 0 || T == 0 || max_q_len == 0 || max_seq_len == 0) return INKLING_OK;
  if (B > 65535 || Hkv > 65535) return INKLING_ERR_UNSUPPORTED;
  const int sms = num_splits > 0 ? 1 : num_sms_current();
  if (sms <= 0) return INKLING_ERR_CUDA;
  const ink::DecodeSplit sp = ink::decode_split(B, Hkv, max_q_len, max_seq_len, window, num_splits, sms);
  if (sp.num_splits > 0x7fffffff) return INKLING_ERR_UNSUPPORTED;
  const size_t need = ink::decode_workspace_bytes(B, Hq, Hkv, max_q_len, sp.num_splits);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return INKLING_ERR_WORKSPACE;
  a.num_splits = sp.num_splits;
  a.pages_per_split = sp.pages_per_split;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  AttnMaps maps;
  const int mrc = build_maps(a, &maps, false);
  if (mrc != INKLING_OK) return mrc;
  return ink::launch_decode(a, maps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? INKLING_OK
             : INKLING_ERR_CUDA;
}

int inkling_rel_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, int32_t max_blocks,
                            const int32_t* cu_q_lens, const int32_t* seq_lens,
                            const float* bias, int32_t R, float scale, int32_t window,
                            void* out, int32_t out_dtype, float* lse, int32_t B, int32_t T,
                            int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
                            int32_t max_seq_len, int32_t num_splits, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status,
                            inkling_stream_t stream) {
  return decode_entry(false, 1.f, 1.f, q, k_cache, v_cache, block_table, max_blocks, cu_q_lens,
                      seq_lens, bias, R, scale, window, out, out_dtype, lse, B, T, Hq, Hkv,
                      num_blocks, max_q_len, max_seq_len, num_splits, workspace,
                      workspace_bytes, dev_status, stream);
}

int inkling_rel_attn_decode_sconv(const void* q, const void* k_raw, const void* v_raw,
                                  const float* w_k, const float* w_v, void* sconv_state,
                                  void* k_cache, void* v_cache, const int32_t* block_table,
                                  int32_t max_blocks, const int32_t* cu_q_lens,
                                  const int32_t* seq_lens, const float* bias, int32_t R,
                                  float scale, int32_t window, void* out, int32_t out_dtype,
                                  float* lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv,
                                  int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
                                  int32_t num_splits, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, inkling_stream_t stream) {
  if (!k_raw || !v_raw || !w_k || !w_v || !sconv_state) return INKLING_ERR_INVALID_ARG;
  if (!aligned16(k_raw) || !aligned16(v_raw) || !aligned16(w_k) || !aligned16(w_v) ||
      !aligned16(sconv_state))
    return INKLING_ERR_INVALID_ARG;
  AttnArgs conv{};
  conv.conv_k_raw = k_raw;
  conv.conv_v_raw = v_raw;
  conv.conv_w_k = w_k;
  conv.conv_w_v = w_v;
  conv.conv_state = sconv_state;
  return decode_entry(false, 1.f, 1.f, q, k_cache, v_cache, block_table, max_blocks, cu_q_lens,
                      seq_lens, bias, R, scale, window, out, out_dtype, lse, B, T, Hq, Hkv,
                      num_blocks, max_q_len, max_seq_len, num_splits, workspace,
                      workspace_bytes, dev_status, stream, &conv);
}

int inkling_rel_attn_decode_fp8(const void* q, const void* k_cache, const void* v_cache,
                                float k_scale, float v_scale, const int32_t* block_table,
                                int32_t max_blocks, const int32_t* cu_q_lens,
                                const int32_t* seq_lens, const float* bias, int32_t R,
                                float scale, int32_t window, void* out, int32_t out_dtype,
                                float* lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv,
                                int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
                                int32_t num_splits, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, inkling_stream_t stream) {
  return decode_entry(true, k_scale, v_scale, q, k_cache, v_cache, block_table, max_blocks,
                      cu_q_lens, seq_lens, bias, R, scale, window, out, out_dtype, lse, B, T,
                      Hq, Hkv, num_blocks, max_q_len, max_seq_len, num_splits, workspace,
                      workspace_bytes, dev_status, stream);
}

}  // extern "C"
