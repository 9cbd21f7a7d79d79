// Prefill over an FP8 (E4M3) KV cache (vLLM Day-0 Inkling blog, "Roadmap": FP8 for the
// global-attention layers).  The prefill is bound by the tensor core, not by its K/V
// reads, so it keeps its bf16 kernel: a first pass widens the pages that the step's
// queries can see into a bf16 page pool in the caller's workspace, with a block table of
// its own, and the prefill kernel then runs on that pool.  E4M3 values are exact in bf16,
// so the widening rounds nothing; k_scale is folded into the logit scale and v_scale into
// the output, as in the FP8 decode.  The widening moves 1 + 2 bytes per cache element of
// the visible pages, small next to the attention's work on them.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ink {

struct WidenParams {
  const uint8_t* k8;        // [num_blocks][Hkv][128][128] E4M3
  const uint8_t* v8;
  const int32_t* block_table;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  uint16_t* k16;            // [B * range_pages][Hkv][128][128] bf16
  uint16_t* v16;
  int32_t* table16;         // [B][max_blocks]: logical page -> page of the bf16 pool
  int* status;
  long long num_blocks;
  int max_blocks, Hkv, window, range_pages, max_q_len;
};

constexpr int kWidenThreads = 256;

__device__ __forceinline__ float f16_to_f32(uint32_t h) {
  float f;
  asm("cvt.f32.f16 %0, %1;" : "=f"(f) : "h"((unsigned short)h));
  return f;
}

// 16 E4M3 bytes -> 16 bf16 values (two 16-byte stores), exactly.
__device__ __forceinline__ void widen16(const uint4 in, uint4* out) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t f16x2 = e4m3x2_to_f16x2((uint16_t)(w[i] >> (16 * h)));
      const float lo = f16_to_f32(f16x2 & 0xffffu);
      const float hi = f16_to_f32(f16x2 >> 16);
      o[2 * i + h] = pack_bf16(lo, hi);
    }
  }
  out[0] = make_uint4(o[0], o[1], o[2], o[3]);
  out[1] = make_uint4(o[4], o[5], o[6], o[7]);
}

// One CTA per (visible page j of sequence b, KV head): widen its K and V pages.
__global__ void __launch_bounds__(kWidenThreads) widen_pages_kernel(const WidenParams p) {
  pdl_wait();
  const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int t0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - t0;
  const int L = p.seq_lens[b];
  if (n <= 0) return;
  if (n > L || n > p.max_q_len || L > p.max_blocks * 128) {
    if (j == 0 && kvh == 0 && threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  // pages any query row of the sequence can see
  const int lo = p.window > 0 ? max(0, (L - n) - p.window + 1) : 0;
  const int kt_lo = lo >> 7, kt_hi = (L - 1) >> 7;
  if (kt_hi - kt_lo + 1 > p.range_pages) {  // host bound max_seq_len too small
    if (j == 0 && kvh == 0 && threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  const int kt = kt_lo + j;
  if (kt > kt_hi) return;
  const int32_t blk = p.block_table[(size_t)b * p.max_blocks + kt];
  const long long dst_page = (long long)b * p.range_pages + j;
  if (kvh == 0 && threadIdx.x == 0) p.table16[(size_t)b * p.max_blocks + kt] = (int32_t)dst_page;
  if (blk < 0 || (long long)blk >= p.num_blocks) {
    if (threadIdx.x == 0) report(p.status, kErrBadBlock);
    return;
  }
  const size_t src = ((size_t)blk * p.Hkv + kvh) * 16384;             // bytes
  const size_t dst = ((size_t)dst_page * p.Hkv + kvh) * 16384;        // bf16 elements
  const uint4* k_in = reinterpret_cast<const uint4*>(p.k8 + src);
  const uint4* v_in = reinterpret_cast<const uint4*>(p.v8 + src);
  uint4* k_out = reinterpret_cast<uint4*>(p.k16 + dst);
  uint4* v_out = reinterpret_cast<uint4*>(p.v16 + dst);
  // 1024 chunks of 16 bytes per page: four per thread per tensor, all loads first
  uint4 kin[4], vin[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    kin[u] = __ldg(k_in + threadIdx.x + u * kWidenThreads);
    vin[u] = __ldg(v_in + threadIdx.x + u * kWidenThreads);
  }
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int c = threadIdx.x + u * kWidenThreads;
    widen16(kin[u], k_out + 2 * c);
    widen16(vin[u], v_out + 2 * c);
  }
}

size_t prefill_fp8_range_pages(int max_q_len, int max_seq_len, int window) {
  long long rp = ((long long)max_seq_len + 127) / 128;
  if (window > 0) {
    const long long w = ((long long)max_q_len + window - 1 + 127) / 128 + 1;
    if (w < rp) rp = w;
  }
  return rp < 1 ? 1 : (size_t)rp;
}

size_t prefill_fp8_workspace_bytes(int B, int Hkv, int max_blocks, int max_q_len,
                                   int max_seq_len, int window) {
  const size_t pages = (size_t)B * prefill_fp8_range_pages(max_q_len, max_seq_len, window);
  return 2 * pages * (size_t)Hkv * 128 * 128 * 2 + (size_t)B * max_blocks * 4;
}

cudaError_t launch_widen_pages(const AttnArgs& a, void* k16, void* v16, int32_t* table16,
                               int range_pages, cudaStream_t stream) {
  WidenParams p;
  p.k8 = static_cast<const uint8_t*>(a.k_cache);
  p.v8 = static_cast<const uint8_t*>(a.v_cache);
  p.block_table = a.block_table;
  p.cu_q_lens = a.cu_q_lens;
  p.seq_lens = a.seq_lens;
  p.k16 = static_cast<uint16_t*>(k16);
  p.v16 = static_cast<uint16_t*>(v16);
  p.table16 = table16;
  p.status = a.dev_status;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.Hkv = a.Hkv;
  p.window = a.window;
  p.range_pages = range_pages;
  p.max_q_len = a.max_q_len;
  const dim3 grid(range_pages, a.Hkv, a.B);
  return launch_pdl(widen_pages_kernel, grid, dim3(kWidenThreads), 0, stream, p);
}

}  // namespace ink
