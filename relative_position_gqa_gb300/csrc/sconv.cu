// Window-4 causal depthwise short convolution on K and V, fused into the paged KV-cache
// write, with the 3-row sconv cache moved forward in place (vLLM Day-0 Inkling blog,
// "Model Architecture / Sconv" and "vLLM Integration & Optimization / Managing the
// sconv cache").
//
// One thread owns 8 consecutive channels of K or of V for a run of kChunk consecutive new
// tokens of one sequence: it keeps the three previous raw rows in registers, so each raw
// row is read once (plus a 3-row halo per run) and each conv output is written once,
// straight into its page.  The thread that owns the first run of a sequence is the only
// reader of the old sconv state for its channels, so it can also write the new state
// without racing anyone.  HBM-bound: 16-byte loads and stores, a warp covers 512
// contiguous bytes of a raw row.
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ink {

constexpr int kChunk = 32;    // new tokens per thread
constexpr int kVec = 8;       // channels per thread (one 16-byte vector of bf16)
constexpr int kSconvThreads = 128;

struct F8 { float v[8]; };

__device__ __forceinline__ F8 unpack8(uint4 u) {
  F8 f;
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f.v[2 * i] = __uint_as_float(w[i] << 16);
    f.v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
  return f;
}

__global__ void __launch_bounds__(kSconvThreads)
sconv_kv_kernel(const uint16_t* __restrict__ k_raw, const uint16_t* __restrict__ v_raw,
                const float* __restrict__ w_k, const float* __restrict__ w_v,
                uint16_t* __restrict__ state, const int32_t* __restrict__ cu_q_lens,
                const int64_t* __restrict__ slot_mapping, uint16_t* __restrict__ k_cache,
                uint16_t* __restrict__ v_cache, int Hkv, long long num_slots, int max_q_len,
                int* __restrict__ status) {
  const int C = Hkv * 128;
  const int vecs_per_kind = C / kVec;
  const int vec = blockIdx.x * kSconvThreads + threadIdx.x;
  if (vec >= 2 * vecs_per_kind) return;
  const int which = vec / vecs_per_kind;  // 0 = K, 1 = V
  const int c0 = (vec % vecs_per_kind) * kVec;
  const int b = blockIdx.z;
  const int t_begin = cu_q_lens[b];
  const int n = cu_q_lens[b + 1] - t_begin;
  if (n < 0 || n > max_q_len) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(status, kErrBadInput);
    return;
  }
  const int ts = blockIdx.y * kChunk;
  if (ts >= n) return;
  const int te = min(ts + kChunk, n);

  const uint16_t* x = which == 0 ? k_raw : v_raw;
  const float* w = which == 0 ? w_k : w_v;
  uint16_t* cache = which == 0 ? k_cache : v_cache;
  uint16_t* st = state + ((size_t)b * 2 + which) * 3 * C + c0;

  float tap[kVec][4];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float4 t4 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(c0 + i) * 4));
    tap[i][0] = t4.x; tap[i][1] = t4.y; tap[i][2] = t4.z; tap[i][3] = t4.w;
  }

  // the three rows before `ts`, oldest first
  uint4 hist_raw[3];
  if (ts == 0) {
#pragma unroll
    for (int r = 0; r < 3; ++r)
      hist_raw[r] = *reinterpret_cast<const uint4*>(st + (size_t)r * C);
  } else {
#pragma unroll
    for (int r = 0; r < 3; ++r)
      hist_raw[r] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + ts - 3 + r) * C + c0));
  }
  const uint4 old_state[3] = {hist_raw[0], hist_raw[1], hist_raw[2]};
  F8 h0 = unpack8(hist_raw[0]), h1 = unpack8(hist_raw[1]), h2 = unpack8(hist_raw[2]);

  const int head = c0 >> 7, d0 = c0 & 127;
  for (int t = ts; t < te; ++t) {
    const int tg = t_begin + t;
    const F8 cur = unpack8(__ldg(reinterpret_cast<const uint4*>(x + (size_t)tg * C + c0)));
    float y[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      float a = tap[i][0] * h0.v[i];
      a = fmaf(tap[i][1], h1.v[i], a);
      a = fmaf(tap[i][2], h2.v[i], a);
      a = fmaf(tap[i][3], cur.v[i], a);
      y[i] = a;
    }
    const long long slot = slot_mapping[tg];
    if (slot >= num_slots) {
      report(status, kErrBadBlock);
    } else if (slot >= 0) {
      const long long blk = slot >> 7, off = slot & 127;
      uint4 o;
      o.x = pack_bf16(y[0], y[1]);
      o.y = pack_bf16(y[2], y[3]);
      o.z = pack_bf16(y[4], y[5]);
      o.w = pack_bf16(y[6], y[7]);
      *reinterpret_cast<uint4*>(cache + (((size_t)blk * Hkv + head) * 128 + off) * 128 + d0) = o;
    }
    h0 = h1; h1 = h2; h2 = cur;
  }

  if (ts == 0) {
    // new state = last three rows of [old state ; new rows]
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int idx = n - 3 + r;  // index among the new rows
      uint4 v;
      if (idx >= 0) {
        v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + idx) * C + c0));
      } else {
        v = old_state[3 + idx];
      }
      *reinterpret_cast<uint4*>(st + (size_t)r * C) = v;
    }
  }
}

cudaError_t launch_sconv_kv(const SconvArgs& a, cudaStream_t stream) {
  const int C = a.Hkv * 128;
  const int total_vecs = 2 * C / kVec;
  dim3 grid((total_vecs + kSconvThreads - 1) / kSconvThreads,
            (a.max_q_len + kChunk - 1) / kChunk, a.B);
  if (grid.y == 0 || grid.z == 0) return cudaSuccess;
  sconv_kv_kernel<<<grid, kSconvThreads, 0, stream>>>(
      static_cast<const uint16_t*>(a.k_raw), static_cast<const uint16_t*>(a.v_raw), a.w_k, a.w_v,
      static_cast<uint16_t*>(a.state), a.cu_q_lens, a.slot_mapping,
      static_cast<uint16_t*>(a.k_cache), static_cast<uint16_t*>(a.v_cache), a.Hkv,
      (long long)a.num_blocks * 128, a.max_q_len, a.dev_status);
  return cudaGetLastError();
}

}  // namespace ink
