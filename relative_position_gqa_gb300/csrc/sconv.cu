// Window-4 causal depthwise short convolution on K and V, fused into the paged KV-cache
// write, with the 3-row sconv cache moved forward in place (vLLM Day-0 Inkling blog,
// "Model Architecture / Sconv" and "vLLM Integration & Optimization / Managing the
// sconv cache").
//
// The same kernel serves the dense form of the op (one stream, output [T, C] instead of
// cache pages), used for the conv on the attention output ("Model Architecture / Sconv":
// the conv also sits after o_proj), and a rollback kernel recomputes the state when a
// speculative step keeps only a prefix of its tokens ("Model Architecture / MTP",
// "Re-computing MTP KV cache").
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

// New tokens per thread, and rows loaded ahead of use, per form (measured on GB300 for
// 4 x 8192 tokens: the paged K/V conv over 1024 channels wants runs long enough that one
// wave of CTAs covers the batch; the dense conv over 4096 channels wants more loads in
// flight and runs of 256 tokens, whose 3-row halo adds 1.2% to the reads where runs of
// 32 added 9% (32 / 64 / 128 / 256 / 512 tokens: 0.092 / 0.091 / 0.090 / 0.089 / 0.116 ms,
// the last with too few CTAs to keep HBM busy)).
template <bool kPaged> struct SconvShape;
template <> struct SconvShape<true> { static constexpr int kChunk = 64, kBatch = 8; };
template <> struct SconvShape<false> { static constexpr int kChunk = 256, kBatch = 16; };
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

// Raw rows come from one or two streams (K and V); the conv output either lands in the
// paged cache at slot_mapping[t] (head-major pages of 128 slots x 128 channels) or in a
// dense [T, C] tensor.  The state is [B][streams][3][C], oldest row first.
struct SconvDev {
  const uint16_t* x[2];
  const float* w[2];
  uint16_t* out[2];  // paged caches, or the dense output (streams == 1)
  uint16_t* state;
  const int32_t* cu_q_lens;
  const int64_t* slot_mapping;
  int T, C, streams, Hkv, max_q_len;
  long long num_slots;
  float inv_scale[2];  // FP8 cache: code = e4m3(y * inv_scale), per stream
  int* status;
};

template <bool kPaged, bool kFp8 = false>
__global__ void __launch_bounds__(kSconvThreads) sconv_kernel(const SconvDev p) {
  pdl_wait();
  pdl_launch_dependents();
  const int C = p.C;
  const int vecs_per_stream = C / kVec;
  const int vec = blockIdx.x * kSconvThreads + threadIdx.x;
  if (vec >= p.streams * vecs_per_stream) return;
  const int which = vec / vecs_per_stream;
  const int c0 = (vec % vecs_per_stream) * kVec;
  const int b = blockIdx.z;
  const int t_begin = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - t_begin;
  if (t_begin < 0 || n < 0 || n > p.max_q_len || t_begin + n > p.T) {
    if (blockIdx.y == 0 && threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  constexpr int kChunk = SconvShape<kPaged>::kChunk;
  const int ts = blockIdx.y * kChunk;
  if (ts >= n) return;
  const int te = min(ts + kChunk, n);

  // selects, not a dynamic index into the parameter arrays (which would copy them to
  // local memory)
  const uint16_t* x = which == 0 ? p.x[0] : p.x[1];
  const float* w = which == 0 ? p.w[0] : p.w[1];
  uint16_t* out = which == 0 ? p.out[0] : p.out[1];
  const float inv_scale = which == 0 ? p.inv_scale[0] : p.inv_scale[1];
  uint16_t* st = p.state + ((size_t)b * p.streams + which) * 3 * C + c0;

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
  // One output row: the four taps over [h0, h1, h2, cur], rounded to bf16, stored.
  auto emit = [&](int tg, const F8& cur) {
    float y[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      float a = tap[i][0] * h0.v[i];
      a = fmaf(tap[i][1], h1.v[i], a);
      a = fmaf(tap[i][2], h2.v[i], a);
      a = fmaf(tap[i][3], cur.v[i], a);
      y[i] = a;
    }
    if (kFp8) {
      // FP8 cache (one byte per channel): e4m3(y / scale), scale folded into inv_scale
      const long long slot = p.slot_mapping[tg];
      if (slot >= p.num_slots) {
        report(p.status, kErrBadBlock);
      } else if (slot >= 0) {
        const long long blk = slot >> 7, off = slot & 127;
        uint2 o8;
        o8.x = pack_e4m3x4(y[0] * inv_scale, y[1] * inv_scale, y[2] * inv_scale, y[3] * inv_scale);
        o8.y = pack_e4m3x4(y[4] * inv_scale, y[5] * inv_scale, y[6] * inv_scale, y[7] * inv_scale);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) +
                                  (((size_t)blk * p.Hkv + head) * 128 + off) * 128 + d0) = o8;
      }
      h0 = h1; h1 = h2; h2 = cur;
      return;
    }
    uint4 o;
    o.x = pack_bf16(y[0], y[1]);
    o.y = pack_bf16(y[2], y[3]);
    o.z = pack_bf16(y[4], y[5]);
    o.w = pack_bf16(y[6], y[7]);
    if (kPaged) {
      const long long slot = p.slot_mapping[tg];
      if (slot >= p.num_slots) {
        report(p.status, kErrBadBlock);
      } else if (slot >= 0) {
        const long long blk = slot >> 7, off = slot & 127;
        *reinterpret_cast<uint4*>(out + (((size_t)blk * p.Hkv + head) * 128 + off) * 128 + d0) = o;
      }
    } else {
      *reinterpret_cast<uint4*>(out + (size_t)tg * C + c0) = o;
    }
    h0 = h1; h1 = h2; h2 = cur;
  };
  // Rows in groups of kBatch: all of a group's loads are issued before its first use,
  // so each thread keeps kBatch 16-byte loads in flight instead of one.
  constexpr int kBatch = SconvShape<kPaged>::kBatch;
  int t = ts;
  for (; t + kBatch <= te; t += kBatch) {
    uint4 raw[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
      raw[u] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + t + u) * C + c0));
#pragma unroll
    for (int u = 0; u < kBatch; ++u) emit(t_begin + t + u, unpack8(raw[u]));
  }
  for (; t < te; ++t)
    emit(t_begin + t, unpack8(__ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + t) * C + c0))));

  if (ts == 0) {
    // new state = last three rows of [old state ; new rows]
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int idx = n - 3 + r;  // index among the new rows
      uint4 v;
      if (idx >= 0) {
        v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + idx) * C + c0));
      } else {
        v = idx == -1 ? old_state[2] : (idx == -2 ? old_state[1] : old_state[0]);
      }
      *reinterpret_cast<uint4*>(st + (size_t)r * C) = v;
    }
  }
}

// Step form of the paged conv, for batches whose sequences all have at most kStepRows new
// tokens (a decode or MTP-verify step): one thread takes every new row of its sequence for
// 8 channels of K or of V.  Such a step moves a few MB and is bound by load latency, so
// each thread issues its loads in two rounds only: the lengths, taps and old state; then
// all its raw rows and their slots at once.  The new state is written from registers.
// Same arithmetic, in the same order, as sconv_kernel: the outputs are bit-identical.
constexpr int kStepRows = 16;

template <bool kFp8>
__global__ void __launch_bounds__(kSconvThreads) sconv_step_kernel(const SconvDev p) {
  pdl_wait();
  pdl_launch_dependents();
  const int C = p.C;
  const int vecs_per_stream = C / kVec;
  const int vec = blockIdx.x * kSconvThreads + threadIdx.x;
  if (vec >= p.streams * vecs_per_stream) return;
  const int which = vec / vecs_per_stream;
  const int c0 = (vec % vecs_per_stream) * kVec;
  const int b = blockIdx.y;
  const uint16_t* x = which == 0 ? p.x[0] : p.x[1];
  const float* w = which == 0 ? p.w[0] : p.w[1];
  uint16_t* out = which == 0 ? p.out[0] : p.out[1];
  const float inv_scale = which == 0 ? p.inv_scale[0] : p.inv_scale[1];
  uint16_t* st = p.state + ((size_t)b * p.streams + which) * 3 * C + c0;

  // first batch of loads: lengths, taps, the three rows before the step
  const int t_begin = p.cu_q_lens[b];
  const int t_end = p.cu_q_lens[b + 1];
  float tap[kVec][4];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    const float4 t4 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(c0 + i) * 4));
    tap[i][0] = t4.x; tap[i][1] = t4.y; tap[i][2] = t4.z; tap[i][3] = t4.w;
  }
  uint4 hist[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) hist[r] = *reinterpret_cast<const uint4*>(st + (size_t)r * C);
  const int n = t_end - t_begin;
  if (t_begin < 0 || n < 0 || n > p.max_q_len || n > kStepRows || t_end > p.T) {
    if (threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  // second batch: every raw row of the step and its slot
  uint4 raw[kStepRows];
  long long slot[kStepRows];
#pragma unroll
  for (int u = 0; u < kStepRows; ++u) {
    if (u < n) {
      raw[u] = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + u) * C + c0));
      slot[u] = p.slot_mapping[t_begin + u];
    } else {
      raw[u] = make_uint4(0, 0, 0, 0);
      slot[u] = -1;
    }
  }
  F8 h0 = unpack8(hist[0]), h1 = unpack8(hist[1]), h2 = unpack8(hist[2]);
  const int head = c0 >> 7, d0 = c0 & 127;
#pragma unroll
  for (int u = 0; u < kStepRows; ++u) {
    if (u >= n) break;
    const F8 cur = unpack8(raw[u]);
    float y[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
      float a = tap[i][0] * h0.v[i];
      a = fmaf(tap[i][1], h1.v[i], a);
      a = fmaf(tap[i][2], h2.v[i], a);
      a = fmaf(tap[i][3], cur.v[i], a);
      y[i] = a;
    }
    if (slot[u] >= p.num_slots) {
      report(p.status, kErrBadBlock);
    } else if (slot[u] >= 0) {
      const long long blk = slot[u] >> 7, off = slot[u] & 127;
      const size_t row = (((size_t)blk * p.Hkv + head) * 128 + off) * 128 + d0;
      if (kFp8) {
        uint2 o8;
        o8.x = pack_e4m3x4(y[0] * inv_scale, y[1] * inv_scale, y[2] * inv_scale, y[3] * inv_scale);
        o8.y = pack_e4m3x4(y[4] * inv_scale, y[5] * inv_scale, y[6] * inv_scale, y[7] * inv_scale);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(out) + row) = o8;
      } else {
        uint4 o;
        o.x = pack_bf16(y[0], y[1]);
        o.y = pack_bf16(y[2], y[3]);
        o.z = pack_bf16(y[4], y[5]);
        o.w = pack_bf16(y[6], y[7]);
        *reinterpret_cast<uint4*>(out + row) = o;
      }
    }
    h0 = h1; h1 = h2; h2 = cur;
  }
  // new state = last three rows of [old state ; new rows], picked by selects (no dynamic
  // register index)
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int idx = n - 3 + r;  // index among the new rows
    uint4 v = idx == -1 ? hist[2] : (idx == -2 ? hist[1] : hist[0]);
#pragma unroll
    for (int u = 0; u < kStepRows; ++u)
      if (u == idx) v = raw[u];
    *reinterpret_cast<uint4*>(st + (size_t)r * C) = v;
  }
}

// State after a speculative step of which only the first accepted[b] new tokens stay:
// the last three rows of [state_before ; first accepted[b] raw rows].  One thread per
// (sequence, stream, 8 channels); it reads all three of its rows before writing any, so
// state_after may be state_before itself.
__global__ void __launch_bounds__(kSconvThreads)
sconv_rollback_kernel(const uint16_t* state_before, const uint16_t* __restrict__ x0,
                      const uint16_t* __restrict__ x1, const int32_t* __restrict__ cu_q_lens,
                      const int32_t* __restrict__ accepted, uint16_t* state_after, int T,
                      int C, int streams, int* __restrict__ status) {
  pdl_wait();
  pdl_launch_dependents();
  const int vecs_per_stream = C / kVec;
  const int vec = blockIdx.x * kSconvThreads + threadIdx.x;
  if (vec >= streams * vecs_per_stream) return;
  const int which = vec / vecs_per_stream;
  const int c0 = (vec % vecs_per_stream) * kVec;
  const int b = blockIdx.y;
  const int t_begin = cu_q_lens[b];
  const int n = cu_q_lens[b + 1] - t_begin;
  const int a = accepted[b];
  if (t_begin < 0 || n < 0 || t_begin + n > T || a < 0 || a > n) {
    if (vec == 0) report(status, kErrBadInput);
    return;
  }
  const uint16_t* x = which == 0 ? x0 : x1;
  const size_t so = ((size_t)b * streams + which) * 3 * C + c0;
  uint4 rows[3];
#pragma unroll
  for (int r = 0; r < 3; ++r) {
    const int idx = a - 3 + r;  // index among the new rows
    rows[r] = idx >= 0 ? __ldg(reinterpret_cast<const uint4*>(x + (size_t)(t_begin + idx) * C + c0))
                       : *reinterpret_cast<const uint4*>(state_before + so + (size_t)(3 + idx) * C);
  }
#pragma unroll
  for (int r = 0; r < 3; ++r) *reinterpret_cast<uint4*>(state_after + so + (size_t)r * C) = rows[r];
}

static dim3 sconv_grid(int streams, int C, int max_q_len, int B, int chunk) {
  const int total_vecs = streams * C / kVec;
  return dim3((total_vecs + kSconvThreads - 1) / kSconvThreads, (max_q_len + chunk - 1) / chunk, B);
}

cudaError_t launch_sconv_kv(const SconvArgs& a, cudaStream_t stream) {
  SconvDev p{};
  p.x[0] = static_cast<const uint16_t*>(a.k_raw);
  p.x[1] = static_cast<const uint16_t*>(a.v_raw);
  p.w[0] = a.w_k;
  p.w[1] = a.w_v;
  p.out[0] = static_cast<uint16_t*>(a.k_cache);
  p.out[1] = static_cast<uint16_t*>(a.v_cache);
  p.state = static_cast<uint16_t*>(a.state);
  p.cu_q_lens = a.cu_q_lens;
  p.slot_mapping = a.slot_mapping;
  p.T = a.T;
  p.C = a.Hkv * 128;
  p.streams = 2;
  p.Hkv = a.Hkv;
  p.max_q_len = a.max_q_len;
  p.num_slots = (long long)a.num_blocks * 128;
  p.status = a.dev_status;
  if (a.max_q_len <= kStepRows) {
    if (a.B == 0 || a.max_q_len == 0) return cudaSuccess;
    const dim3 sg((2 * p.C / kVec + kSconvThreads - 1) / kSconvThreads, a.B);
    if (a.fp8) {
      p.inv_scale[0] = (float)(1.0 / (double)a.k_scale);
      p.inv_scale[1] = (float)(1.0 / (double)a.v_scale);
      return launch_pdl(sconv_step_kernel<true>, sg, dim3(kSconvThreads), 0, stream, p);
    }
    return launch_pdl(sconv_step_kernel<false>, sg, dim3(kSconvThreads), 0, stream, p);
  }
  const dim3 grid = sconv_grid(2, p.C, a.max_q_len, a.B, SconvShape<true>::kChunk);
  if (grid.y == 0 || grid.z == 0) return cudaSuccess;
  if (a.fp8) {
    p.inv_scale[0] = (float)(1.0 / (double)a.k_scale);
    p.inv_scale[1] = (float)(1.0 / (double)a.v_scale);
    return launch_pdl(sconv_kernel<true, true>, grid, dim3(kSconvThreads), 0, stream, p);
  }
  return launch_pdl(sconv_kernel<true>, grid, dim3(kSconvThreads), 0, stream, p);
}

cudaError_t launch_sconv_dense(const SconvDenseArgs& a, cudaStream_t stream) {
  SconvDev p{};
  p.x[0] = p.x[1] = static_cast<const uint16_t*>(a.x);
  p.w[0] = p.w[1] = a.w;
  p.out[0] = p.out[1] = static_cast<uint16_t*>(a.y);
  p.state = static_cast<uint16_t*>(a.state);
  p.cu_q_lens = a.cu_q_lens;
  p.T = a.T;
  p.C = a.C;
  p.streams = 1;
  p.max_q_len = a.max_q_len;
  p.status = a.dev_status;
  const dim3 grid = sconv_grid(1, a.C, a.max_q_len, a.B, SconvShape<false>::kChunk);
  if (grid.y == 0 || grid.z == 0) return cudaSuccess;
  return launch_pdl(sconv_kernel<false>, grid, dim3(kSconvThreads), 0, stream, p);
}

cudaError_t launch_sconv_rollback(const SconvRollbackArgs& a, cudaStream_t stream) {
  const int total_vecs = a.streams * a.C / kVec;
  const dim3 grid((total_vecs + kSconvThreads - 1) / kSconvThreads, a.B);
  if (grid.y == 0) return cudaSuccess;
  return launch_pdl(sconv_rollback_kernel, grid, dim3(kSconvThreads), 0, stream,
                    static_cast<const uint16_t*>(a.state_before),
                    static_cast<const uint16_t*>(a.x0),
                    static_cast<const uint16_t*>(a.x1 ? a.x1 : a.x0), a.cu_q_lens, a.accepted,
                    static_cast<uint16_t*>(a.state_after), a.T, a.C, a.streams, a.dev_status);
}

}  // namespace ink
