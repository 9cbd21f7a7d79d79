// Split-KV paged decode for relative-bias GQA with up to 9 new tokens per sequence
// (vLLM Day-0 Inkling blog: "Model Architecture / MTP" for the 9-token verify step,
// "FA4 with sheared bias" for the per-configuration num_splits).
//
// One CTA = (split, KV head, sequence).  The n_b new tokens x G query heads that share
// the KV head are packed as rows r = t*G + g of one 128-row tile (72 rows for 9 tokens
// and G = 8), so each K/V page is read from HBM once per KV head.  The packed Q lives in
// tensor memory (64 columns of bf16 pairs) and both contractions run on the tensor core:
// S = Q K^T with Q from TMEM (TS form), O += P V with P from TMEM.
//   warps 0-7   softmax: the pair w, w + 4 shares packed rows 32 (w % 4) .. + 31 (their
//               TMEM lanes) and splits their 128 columns, trading partial maxima once
//               per page; thread (r, half) does bias, mask, online softmax, P and the
//               epilogue for its 64 columns of row r.
//   warp 8      TMA producer: K/V pages of the split (three-stage ring of 64 KB).
//   warp 9      MMA issuer; S is double-buffered so S(i+1) overlaps softmax(i).  Page i's
//               "P ready" barrier is p_full[i & 1]: S(i+1) is issued before P(i) is
//               consumed, so a fast warp may finish page i+1 while a slow one is still on
//               page i, and one barrier for both pages would complete too early.  Over a
//               bf16 cache each product's eight k-steps are one elected asm block.
//   warp 10     bias stager: cp.async each page's bias slices (G heads) into a ring of
//               its own, whose slots the softmax frees as soon as it has added the bias,
//               so the slices of later pages load while the current one is processed.
//   warp 11     (the fused-conv call only) the sconv of the step's new K/V rows that fall
//               in the CTA's pages, for its KV head's 128 channels, written into the
//               cache before the producer loads those pages.
//   warps 12-19 (FP8 cache only) converters: E4M3 pages widened to f16 for the MMAs.
// TMEM columns: Q [0,64), S0 [128,256), S1 [256,384), O [384,512).
// A sequence whose key range fits one split writes its output directly; otherwise every
// split writes (m, l, unnormalised O) to the workspace and combine_kernel merges them:
//   O = sum_s e^(m_s - M) O_s / sum_s e^(m_s - M) l_s,  M = max_s m_s.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ink {
namespace decode {

constexpr int kStages = 3;
// Warps 0-7 softmax (the pair w, w+4 shares TMEM lanes 32(w%4).. and splits the 128
// columns of those rows), 8 TMA producer, 9 MMA issuer, 10 bias stager, 11 the fused
// conv (idle in the plain decode).
// Register split (setmaxnreg): built for 168 registers a thread at launch (65536 / 384),
// the two softmax warpgroups grow to 216 and the third gives back down to 64:
// 256*216 + 128*64 = 63488 <= 384*168.  The host refuses the launch unless the built
// count is 168.
constexpr int kThreads = 384;
constexpr int kLaunchRegs = 168, kSoftmaxRegs = 216, kOtherRegs = 64;
static_assert(256 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpBias = 10, kWarpConvRows = 11, kWarpConv = 12;
// FP8 cache: two more warpgroups, warps 12-15 widen the E4M3 K pages and 16-19 the V
// pages (32 rows each).  Widening a page with two warps took 0.8 us and, with one f16
// page per tensor, set the page period (a clock64 trace: widen V(j) -> PV(j) -> widen
// V(j+1)); four halve it.  Built for 96 registers a thread at launch (65536 / 640,
// rounded down to 8): softmax 152, the rest 56: 256*152 + 384*56 = 60416 <= 640*96.
constexpr int kThreadsF8 = 640;
constexpr int kF8LaunchRegs = 96, kF8SoftmaxRegs = 152, kF8OtherRegs = 56;
constexpr int kConvWarps = 4;  // per tensor
static_assert(256 * kF8SoftmaxRegs + (kThreadsF8 - 256) * kF8OtherRegs <= kThreadsF8 * kF8LaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kMaxG = 16;
// floats per staged head (>= 127 + 9 + 3, a multiple of 4 so that each head's slot is
// 16-byte aligned); 164 = 4 (mod 32), so the G heads x 4 tokens of a warp
// (lane = t*G + g) hit distinct banks when they read column c
constexpr int kBiasStride = 164;
constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);
constexpr uint32_t kIdescQK16 = idesc_f16(128, 128, false, false);
constexpr uint32_t kIdescPV16 = idesc_f16(128, 128, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 5.545177444479562f;  // 8 ln 2: rescale O past 256x growth
constexpr uint32_t kColQ = 0, kColS0 = 128, kColO = 384;

struct __align__(1024) Smem {
  uint8_t k[kStages][2][16384];
  uint8_t v[kStages][2][16384];
  float bias[kStages][kMaxG * kBiasStride];  // raw table values, staged per page by the bias warp
  // k_full / v_full: kStages bf16 stages or kStagesF8 (4) E4M3 stages
  uint64_t k_full[4], v_full[4], kv_empty[kStages], b_full[kStages], b_empty[kStages];
  uint64_t q_ready, s_full[2], p_full[2], pv_done, o_full, drain, conv_done;
  // the two column halves of a row trade partial maxima (per page parity), and at the
  // end their sums (in the slot of the parity after the last page's)
  uint64_t x_full[4][2], l_full;  // x_full[q]: warps q and q + 4 (the two halves of rows 32q..)
  float xm[2][2][128];
  // FP8 cache only: the converters' hand-offs (see convert_rows)
  uint64_t k8_empty[4], v8_empty[4], kh_full[2], kh_empty[2], vh_full[2], vh_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

// 227 KB per CTA, with 1 KB of slack to align the dynamic buffer to 1024 bytes
static_assert(sizeof(Smem) + 1024 <= 232448, "decode shared memory exceeds 227 KB");

struct Params {
  const uint16_t* q;
  const int32_t* block_table;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const float* bias;
  void* out;
  float* lse;
  float* part_o;   // [B][Hkv][S][rmax][128]
  float* part_ml;  // [B][Hkv][S][rmax][2]
  int* status;
  int max_blocks, R, window, out_dtype;
  float v_scale;  // FP8 cache: V = code * v_scale, applied to O (1 for a bf16 cache)
  int B, T, Hq, Hkv, G, max_q_len, rmax, num_splits, pages_per_split;
  long long num_blocks;
  float scale;
  // the step's conv fused into the prologue (conv_x[0] == nullptr: conv done separately)
  const uint16_t* conv_x[2];  // raw K, V rows of the new tokens [T][Hkv*128]
  const float* conv_w[2];     // taps [Hkv*128][4]
  uint16_t* conv_state;       // [B][2][3][Hkv*128], in/out
  uint16_t* cache_w[2];       // the bf16 caches, written at the new rows' slots
};

// Key pages a sequence's decode rows can see: [kt_lo, kt_hi].
__device__ __forceinline__ void page_range(int L, int n, int window, int& kt_lo, int& kt_hi) {
  const int k_lo = window > 0 ? max(0, L - n - window + 1) : 0;
  kt_lo = k_lo >> 7;
  kt_hi = (L - 1) >> 7;
}

// Packed rows.  When G divides 32, every warp holds tokens of one parity: the even tokens
// fill the first ceil(ceil(n/2) G / 32) warps and the odd tokens the next ones (with G = 8
// and 9 tokens: 0 2 4 6 | 1 3 5 7 | 8), so that the bias pairs of a warp's threads share
// one alignment (see the softmax).  Otherwise row r is token r / G, head r % G.  Rows
// past a parity's tokens are padding: they take its last token and their lane's head.
__host__ __device__ __forceinline__ int packed_warps(int n, int G) {
  if (32 % G != 0) return (n * G + 31) / 32;
  return ((n + 1) / 2 * G + 31) / 32 + (n / 2 * G + 31) / 32;
}
__device__ __forceinline__ bool packed_row(int r, int n, int G, int& t, int& g) {
  if (32 % G != 0) {
    t = min(r / G, n - 1);
    g = r % G;
    return r < n * G;
  }
  const int ne = (n + 1) / 2, we = (ne * G + 31) / 32;
  const int w = r >> 5, par = w >= we ? 1 : 0;
  const int k = ((w - par * we) * 32 + (r & 31)) / G;
  const int cnt = par ? n / 2 : ne;
  g = r % G;
  t = 2 * min(k, cnt - 1) + par;
  return k < cnt;
}

__device__ __forceinline__ uint64_t desc_k(const uint8_t (*atoms)[16384], int ks) {
  return sdesc_sw128(smem_u32(atoms[ks >> 2]) + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_v(const uint8_t (*atoms)[16384], int ks) {
  return sdesc_sw128(smem_u32(atoms[0]) + ks * 2048, 16384, 1024);
}

// FP8 cache layout in shared memory, carved out of the bf16 K/V ring (192 KB = twelve
// 16 KB slots): E4M3 pages as the TMA writes them (one 128-byte-swizzled box of 128 slots
// x 128 bytes), three stages each for K (slots 0-2) and V (slots 3-5), and f16 pages for
// K (s.v[0], s.v[1] when two) and V (s.v[2]) in the layout of the bf16 ring, which the
// MMAs read.
constexpr int kStagesF8 = 3;
constexpr int kF16BufsK = 1, kF16BufsV = 1;
static_assert(kStagesF8 <= 4 &&
                  2 * kStagesF8 * 16384 + (kF16BufsK + kF16BufsV) * 32768 <= 2 * kStages * 32768,
              "E4M3 stages and f16 pages must fit in the bf16 K/V ring");
__device__ __forceinline__ uint8_t* f8_page(Smem& s, int which, int st) {
  return &s.k[0][0][0] + (which * kStagesF8 + st) * 16384;
}
__device__ __forceinline__ uint8_t (*f16_page(Smem& s, int which, int buf))[16384] {
  return which == 0 ? s.v[buf] : s.v[2];
}

// E4M3 page (16 KB, rows of 128 bytes, 16-byte chunk c of row r stored at chunk c ^ (r%8))
// -> f16 page (two 64-wide d halves of 128-byte rows, same swizzle), exactly: every E4M3
// value is an f16 value.  Rows r >= r0 (slots past the end of the sequence) become 0.
// One warp converts 128 / kConvWarps rows from row_base: lane l takes rows row_base + l,
// row_base + l + 32, ...
__device__ __forceinline__ void convert_rows(const uint8_t* src, uint8_t (*dst)[16384], int r0,
                                             int row_base, int lane) {
#pragma unroll
  for (int rr = 0; rr < 4 / kConvWarps; ++rr) {
    const int r = row_base + lane + 32 * rr;
    const int sw = r & 7;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 in = make_uint4(0, 0, 0, 0);
      if (r < r0) in = *reinterpret_cast<const uint4*>(src + r * 128 + ((c ^ sw) << 4));
      const uint32_t w[4] = {in.x, in.y, in.z, in.w};
      uint32_t h[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        h[2 * j] = e4m3x2_to_f16x2((uint16_t)(w[j] & 0xffffu));
        h[2 * j + 1] = e4m3x2_to_f16x2((uint16_t)(w[j] >> 16));
      }
      uint8_t* half = dst[c >> 2] + r * 128;
      const int c0 = (c & 3) * 2;
      *reinterpret_cast<uint4*>(half + ((c0 ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(half + (((c0 + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
}

template <bool kFp8>
__global__ void __launch_bounds__(kFp8 ? kThreadsF8 : kThreads, 1)
decode_kernel(const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = warp_id(), lane = lane_id();
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  constexpr int NS = kFp8 ? kStagesF8 : kStages;  // K/V load stages
  pdl_wait();
  const int t_seq0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - t_seq0;
  if (n == 0) return;
  const int L = p.seq_lens[b];
  if (n < 0 || n > p.max_q_len || n > L || L > p.max_blocks * 128) {
    if (split == 0 && kvh == 0 && threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  int kt_lo, kt_hi;
  page_range(L, n, p.window, kt_lo, kt_hi);
  const int npages_seq = kt_hi - kt_lo + 1;
  const int nsplit_b = (npages_seq + p.pages_per_split - 1) / p.pages_per_split;
  if (split >= nsplit_b) return;
  if (nsplit_b > p.num_splits) {  // host-side max_seq_len was too small
    if (split == 0 && threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  const int pg0 = kt_lo + split * p.pages_per_split;
  const int np = min(p.pages_per_split, kt_hi + 1 - pg0);
  // fused conv: the new rows t whose position L - n + t lies in this CTA's pages
  const bool conv = !kFp8 && p.conv_x[0] != nullptr;
  const int conv_t_lo = max(0, pg0 * 128 - (L - n));
  const int conv_t_hi = min(n, (pg0 + np) * 128 - (L - n));
  const bool conv_here = conv && conv_t_lo < conv_t_hi;
  const int conv_page0 = (L - n + conv_t_lo) >> 7;  // the first page holding a new row
  // softmax warps that own packed rows; the others sit out (their TMEM lanes hold rows
  // nobody reads, and the MMA rows are independent of each other)
  const int nwarps = packed_warps(n, p.G);
  const int nact = nwarps * 32;
  const int32_t* table = p.block_table + (size_t)b * p.max_blocks;

  // Page ids are checked by whoever uses them first, before the use: the producer before
  // each page's loads (ids read three pages ahead), the fused conv before its writes.  A
  // bad id is reported (first error wins) and raises the abort flag, which stops the other
  // roles; no access is made through it.
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
      mbar_init(&s.b_full[i], 32);
      mbar_init(&s.b_empty[i], 2 * nact);
    }
    mbar_init(&s.q_ready, 2 * nact);
    for (int q = 0; q < 4; ++q) {
      mbar_init(&s.x_full[q][0], 64);
      mbar_init(&s.x_full[q][1], 64);
    }
    mbar_init(&s.l_full, 2 * nact);
    mbar_init(&s.s_full[0], 1);
    mbar_init(&s.s_full[1], 1);
    mbar_init(&s.p_full[0], 2 * nact);
    mbar_init(&s.p_full[1], 2 * nact);
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.drain, 1);
    mbar_init(&s.conv_done, 1);
    if (kFp8) {
      for (int i = 0; i < kStagesF8; ++i) {
        if (i >= kStages) {  // the stages past the bf16 ring's
          mbar_init(&s.k_full[i], 1);
          mbar_init(&s.v_full[i], 1);
        }
        mbar_init(&s.k8_empty[i], kConvWarps);
        mbar_init(&s.v8_empty[i], kConvWarps);
      }
      for (int i = 0; i < 2; ++i) {
        mbar_init(&s.kh_full[i], kConvWarps);
        mbar_init(&s.kh_empty[i], 1);
        mbar_init(&s.vh_full[i], kConvWarps);
        mbar_init(&s.vh_empty[i], 1);
      }
    }
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kFp8 ? kF8OtherRegs : kOtherRegs));
   if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer ---
    // Lane 0 issues the K/V page loads, up to kStages pages ahead of the softmax.
    const uint64_t pol = l2_policy_evict_first();
    if (lane == 0) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      auto page_id = [&](int i) -> int32_t { return i < np ? table[pg0 + i] : 0; };
      int32_t id1 = page_id(0), id2 = page_id(1), id3 = page_id(2);
      for (int i = 0; i < np; ++i) {
        const int st = i % NS;
        const int32_t blk = id1;
        id1 = id2;
        id2 = id3;
        id3 = page_id(i + 3);
        if (blk < 0 || (long long)blk >= p.num_blocks) {
          report(p.status, kErrBadBlock);
          __threadfence();  // the report lands before any role that sees the flag reports
          s.abort_flag = 1;
          break;
        }
        const int page = blk * p.Hkv + kvh;
        if (kFp8) {
          // one 16 KB E4M3 box per K and V page; a stage is free once converted
          const uint32_t eph = ((i / NS) - 1) & 1;
          if (i >= NS && !mbar_wait(&s.k8_empty[st], eph, abort_flag, p.status)) {
            report(p.status, kErrTimeout);
            s.abort_flag = 1;
            break;
          }
          mbar_arrive_expect_tx(&s.k_full[st], 16384u);
          tma_load_3d_hint(f8_page(s, 0, st), &map_k, &s.k_full[st], 0, 0, page, pol);
          if (i >= NS && !mbar_wait(&s.v8_empty[st], eph, abort_flag, p.status)) {
            report(p.status, kErrTimeout);
            s.abort_flag = 1;
            issued = i;  // this page's K is in flight too: let it land
            volatile int never = 0;
            mbar_wait(&s.k_full[st], (i / NS) & 1, &never);
            break;
          }
          mbar_arrive_expect_tx(&s.v_full[st], 16384u);
          tma_load_3d_hint(f8_page(s, 1, st), &map_v, &s.v_full[st], 0, 0, page, pol);
          issued = i + 1;
          continue;
        }
        if (i >= kStages &&
            !mbar_wait(&s.kv_empty[st], ((i / kStages) - 1) & 1, abort_flag, p.status)) {
          report(p.status, kErrTimeout);
          s.abort_flag = 1;
          break;
        }
        // the pages holding new rows are read once the fused conv has written them
        if (conv_here && pg0 + i == conv_page0 &&
            !mbar_wait(&s.conv_done, 0, abort_flag, p.status)) {
          report(p.status, kErrTimeout);
          s.abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&s.k_full[st], 32768u);
        tma_load_3d_hint(s.k[st][0], &map_k, &s.k_full[st], 0, 0, page, pol);
        tma_load_3d_hint(s.k[st][1], &map_k, &s.k_full[st], 64, 0, page, pol);
        mbar_arrive_expect_tx(&s.v_full[st], 32768u);
        tma_load_3d_hint(s.v[st][0], &map_v, &s.v_full[st], 0, 0, page, pol);
        tma_load_3d_hint(s.v[st][1], &map_v, &s.v_full[st], 64, 0, page, pol);
        issued = i + 1;
      }
      if (*abort_flag) {
        // let the copies already in flight land before the CTA goes away
        for (int i = max(0, issued - NS); i < issued; ++i) {
          const int st = i % NS;
          const uint32_t ph = (i / NS) & 1;
          volatile int never = 0;
          mbar_wait(&s.k_full[st], ph, &never);
          mbar_wait(&s.v_full[st], ph, &never);
        }
      }
    }
  } else if (kFp8 && warp >= kWarpConv) {
    // ------------------------------------------------------------ FP8 converters ---
    // Warps 12-15 widen K pages, 16-19 V pages, 32 rows each: page j's K goes to its f16
    // page once QK has read the page's previous occupant, its V once PV has.
    const int which = (warp - kWarpConv) / kConvWarps;
    const int row_base = ((warp - kWarpConv) % kConvWarps) * (128 / kConvWarps);
    const int r_end = L - pg0 * 128;  // rows of page j at or past r_end - 128 j are empty
    uint64_t* full8 = which == 0 ? s.k_full : s.v_full;
    uint64_t* empty8 = which == 0 ? s.k8_empty : s.v8_empty;
    uint64_t* full_h = which == 0 ? s.kh_full : s.vh_full;
    uint64_t* empty_h = which == 0 ? s.kh_empty : s.vh_empty;
    bool ok = true;
    for (int j = 0; ok && j < np; ++j) {
      const int nb = which == 0 ? kF16BufsK : kF16BufsV;
      const int st = j % NS, hb = j % nb;
      ok = mbar_wait(&full8[st], (j / NS) & 1, abort_flag, p.status) &&
           (j < nb || mbar_wait(&empty_h[hb], ((j / nb) - 1) & 1, abort_flag, p.status));
      if (!ok) break;
      convert_rows(f8_page(s, which, st), f16_page(s, which, hb), min(128, r_end - 128 * j),
                   row_base, lane);
      if (lane == 0) {
        mbar_arrive(&full_h[hb]);
        mbar_arrive(&empty8[st]);
      }
    }
    if (!ok) {
      report(p.status, kErrTimeout);
      s.abort_flag = 1;
    }
  } else if (!kFp8 && warp == kWarpConvRows) {
    // ------------------------------------------------------------ fused conv ---
    // Lane l: channels 4l .. 4l+3 of this KV head, K then V, over the new rows up to the
    // CTA's last one (earlier rows only feed the window of three).  The arithmetic and
    // its order are those of the separate step conv, so the cache rows are bit-identical.
    // The sequence's only CTA (one split) also writes the new state; with more splits the
    // merge kernel does, once no CTA can still be reading the old one.
    if (conv_here) {
      const int C = p.Hkv * 128;
      const int c = kvh * 128 + lane * 4;
      auto bf = [](uint32_t w, int hi) { return __uint_as_float(hi ? (w & 0xffff0000u) : (w << 16)); };
      for (int which = 0; which < 2; ++which) {
        const uint16_t* x = p.conv_x[which];
        const float* w = p.conv_w[which];
        uint16_t* st = p.conv_state + ((size_t)b * 2 + which) * 3 * C + c;
        float tap[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t4 = __ldg(reinterpret_cast<const float4*>(w + (size_t)(c + i) * 4));
          tap[i][0] = t4.x; tap[i][1] = t4.y; tap[i][2] = t4.z; tap[i][3] = t4.w;
        }
        uint2 h0 = *reinterpret_cast<const uint2*>(st);
        uint2 h1 = *reinterpret_cast<const uint2*>(st + C);
        uint2 h2 = *reinterpret_cast<const uint2*>(st + 2 * C);
        for (int t = 0; t < conv_t_hi; ++t) {
          const uint2 cur = __ldg(reinterpret_cast<const uint2*>(x + (size_t)(t_seq0 + t) * C + c));
          if (t >= conv_t_lo) {
            float y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t w0 = i < 2 ? h0.x : h0.y, w1 = i < 2 ? h1.x : h1.y;
              const uint32_t w2 = i < 2 ? h2.x : h2.y, w3 = i < 2 ? cur.x : cur.y;
              float a = tap[i][0] * bf(w0, i & 1);
              a = fmaf(tap[i][1], bf(w1, i & 1), a);
              a = fmaf(tap[i][2], bf(w2, i & 1), a);
              a = fmaf(tap[i][3], bf(w3, i & 1), a);
              y[i] = a;
            }
            const int pos = L - n + t;
            const int32_t blk = table[pos >> 7];
            if (blk < 0 || (long long)blk >= p.num_blocks) {
              report(p.status, kErrBadBlock);  // no write; the producer stops at this page
            } else {
              uint16_t* dst = p.cache_w[which] +
                              (((size_t)blk * p.Hkv + kvh) * 128 + (pos & 127)) * 128 + lane * 4;
              *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]));
            }
          }
          h0 = h1;
          h1 = h2;
          h2 = cur;
        }
        if (nsplit_b == 1) {  // conv_t_hi == n here: h0..h2 are the last three rows
          *reinterpret_cast<uint2*>(st) = h0;
          *reinterpret_cast<uint2*>(st + C) = h1;
          *reinterpret_cast<uint2*>(st + 2 * C) = h2;
        }
      }
      // the rows are read next by this CTA's TMA loads (the async proxy)
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&s.conv_done);
    }
  } else if (warp == kWarpBias) {
    // ------------------------------------------------------------ bias stager ---
    // Slot m of head g's slice holds b[kvh*G + g][a0 + m], a0 = the page's smallest
    // distance rounded down to a multiple of 4, so the slice is one aligned run of the
    // table: lane 0 fetches it with one bulk copy per head.  Slices that need clamping
    // (distances below 0 or past R-1) are staged by all lanes with 4-byte cp.async
    // copies of the clamped entries.  Both ways 32 arrivals complete b_full[slot]; a
    // slot is reused once every softmax thread has added the slice it held (b_empty).
    const int R = p.R;
    const bool bulk_ok = ((reinterpret_cast<uintptr_t>(p.bias) & 15) == 0) && (R & 3) == 0;
    int staged = 0;
    for (int i = 0; i < np; ++i) {
      const int st = i % kStages;
      int ok = 1;
      if (lane == 0 && i >= kStages)
        ok = mbar_wait(&s.b_empty[st], ((i / kStages) - 1) & 1, abort_flag, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) {
          report(p.status, kErrTimeout);
          s.abort_flag = 1;
        }
        break;
      }
      staged = i + 1;
      const int k0 = (pg0 + i) * 128;
      const int dmax = (L - 1) - k0;    // largest distance in the page
      const int dmin = (L - n) - k0 - 127;  // smallest, over all rows
      const int a0 = dmin & ~3;
      const int cnt = (dmax - a0 + 4) & ~3;  // <= 127 + 9 + 3, rounded up to 4: fits the stride
      if (dmin < R - 1) {                    // not every distance clamped
        if (bulk_ok && a0 >= 0 && a0 + cnt <= R) {
          if (lane == 0) {
            mbar_arrive_expect_tx(&s.b_full[st], (uint32_t)(p.G * cnt * 4));
            for (int gg = 0; gg < p.G; ++gg)
              bulk_g2s(s.bias[st] + gg * kBiasStride, p.bias + (size_t)(kvh * p.G + gg) * R + a0,
                       (uint32_t)(cnt * 4), &s.b_full[st]);
          } else {
            mbar_arrive(&s.b_full[st]);
          }
          continue;
        }
        for (int gg = 0; gg < p.G; ++gg) {
          float* dst = s.bias[st] + gg * kBiasStride;
          const float* src = p.bias + (size_t)(kvh * p.G + gg) * R;
          for (int m = lane; m < cnt; m += 32) {
            int d = a0 + m;
            d = d < 0 ? 0 : (d > R - 1 ? R - 1 : d);
            cp_async_4(dst + m, src + d);
          }
        }
      }
      cp_async_mbar_arrive(&s.b_full[st]);
    }
    // let outstanding copies land before the CTA can exit (bulk copies: their b_full)
    if (lane == 0) {
      for (int i = max(0, staged - kStages); i < staged; ++i) {
        volatile int never = 0;
        mbar_wait(&s.b_full[i % kStages], (i / kStages) & 1, &never);
      }
    }
    __syncwarp();
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer ---
    // FP8: K and V come from the converters' f16 pages (f16_page), f16 MMAs
    constexpr uint32_t idQK = kFp8 ? kIdescQK16 : kIdescQK;
    constexpr uint32_t idPV = kFp8 ? kIdescPV16 : kIdescPV;
    // Over a bf16 cache the whole warp runs this loop converged: the products are issued
    // as elected eight-MMA blocks (their commits elect the same lane), and each wait's
    // outcome is made warp-uniform before it is acted on.  Over an FP8 cache the kernel
    // is bound by its converter warps; there lane 0 issues single-MMA statements and
    // commits, the warp meeting at a __syncwarp after each (that form measured 2-4%
    // faster than the elected blocks on the long FP8 decodes).
    auto qk = [&](uint32_t dS, const uint8_t (*kp)[16384]) {
      if constexpr (kFp8) {
        if (lane == 0) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_ts(dS, tmem + kColQ + ks * 8, desc_k(kp, ks), idQK, ks > 0);
        }
        __syncwarp();
      } else {
        mma8_ts_kmajor<idQK>(dS, tmem + kColQ, desc_k(kp, 0), 0);
      }
    };
    auto pv = [&](uint32_t aP, const uint8_t (*vp)[16384], bool acc) {
      if constexpr (kFp8) {
        if (lane == 0) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            umma_ts(tmem + kColO, aP + ks * 8, desc_v(vp, ks), idPV, (acc || ks > 0));
        }
        __syncwarp();
      } else {
        mma8_ts_mnmajor<idPV>(tmem + kColO, aP, desc_v(vp, 0), acc ? 1u : 0u);
      }
    };
    auto commit = [&](uint64_t* bar) {
      if constexpr (kFp8) {
        if (lane == 0) umma_commit(bar);
        __syncwarp();
      } else {
        umma_commit_elected(bar);
      }
    };
    bool ok = mbar_wait(&s.q_ready, 0, abort_flag, p.status) &&
              (kFp8 ? mbar_wait(&s.kh_full[0], 0, abort_flag, p.status)
                    : mbar_wait(&s.k_full[0], 0, abort_flag, p.status));
    if constexpr (!kFp8) ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    if (ok) {
      tc_fence_after();
      const uint8_t (*kp)[16384] = kFp8 ? f16_page(s, 0, 0) : s.k[0];
      qk(tmem + kColS0, kp);
      commit(&s.s_full[0]);
      if (kFp8) commit(&s.kh_empty[0]);
      issued_any = true;
    }
    for (int i = 0; ok && i < np; ++i) {
      const int st = i % kStages;
      if (i + 1 < np) {
        const int st1 = (i + 1) % kStages;
        ok = kFp8 ? mbar_wait(&s.kh_full[(i + 1) % kF16BufsK], ((i + 1) / kF16BufsK) & 1, abort_flag,
                              p.status)
                  : mbar_wait(&s.k_full[st1], ((i + 1) / kStages) & 1, abort_flag, p.status);
        if constexpr (!kFp8) ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dS = tmem + kColS0 + ((i + 1) & 1) * 128;
        const uint8_t (*kp)[16384] = kFp8 ? f16_page(s, 0, (i + 1) % kF16BufsK) : s.k[st1];
        qk(dS, kp);
        commit(&s.s_full[(i + 1) & 1]);
        if (kFp8) commit(&s.kh_empty[(i + 1) % kF16BufsK]);
      }
      ok = mbar_wait(&s.p_full[i & 1], (i >> 1) & 1, abort_flag, p.status) &&
           (kFp8 ? mbar_wait(&s.vh_full[0], i & 1, abort_flag, p.status)
                 : mbar_wait(&s.v_full[st], (i / kStages) & 1, abort_flag, p.status));
      if constexpr (!kFp8) ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int kt = pg0 + i;
      if (!kFp8 && (kt + 1) * 128 > L) {  // (the converter zeroes the f16 page's tail)
        // slots past the end of the sequence: P is 0 there but the stale V could be NaN
        const int r0 = L - kt * 128;
        const int chunks = (128 - r0) * 8;
        for (int c = lane; c < 2 * chunks; c += 32) {
          const int half = c / chunks, cc = c % chunks;
          *reinterpret_cast<uint4*>(s.v[st][half] + (size_t)(r0 + cc / 8) * 128 + (cc % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc_fence_after();
      const uint32_t aP = tmem + kColS0 + (i & 1) * 128;
      const uint8_t (*vp)[16384] = kFp8 ? f16_page(s, 1, 0) : s.v[st];
      pv(aP, vp, i > 0);
      commit(kFp8 ? &s.vh_empty[0] : &s.kv_empty[st]);
      commit(&s.pv_done);
    }
    if (ok) {
      commit(&s.o_full);
    } else {
      report(p.status, kErrTimeout);
      s.abort_flag = 1;
      if (issued_any) {
        commit(&s.drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&s.drain, 0, &never);
      }
    }
    __syncwarp();
   }
  } else {
   asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kFp8 ? kF8SoftmaxRegs : kSoftmaxRegs));
   if ((warp & 3) < nwarps) {
    // ------------------------------------------------------------ softmax group ---
    // Thread (r, hf): packed row r = TMEM lane, columns 64 hf .. 64 hf + 63 of S, P, O.
    // The two halves of a row trade their partial maxima through shared memory (an
    // mbarrier per warp pair and page parity: the pairs do not wait for one another), so
    // both use the same running max; each keeps its own
    // partial sum, and the sums meet once at the end.
    const int r = (warp & 3) * 32 + lane;
    const int hf = warp >> 2, c0 = hf * 64;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // A padding row takes the head of its lane and the last token of its warp's parity:
    // its bias reads then fall on the words of valid rows (shared, not conflicting), so a
    // warp's lanes hit distinct banks.  Its Q is zero and nothing of it is stored.
    int t, g;
    const bool valid = packed_row(r, n, p.G, t, g);
    const int h = kvh * p.G + g;

    // packed Q rows into TMEM columns [0, 64): this thread's half of the d range
    {
      uint32_t qr[32];
      if (valid) {
        const uint4* src =
            reinterpret_cast<const uint4*>(p.q + ((size_t)(t_seq0 + t) * p.Hq + h) * 128 + c0);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 w = __ldg(src + j);
          qr[4 * j] = w.x; qr[4 * j + 1] = w.y; qr[4 * j + 2] = w.z; qr[4 * j + 3] = w.w;
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) qr[j] = 0u;
      }
      if (kFp8) {  // the f16 MMAs take Q as f16 (exact for |q| < 65504)
#pragma unroll
        for (int j = 0; j < 32; ++j)
          qr[j] = pack_f16(__uint_as_float(qr[j] << 16), __uint_as_float(qr[j] & 0xffff0000u));
      }
      tmem_st32(tmem + lane_base + kColQ + hf * 32, qr);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.q_ready);
    }

    const float* brow = p.bias + (size_t)h * p.R;
    const int R = p.R, W = p.window;
    const float bconst = __ldg(brow + R - 1);
    const int pq = L - n + t;  // position of this row's token
    float m = -INFINITY;
    float2 l2 = make_float2(0.f, 0.f);
    const float2 sc2 = make_float2(p.scale, p.scale);
    const float2 bc2 = make_float2(bconst, bconst);
    const float2 lg2 = make_float2(kLog2e, kLog2e);
    bool ok = true;
    for (int i = 0; i < np; ++i) {
      const int k0 = (pg0 + i) * 128;
      const int dmin = (L - n) - k0 - 127;  // smallest distance in the page over all rows
      const int dmax = (L - 1) - k0;
      const bool clamped = dmin >= R - 1;
      const bool masked = dmin < 0 || (W > 0 && dmax > W - 1);
      const float* bias_buf = s.bias[i % kStages];
      if (!clamped && !mbar_wait(&s.b_full[i % kStages], (i / kStages) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (!mbar_wait(&s.s_full[i & 1], (i >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + kColS0 + (i & 1) * 128;
      uint32_t sr[64];  // this half of the S row, then its packed P pairs
      tmem_ld32(tS + c0, sr);
      tmem_ld32(tS + c0 + 32, sr + 32);
      tmem_wait_ld();
      reg_fence<64>(sr);
      float2 x[32];  // logits in natural units, pairs of columns
      if (clamped) {
#pragma unroll
        for (int k = 0; k < 32; ++k)
          x[k] = __ffma2_rn(make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1])),
                            sc2, bc2);
      } else if (32 % p.G == 0) {
        // pairs of columns by 8-byte loads.  The slot of column c0 is `base`; its parity
        // is that of the token, so it is the same for the whole warp (packed_row).  base
        // odd: the pair (c0 + 2k, c0 + 2k + 1) is the aligned word at base - 1 - 2k, higher
        // column first.  base even: the aligned words at base - 2j hold (c0 + 2j,
        // c0 + 2j - 1), so pair k takes the first half of word k and the second of word
        // k + 1 (33 loads).  Slices 164 words (4 mod 32) apart put the 8 heads of a token
        // on distinct bank pairs and token t + 2 two words over: a half-warp's 16 loads
        // are conflict-free.
        const int base = (pq - k0 - (dmin & ~3)) - c0;
        const float* bb = bias_buf + g * kBiasStride + base;
        if (base & 1) {
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float2 w2 = *reinterpret_cast<const float2*>(bb - 1 - 2 * k);
            x[k] = __ffma2_rn(make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1])),
                              sc2, make_float2(w2.y, w2.x));
          }
        } else {
          float2 prev = *reinterpret_cast<const float2*>(bb);
#pragma unroll
          for (int k = 0; k < 32; ++k) {
            const float2 nxt = *reinterpret_cast<const float2*>(bb - 2 - 2 * k);
            x[k] = __ffma2_rn(make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1])),
                              sc2, make_float2(prev.x, nxt.y));
            prev = nxt;
          }
        }
      } else {
        // slot of column c: distance pq - k0 - c minus the slice start a0
        const float* bp = bias_buf + g * kBiasStride + (pq - k0 - (dmin & ~3)) - c0;
#pragma unroll
        for (int kb = 0; kb < 32; kb += 16) {
#pragma unroll
          for (int k = kb; k < kb + 16; ++k)
            x[k] = __ffma2_rn(make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1])),
                              sc2, make_float2(bp[-2 * k], bp[-2 * k - 1]));
          asm volatile("" ::: "memory");
        }
      }
      // this page's bias slot may be refilled (the loads above are ordered before it)
      mbar_arrive(&s.b_empty[i % kStages]);
      if (masked) {
        const int d0 = pq - k0 - c0;
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const int d = d0 - 2 * k;
          const bool a0 = d >= 0 && (W == 0 || d <= W - 1);
          const bool a1 = d - 1 >= 0 && (W == 0 || d - 1 <= W - 1);
          x[k].x = a0 ? x[k].x : -INFINITY;
          x[k].y = a1 ? x[k].y : -INFINITY;
        }
      }
      float mx0 = fmax3(x[0].x, x[0].y, x[1].x), mx1 = fmax3(x[1].y, x[2].x, x[2].y);
      float mx2 = fmax3(x[3].x, x[3].y, x[4].x), mx3 = fmax3(x[4].y, x[5].x, x[5].y);
#pragma unroll
      for (int k = 6; k < 30; k += 4) {
        mx0 = fmax3(mx0, x[k].x, x[k].y);
        mx1 = fmax3(mx1, x[k + 1].x, x[k + 1].y);
        mx2 = fmax3(mx2, x[k + 2].x, x[k + 2].y);
        mx3 = fmax3(mx3, x[k + 3].x, x[k + 3].y);
      }
      mx0 = fmax3(mx0, x[30].x, x[30].y);
      mx1 = fmax3(mx1, x[31].x, x[31].y);
      // the other half's maximum of this page.  Slot xm[i & 1][hf][r] is read only by the
      // partner warp (hf ^ 1, the same lanes), and this thread writes it again at page i + 2
      // only after both warps have passed page i + 1's exchange, which the partner enters
      // after its read: ordering within the warp pair is enough, and the pairs need not
      // wait for one another.
      const float pm = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      s.xm[i & 1][hf][r] = pm;
      mbar_arrive(&s.x_full[warp & 3][i & 1]);
      if (!mbar_wait(&s.x_full[warp & 3][i & 1], (i >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const float m_new = fmax3(m, pm, s.xm[i & 1][hf ^ 1][r]);
      const bool need = m_new > m + kRescaleThreshold || (m == -INFINITY && m_new > -INFINITY);
      const float alpha = need ? ex2((m - m_new) * kLog2e) : 1.f;
      if (need) {
        l2.x *= alpha;
        l2.y *= alpha;
        m = m_new;
      }
      const float nm = m == -INFINITY ? 0.f : -m * kLog2e;  // p = 2^(x log2 e - m log2 e)
      const float2 nm2 = make_float2(nm, nm);
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float2 d2 = __ffma2_rn(x[k], lg2, nm2);
        const float2 e2 = make_float2(ex2(d2.x), ex2(d2.y));
        l2 = __fadd2_rn(l2, e2);
        sr[k] = kFp8 ? pack_f16(e2.x, e2.y) : pack_bf16(e2.x, e2.y);
      }
      // rescale this half of O (warp-wide, only when some row's max grew past the threshold)
      if (__any_sync(0xffffffffu, need) && i > 0) {
        // O must hold PV(i-1) before it is scaled
        if (!mbar_wait(&s.pv_done, (i - 1) & 1, abort_flag, p.status)) ok = false;
        tc_fence_after();
        uint32_t orr[32];
        const uint32_t tO = tmem + lane_base + kColO + c0;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_ld32(tO + c * 32, orr);
          tmem_wait_ld();
          reg_fence<32>(orr);
#pragma unroll
          for (int j = 0; j < 32; ++j) orr[j] = __float_as_uint(__uint_as_float(orr[j]) * alpha);
          tmem_st32(tO + c * 32, orr);
        }
      }
      tmem_st32(tS + hf * 32, sr);  // P words 32 hf .. 32 hf + 31 (keys c0 .. c0 + 63)
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full[i & 1]);
      if (!ok) break;
    }
    // the two halves' sums
    const float l_mine = l2.x + l2.y;
    float l = l_mine;
    if (ok) {
      // slot np % 2 was last used by page np - 2, whose reads (by the partner warp only)
      // page np - 1's exchange ordered
      s.xm[np & 1][hf][r] = l_mine;
      mbar_arrive(&s.l_full);
      ok = mbar_wait(&s.l_full, 0, abort_flag, p.status);
      if (ok) l = l_mine + s.xm[np & 1][hf ^ 1][r];
    }
    if (ok) ok = mbar_wait(&s.o_full, 0, abort_flag, p.status);
    if (!ok) {
      report(p.status, kErrTimeout);
      s.abort_flag = 1;
    } else {
      tc_fence_after();
      const uint32_t tO = tmem + lane_base + kColO + c0;
      const bool direct = nsplit_b == 1;
      // V = code * v_scale for an FP8 cache: scaled here, partials included
      const float inv_l = direct ? p.v_scale / l : p.v_scale;
      const size_t prow = (((size_t)b * p.Hkv + kvh) * p.num_splits + split) * p.rmax + r;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t orr[32];
        tmem_ld32(tO + c * 32, orr);
        tmem_wait_ld();
        reg_fence<32>(orr);
        if (!valid) continue;
        const int col = c0 + c * 32;
        if (!direct) {
          float4* dst = reinterpret_cast<float4*>(p.part_o + prow * 128 + col);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dst[j] = make_float4(__uint_as_float(orr[4 * j]) * inv_l, __uint_as_float(orr[4 * j + 1]) * inv_l,
                                 __uint_as_float(orr[4 * j + 2]) * inv_l, __uint_as_float(orr[4 * j + 3]) * inv_l);
        } else {
          const size_t obase = ((size_t)(t_seq0 + t) * p.Hq + h) * 128 + col;
          if (p.out_dtype == 0) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + obase);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 w;
              w.x = pack_bf16(__uint_as_float(orr[8 * j + 0]) * inv_l, __uint_as_float(orr[8 * j + 1]) * inv_l);
              w.y = pack_bf16(__uint_as_float(orr[8 * j + 2]) * inv_l, __uint_as_float(orr[8 * j + 3]) * inv_l);
              w.z = pack_bf16(__uint_as_float(orr[8 * j + 4]) * inv_l, __uint_as_float(orr[8 * j + 5]) * inv_l);
              w.w = pack_bf16(__uint_as_float(orr[8 * j + 6]) * inv_l, __uint_as_float(orr[8 * j + 7]) * inv_l);
              dst[j] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(orr[4 * j + 0]) * inv_l, __uint_as_float(orr[4 * j + 1]) * inv_l,
                                   __uint_as_float(orr[4 * j + 2]) * inv_l, __uint_as_float(orr[4 * j + 3]) * inv_l);
          }
        }
      }
      if (valid && hf == 0) {
        if (nsplit_b == 1) {
          if (p.lse != nullptr) p.lse[(size_t)(t_seq0 + t) * p.Hq + h] = m + __log2f(l) * kLn2;
        } else {
          p.part_ml[prow * 2 + 0] = m;
          p.part_ml[prow * 2 + 1] = l;
        }
      }
    }
   }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the split partials of every (sequence, KV head) that needed more than one split.
// One warp per packed row (grid: row groups x KV heads x sequences); each lane owns 4 of
// the 128 output columns.  The split loop has no data-dependent branch, so the loads of
// several splits are in flight at once (a row with no allowed key in a split has m = -inf,
// l = 0 and O = 0 there, and gets weight 0).
constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const Params p) {
  const int kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * kCombineWarps + warp;
  pdl_wait();
  const int t_seq0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - t_seq0;
  if (p.conv_x[0] != nullptr && blockIdx.x == 0 && n > 0 && n <= p.max_q_len) {
    // fused conv: the new state of a sequence split over several CTAs (they have all read
    // the old one by now), the last three rows of [old state ; new rows], this KV head's
    // 128 channels of K and V, one thread per channel
    const int L = p.seq_lens[b];
    int kt_lo, kt_hi;
    page_range(L, n, p.window, kt_lo, kt_hi);
    const int nsp = (kt_hi - kt_lo + 1 + p.pages_per_split - 1) / p.pages_per_split;
    if (n <= L && L <= p.max_blocks * 128 && nsp > 1 && nsp <= p.num_splits) {
      const int C = p.Hkv * 128;
      const int which = threadIdx.x >> 7, c = kvh * 128 + (threadIdx.x & 127);
      uint16_t* st = p.conv_state + ((size_t)b * 2 + which) * 3 * C + c;
      uint16_t v[3];
#pragma unroll
      for (int k = 0; k < 3; ++k)
        v[k] = n + k < 3 ? st[(size_t)(n + k) * C] : p.conv_x[which][(size_t)(t_seq0 + n + k - 3) * C + c];
#pragma unroll
      for (int k = 0; k < 3; ++k) st[(size_t)k * C] = v[k];
    }
  }
  if (n <= 0 || n > p.max_q_len || r >= p.rmax) return;
  int t, g;
  if (!packed_row(r, n, p.G, t, g)) return;
  const int L = p.seq_lens[b];
  if (n > L || L > p.max_blocks * 128) return;
  int kt_lo, kt_hi;
  page_range(L, n, p.window, kt_lo, kt_hi);
  const int nsp = (kt_hi - kt_lo + 1 + p.pages_per_split - 1) / p.pages_per_split;
  if (nsp <= 1 || nsp > p.num_splits) return;
  const size_t base = ((size_t)b * p.Hkv + kvh) * p.num_splits;
  float M = -INFINITY;
  for (int sp = lane; sp < nsp; sp += 32) M = fmaxf(M, p.part_ml[((base + sp) * p.rmax + r) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float lsum = 0.f;
#pragma unroll 8
  for (int sp = 0; sp < nsp; ++sp) {
    const size_t prow = (base + sp) * p.rmax + r;
    const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + prow * 2);
    const float4 o = reinterpret_cast<const float4*>(p.part_o + prow * 128)[lane];
    const float wgt = ex2((ml.x - M) * kLog2e);  // m = -inf gives 0
    acc.x = fmaf(wgt, o.x, acc.x);
    acc.y = fmaf(wgt, o.y, acc.y);
    acc.z = fmaf(wgt, o.z, acc.z);
    acc.w = fmaf(wgt, o.w, acc.w);
    lsum = fmaf(wgt, ml.y, lsum);
  }
  const float inv = 1.f / lsum;
  const int h = kvh * p.G + g;
  const size_t obase = ((size_t)(t_seq0 + t) * p.Hq + h) * 128 + lane * 4;
  if (p.out_dtype == 0) {
    uint2 w;
    w.x = pack_bf16(acc.x * inv, acc.y * inv);
    w.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.out) + obase) = w;
  } else {
    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + obase) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (lane == 0 && p.lse != nullptr) p.lse[(size_t)(t_seq0 + t) * p.Hq + h] = M + __log2f(lsum) * kLn2;
}

}  // namespace decode

DecodeSplit decode_split(int B, int Hkv, int max_q_len, int max_seq_len, int window,
                         int num_splits_req, int num_sms) {
  // pages a sequence's decode rows can span (a window range may straddle one more page)
  long long range_pages = ((long long)max_seq_len + 127) / 128;
  if (window > 0) {
    const long long w_pages = ((long long)window + max_q_len - 1 + 127) / 128 + 1;
    if (w_pages < range_pages) range_pages = w_pages;
  }
  if (range_pages < 1) range_pages = 1;
  long long ns;
  if (num_splits_req > 0) {
    ns = num_splits_req;
  } else {
    // One CTA holds an SM (its K/V stages fill shared memory), so the grid runs in waves
    // of num_sms CTAs.
    const long long pairs = (B > 0 && Hkv > 0) ? (long long)B * Hkv : 1;
    if (pairs >= num_sms) {
      // Many sequences: about 8 CTAs per SM balance their ragged lengths, but a split
      // shorter than 32 pages costs more in pipeline fill and partial traffic than the
      // balance gains (a 4096-token window is not split at all).
      ns = (8LL * num_sms + pairs - 1) / pairs;
      long long cap = range_pages / 32;
      if (cap < 1) cap = 1;
      if (ns > cap) ns = cap;
    } else {
      // Few sequences (long context): equal splits that fill whole waves, the fewest
      // waves whose last one is at least 85% full; splits of at least 16 pages.
      long long cap = range_pages / 16;
      if (cap < 1) cap = 1;
      ns = 1;
      for (long long w = 1; w <= 8; ++w) {
        long long n_w = w * num_sms / pairs;
        if (n_w > cap) n_w = cap;
        if (n_w < 1) continue;
        ns = n_w;
        const long long ctas = n_w * pairs;
        const long long waves = (ctas + num_sms - 1) / num_sms;
        if (n_w == cap || ctas * 100 >= 85LL * waves * num_sms) break;
      }
    }
  }
  if (ns < 1) ns = 1;
  if (ns > range_pages) ns = range_pages;
  const long long pps = (range_pages + ns - 1) / ns;
  ns = (range_pages + pps - 1) / pps;
  return DecodeSplit{(int)ns, (int)pps};
}

// Rows of a packed tile for up to max_q_len tokens (whole warps when G divides 32).
static int decode_rmax(int max_q_len, int G) {
  return 32 % G == 0 ? 32 * decode::packed_warps(max_q_len, G) : max_q_len * G;
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int max_q_len, int num_splits) {
  if (num_splits <= 1) return 0;
  const size_t rmax = (size_t)decode_rmax(max_q_len, Hq / Hkv);
  const size_t rows = (size_t)B * Hkv * num_splits * rmax;
  return rows * 128 * sizeof(float) + rows * 2 * sizeof(float) + 256;
}

cudaError_t launch_decode(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
  using namespace decode;
  Params p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.block_table = a.block_table;
  p.cu_q_lens = a.cu_q_lens;
  p.seq_lens = a.seq_lens;
  p.bias = a.bias;
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.dev_status;
  p.max_blocks = a.max_blocks;
  p.R = a.R;
  p.window = a.window;
  p.out_dtype = a.out_dtype;
  p.B = a.B;
  p.T = a.T;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.max_q_len = a.max_q_len;
  p.rmax = decode_rmax(a.max_q_len, p.G);
  p.num_splits = a.num_splits;
  p.pages_per_split = a.pages_per_split;
  p.num_blocks = a.num_blocks;
  p.scale = a.kv_fp8 ? a.scale * a.k_scale : a.scale;  // K = code * k_scale
  p.v_scale = a.kv_fp8 ? a.v_scale : 1.f;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.conv_x[0] = static_cast<const uint16_t*>(a.conv_k_raw);
  p.conv_x[1] = static_cast<const uint16_t*>(a.conv_v_raw);
  p.conv_w[0] = a.conv_w_k;
  p.conv_w[1] = a.conv_w_v;
  p.conv_state = static_cast<uint16_t*>(a.conv_state);
  p.cache_w[0] = static_cast<uint16_t*>(const_cast<void*>(a.k_cache));
  p.cache_w[1] = static_cast<uint16_t*>(const_cast<void*>(a.v_cache));
  if (a.num_splits > 1) {
    const size_t rows = (size_t)a.B * a.Hkv * a.num_splits * p.rmax;
    uintptr_t w = (reinterpret_cast<uintptr_t>(a.workspace) + 255) & ~uintptr_t(255);
    p.part_o = reinterpret_cast<float*>(w);
    p.part_ml = p.part_o + rows * 128;
  }
  if (a.B == 0) return cudaSuccess;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(a.kv_fp8 ? decode_kernel<true> : decode_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.num_splits, a.Hkv, a.B);
  {
    // an increase that the launch allocation cannot cover would wait forever
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, a.kv_fp8 ? decode_kernel<true> : decode_kernel<false>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != (a.kv_fp8 ? kF8LaunchRegs : kLaunchRegs)) return cudaErrorInvalidConfiguration;
  }
  e = a.kv_fp8 ? launch_pdl(decode_kernel<true>, grid, dim3(kThreadsF8), smem, stream, maps.k,
                            maps.v, p)
               : launch_pdl(decode_kernel<false>, grid, dim3(kThreads), smem, stream, maps.k,
                            maps.v, p);
  if (e != cudaSuccess || a.num_splits <= 1) return e;
  return launch_pdl(combine_kernel, dim3((p.rmax + kCombineWarps - 1) / kCombineWarps, a.Hkv, a.B),
                    dim3(kCombineWarps * 32), 0, stream, p);
}

}  // namespace ink
