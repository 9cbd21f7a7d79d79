// Relative-bias GQA prefill attention on the fifth-generation tensor core (sm_103a).
//
// What it computes (vLLM Day-0 Inkling blog, "Model Architecture / Attention"): for each
// new token at position p and query head h,
//   out = sum_j softmax_j(scale * q.K[j] + b[h][min(p - j, R-1)]) V[j]
// over keys j with 0 <= p - j (and p - j <= window - 1 for sliding-window layers), keys
// and values read from the paged bf16 cache.
//
// Design (one CTA = 128 query tokens x two query heads of one KV group):
//   warp 8      TMA producer: Q tiles once, then K and V pages (two-stage ring).
//   warp 9      MMA issuer: S = Q K^T (SS form), O += P V (P read from tensor memory,
//               TS form), each product's eight k-steps issued by the lane elect.sync
//               picks from one asm block (mma8_*), commits to mbarriers.  Owns the TMEM
//               allocation.  Waits for V(i) and K(i+1) before P_A(i).
//   warps 10-11 bias stagers (one per head): stage the tile's slice of the bias table
//               in shared memory, one stage ahead (one bulk copy expanded into four
//               shifted copies, or 4-byte cp.async where entries need clamping).
//   warps 0-3   softmax for head A, warps 4-7 softmax for head B: thread r owns query row
//               r (= TMEM lane r).  It loads its S row, adds the relative bias (which
//               carries the mask), keeps a running max / sum (rescaling O in TMEM only when the max grew by
//               more than 2^8), writes P as bf16 over the S columns, and finally
//               normalises O and stores it.
// Tensor memory (512 columns): S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512);
// P_X overlays the first 64 columns of S_X.  The issuer issues
//   S_A0 S_B0 | PV_A0 S_A1 | PV_B0 S_B1 | PV_A1 S_A2 | ...
// so each softmax group works while the tensor core serves the other (ping-pong).  Each
// head's O is signalled right after its own last PV, so head A's epilogue runs while head
// B finishes its last tile.
//
// The relative bias ("sheared" along the tile diagonals): within a 128x128 tile the
// distance is delta + r - c with delta = p0 - k0, so row r needs a contiguous run of the
// table, reversed.  The stager warp puts the 255 values a tile needs in shared memory in
// reversed order, four times: copy j shifted by j words, the copies 264 words apart.  Row
// r then reads its run as 16-byte loads from copy (127 - r) mod 4, and the eight loads of
// each quarter-warp land in distinct banks (a quarter of the load instructions of 4-byte
// reads, with no bank conflicts).  The mask rides on the slice: a distance that is not
// attended (negative, or past the window) is staged as -inf, so tiles on the causal
// diagonal or the window edge run the same code as the others, and the rows of K and V
// past the end of the sequence are zeroed in shared memory so that stale slots cannot
// put a NaN into the logits.  Tiles whose smallest distance is already past R-1, and
// that need no mask, use the single clamped value instead (no copies, no loads).
// Logits are kept in natural units (x = scale * q.k + b) and log2 e is folded into the
// exponent's FMA.  Key tiles are visited from the diagonal backwards; tiles outside the
// window are never visited.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.h"
#include "ptx.cuh"

namespace ink {
namespace prefill {

// Source of the masked bias slots: the stagers copy it like any other table entry.
__device__ const float kMaskedBias = -INFINITY;

constexpr int kTile = 128;
constexpr int kStages = 2;
constexpr int kThreads = 384;  // three warpgroups: softmax A, softmax B, producer/MMA
// Register split (setmaxnreg): the kernel is built for 168 registers a thread at launch
// (65536 / 384, rounded down to 8), i.e. 64512 for the CTA.  The producer/MMA warpgroup
// gives back down to 64 and each softmax warpgroup grows to 216: 2*128*216 + 128*64 =
// 63488 <= 64512.  The host refuses to launch unless the built register count is 168,
// since an increase that the launch cannot cover would wait forever.
constexpr int kLaunchRegs = 168;
constexpr int kSoftmaxRegs = 216;
constexpr int kOtherRegs = 64;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kOtherRegs <= kThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 128, false, true);
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 5.545177444479562f;  // 8 ln 2: rescale O past 256x growth
// Bias slice layout: copy j (j = 0..3) holds rev[i + j] at word j * kBiasCopyStride + i.
// 264 = 256 + 8 words puts the copies' 16-byte chunks in different bank groups for the
// eight consecutive rows of a quarter-warp, whatever the row offset.
constexpr int kBiasCopyStride = 264;
constexpr int kBiasWords = 3 * kBiasCopyStride + 256;

struct __align__(1024) Smem {
  uint8_t q[2][2][16384];        // [head slot][d half][128 rows x 128 B], swizzled
  uint8_t k[kStages][2][16384];  // [stage][d half][128 keys x 128 B]
  uint8_t v[kStages][2][16384];
  // [stage][head slot][copy layout]: rev[j] = b[h][clamp(delta + 127 - j)], four shifted copies
  float bias[kStages][2][kBiasWords];
  float bias_raw[kStages][2][264];  // the tile's run of the table, as one bulk copy landed it
  uint64_t q_full;
  // a K stage is free once the tile's last QK^T is done, a V stage once its last PV is
  // done: K for the next tile is fetched while the current tile's softmax and PV run
  uint64_t k_full[kStages], v_full[kStages], k_empty[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], drain, b_full[kStages];
  uint64_t raw_full[kStages][2];
  uint32_t tmem_base;
  int abort_flag;
};

struct Params {
  const int32_t* block_table;
  const int32_t* cu_q_lens;
  const int32_t* seq_lens;
  const float* bias;
  void* out;
  float* lse;
  int* status;
  int max_blocks, R, window, out_dtype;
  int B, T, Hq, Hkv, G, pairs_per_group, head_pairs, q_tiles, max_q_len;
  long long num_blocks;
  float scale;
  float out_scale;  // output factor (v_scale of a widened FP8 cache, else 1)
};

__device__ __forceinline__ uint64_t desc_kmajor(const uint8_t (*atoms)[16384], int ks) {
  return sdesc_sw128(smem_u32(atoms[ks >> 2]) + (ks & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_v(const uint8_t (*atoms)[16384], int ks) {
  // V tile [128 keys][128 d] as two 64-wide d halves: MN-major B operand,
  // 16 keys per MMA = 2048 bytes, the two d halves 16 KB apart.
  return sdesc_sw128(smem_u32(atoms[0]) + ks * 2048, 16384, 1024);
}
// A value the compiler must treat as new at this point: keeps it from precomputing, and
// holding in the issuer's few registers, the k-step descriptors of the Q tiles.
__device__ __forceinline__ uint64_t opaque(uint64_t x) {
  asm volatile("" : "+l"(x));
  return x;
}


__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap map_q,
               const __grid_constant__ CUtensorMap map_k,
               const __grid_constant__ CUtensorMap map_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const int warp = warp_id(), lane = lane_id();
  pdl_wait();

  // ---- work item: one KV group after another, so that the CTAs resident at a time
  // share the K/V of one or two groups (a group's whole history, 32 MB at 64K tokens,
  // stays in L2 while they stream it) and each group's K/V is read from HBM about once;
  // within a group, heavy (late) query tiles first, then sequences, then the group's
  // head pairs ----
  const int idx = blockIdx.x;
  const int per_tile = p.B * p.pairs_per_group;  // items of one query tile and KV group
  const int per_group = p.q_tiles * per_tile;
  const int kvg = idx / per_group;
  int rr = idx - kvg * per_group;
  const int qt_rank = rr / per_tile;
  rr -= qt_rank * per_tile;
  const int b = rr / p.pairs_per_group;
  const int hp = kvg * p.pairs_per_group + (rr - b * p.pairs_per_group);
  const int qt = p.q_tiles - 1 - qt_rank;
  const int t_seq0 = p.cu_q_lens[b];
  const int n = p.cu_q_lens[b + 1] - t_seq0;
  if (qt * kTile >= n) return;  // whole CTA, before any barrier
  const int L = p.seq_lens[b];
  if (n > L || n > p.max_q_len || L > p.max_blocks * kTile) {
    if (threadIdx.x == 0) report(p.status, kErrBadInput);
    return;
  }
  const int P0 = L - n + qt * kTile;  // position of row 0
  const int rows = min(kTile, n - qt * kTile);
  const int lo = p.window > 0 ? max(0, P0 - p.window + 1) : 0;
  const int hi = P0 + rows - 1;
  const int kt_lo = lo / kTile, kt_hi = hi / kTile;
  const int ntiles = kt_hi - kt_lo + 1;
  const int kvh = hp / p.pairs_per_group;
  const int h0 = kvh * p.G + 2 * (hp % p.pairs_per_group);
  const bool has_b = (2 * (hp % p.pairs_per_group) + 1) < p.G;
  const int t_glob0 = t_seq0 + qt * kTile;
  const int32_t* table = p.block_table + (size_t)b * p.max_blocks;

  // Page ids are checked by the producer as it reaches them (a TMA load with an id
  // outside the cache would only read the fill value, but the call must report it).
  if (threadIdx.x == 0) {
    s.abort_flag = 0;
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_empty[i], 1);
      mbar_init(&s.b_full[i], 64);
      mbar_init(&s.raw_full[i][0], 1);
      mbar_init(&s.raw_full[i][1], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    mbar_init(&s.o_full[0], 1);
    mbar_init(&s.o_full[1], 1);
    mbar_init(&s.drain, 1);
    fence_barrier_init();
  }
  if (warp == 9) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  volatile int* abort_flag = &s.abort_flag;

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kOtherRegs));
   if (warp == 8) {
    // ------------------------------------------------------------ TMA producer ---
    if (lane == 0) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&s.q_full, has_b ? 65536u : 32768u);
      tma_load_3d(s.q[0][0], &map_q, &s.q_full, 0, h0, t_glob0);
      tma_load_3d(s.q[0][1], &map_q, &s.q_full, 64, h0, t_glob0);
      if (has_b) {
        tma_load_3d(s.q[1][0], &map_q, &s.q_full, 0, h0 + 1, t_glob0);
        tma_load_3d(s.q[1][1], &map_q, &s.q_full, 64, h0 + 1, t_glob0);
      }
      int issued = 0;
      // page ids read three tiles ahead, so no TMA issue waits on a block-table load
      auto page_id = [&](int j) -> int32_t { return j < ntiles ? table[kt_hi - j] : 0; };
      int32_t id1 = page_id(0), id2 = page_id(1), id3 = page_id(2);
      for (int i = 0; i < ntiles; ++i) {
        const int st = i % kStages;
        const uint32_t eph = ((i / kStages) - 1) & 1;
        const int32_t blk = id1;
        id1 = id2;
        id2 = id3;
        id3 = page_id(i + 3);
        if (i >= kStages && !mbar_wait(&s.k_empty[st], eph, abort_flag, p.status)) {
          report(p.status, kErrTimeout);
          s.abort_flag = 1;
          break;
        }
        if (blk < 0 || (long long)blk >= p.num_blocks) {
          report(p.status, kErrBadBlock);  // first error wins: reported before the abort
          s.abort_flag = 1;
          issued = i;
          break;
        }
        const int page = blk * p.Hkv + kvh;
        mbar_arrive_expect_tx(&s.k_full[st], 32768u);
        tma_load_3d(s.k[st][0], &map_k, &s.k_full[st], 0, 0, page);
        tma_load_3d(s.k[st][1], &map_k, &s.k_full[st], 64, 0, page);
        if (i >= kStages && !mbar_wait(&s.v_empty[st], eph, abort_flag, p.status)) {
          report(p.status, kErrTimeout);
          s.abort_flag = 1;
          issued = i;  // this tile's K is in flight too: let it land
          volatile int never = 0;
          mbar_wait(&s.k_full[st], (i / kStages) & 1, &never);
          break;
        }
        mbar_arrive_expect_tx(&s.v_full[st], 32768u);
        tma_load_3d(s.v[st][0], &map_v, &s.v_full[st], 0, 0, page);
        tma_load_3d(s.v[st][1], &map_v, &s.v_full[st], 64, 0, page);
        issued = i + 1;
      }
      if (*abort_flag) {
        // let the copies already in flight land before the CTA goes away
        volatile int never_q = 0;
        mbar_wait(&s.q_full, 0, &never_q);
        for (int i = max(0, issued - kStages); i < issued; ++i) {
          const int st = i % kStages;
          const uint32_t ph = (i / kStages) & 1;
          volatile int never = 0;
          mbar_wait(&s.k_full[st], ph, &never);
          mbar_wait(&s.v_full[st], ph, &never);
        }
      }
    }
   } else if (warp >= 10) {
    // ---------------------------------------------------------- bias stagers ---
    // warp 10 stages head A's slice, warp 11 head B's: rev[j] = b[h][min(d, R-1)] at
    // distance d = delta + 127 - j, j < 256, or -inf where d is not attended (d < 0, or
    // past the window), written to the four shifted copies, so softmax thread r reads
    // its run rev[127 - r + c], c = 0..127, four values at a time.  When the tile's
    // distances need no clamping, lane 0 fetches their run of the table with one
    // 16-byte-aligned bulk copy and the warp expands it into the copies from shared
    // memory; otherwise all lanes copy the clamped entries with 4-byte cp.async.  Both
    // warps arrive on b_full[stage] for every tile (count 64).
    const int slot = warp - 10;
    const bool mine = slot == 0 || has_b;
    const float* brow = p.bias + (size_t)(h0 + slot) * p.R;
    const int R = p.R, W = p.window;
    const bool bulk_ok = ((reinterpret_cast<uintptr_t>(p.bias) & 15) == 0) && (R & 3) == 0;
    // raw_full[stage] completes once per bulk copy into that stage, and only some tiles
    // take the bulk path: count the uses per stage to know which phase to wait for
    uint32_t raw_uses = 0;  // bit st: parity of the next use of stage st (kStages <= 32)
    for (int i = 0; i < ntiles; ++i) {
      const int st = i % kStages;
      int ok = 1;
      if (lane == 0 && i >= kStages)
        ok = mbar_wait(&s.v_empty[st], ((i / kStages) - 1) & 1, abort_flag, p.status);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int delta = P0 - (kt_hi - i) * kTile;
      const bool masked = delta < 127 || (W > 0 && delta + 127 > W - 1);
      const int a0 = (delta - 127) & ~3;              // the run starts 16-byte aligned
      const int cnt = (delta + 127 - a0 + 4) & ~3;    // <= 258, rounded up to 4
      float* dst = &s.bias[st][slot][0];
      if (mine && (delta - 127 < R - 1 || masked) && bulk_ok && a0 >= 0 && a0 + cnt <= R) {
        float* raw = &s.bias_raw[st][slot][0];
        uint64_t* rf = &s.raw_full[st][slot];
        if (lane == 0) {
          mbar_arrive_expect_tx(rf, (uint32_t)(cnt * 4));
          bulk_g2s(raw, brow + a0, (uint32_t)(cnt * 4), rf);
        }
        const uint32_t par = (raw_uses >> st) & 1u;
        raw_uses ^= 1u << st;
        if (!mbar_wait(rf, par, abort_flag, p.status)) {
          volatile int never = 0;  // the copy may still be in flight: let it land
          if (lane == 0) mbar_wait(rf, par, &never);
          __syncwarp();
          break;
        }
#pragma unroll
        for (int j = lane; j < 256; j += 32) {
          const int d = delta + 127 - j;
          const bool off = d < 0 || (W > 0 && d > W - 1);
          const float v = off ? -INFINITY : raw[d - a0];
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (j >= c) dst[c * kBiasCopyStride + j - c] = v;
        }
        __syncwarp();
        mbar_arrive(&s.b_full[st]);  // release: the stores above are seen by the waiters
        continue;
      }
      if (mine && (delta - 127 < R - 1 || masked)) {
#pragma unroll
        for (int j = lane; j < 256; j += 32) {
          const int d = delta + 127 - j;
          const bool off = d < 0 || (W > 0 && d > W - 1);
          const float* src = off ? &kMaskedBias : brow + (d > R - 1 ? R - 1 : d);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (j >= c) cp_async_4(dst + c * kBiasCopyStride + j - c, src);
        }
      }
      cp_async_mbar_arrive(&s.b_full[st]);
    }
    // let outstanding copies land before the CTA can exit
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer ---
    // The whole warp runs this loop converged (the issue blocks and their commits elect
    // one lane); each wait's outcome is made warp-uniform before it is acted on.
    const uint64_t dq0 = desc_kmajor(s.q[0], 0), dq1 = desc_kmajor(s.q[1], 0);
    auto qk = [&](uint32_t tmem_d, uint64_t dq, const uint8_t (*k_atoms)[16384]) {
      mma8_ss_kmajor<kIdescQK>(tmem_d, opaque(dq), desc_kmajor(k_atoms, 0), 0);
    };
    auto pv = [&](uint32_t tmem_d, uint32_t tmem_p, const uint8_t (*v_atoms)[16384], bool acc) {
      mma8_ts_mnmajor<kIdescPV>(tmem_d, tmem_p, desc_v(v_atoms, 0), acc ? 1u : 0u);
    };
    bool ok = mbar_wait(&s.q_full, 0, abort_flag, p.status) && mbar_wait(&s.k_full[0], 0, abort_flag, p.status);
    ok = __all_sync(0xffffffffu, ok);
    bool issued_any = false;
    if (ok) {
      // tile 0 holds the diagonal: keys past the end of the sequence are stale slots
      if ((kt_hi + 1) * kTile > L) zero_tail_rows(s.k[0], L - kt_hi * kTile, lane);
      tc_fence_after();
      qk(tmem + 0, dq0, s.k[0]);
      umma_commit_elected(&s.s_full[0]);
      if (has_b) {
        qk(tmem + 128, dq1, s.k[0]);
        umma_commit_elected(&s.s_full[1]);
      }
      umma_commit_elected(&s.k_empty[0]);  // tile 0's K has been read by both QK^T
      issued_any = true;
    }
    for (int i = 0; ok && i < ntiles; ++i) {
      const int st = i % kStages;
      const uint32_t ph = (i / kStages) & 1;
      const bool more = i + 1 < ntiles;
      const int st1 = (i + 1) % kStages;
      // V(i) and K(i+1) have normally landed long before P_A(i) (their stages were freed
      // a tile earlier): wait for them first, so that PV_A(i) and S_A(i+1) follow P_A(i)
      // back to back.
      ok = mbar_wait(&s.v_full[st], ph, abort_flag, p.status) &&
           (!more || mbar_wait(&s.k_full[st1], ((i + 1) / kStages) & 1, abort_flag, p.status));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // keys past the end of the sequence: their P is 0, but junk V could be NaN
      if (i == 0 && (kt_hi + 1) * kTile > L) zero_tail_rows(s.v[st], L - kt_hi * kTile, lane);
      ok = mbar_wait(&s.p_full[0], i & 1, abort_flag, p.status);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      pv(tmem + 256, tmem + 0, s.v[st], i > 0);
      if (!more) umma_commit_elected(&s.o_full[0]);  // head A's O is final
      if (more) {
        qk(tmem + 0, dq0, s.k[st1]);
        umma_commit_elected(&s.s_full[0]);
      }
      if (has_b) {
        ok = mbar_wait(&s.p_full[1], i & 1, abort_flag, p.status);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        pv(tmem + 384, tmem + 128, s.v[st], i > 0);
        if (!more) umma_commit_elected(&s.o_full[1]);
      }
      umma_commit_elected(&s.v_empty[st]);  // both PV of tile i are issued
      if (has_b && more) {
        qk(tmem + 128, dq1, s.k[st1]);
        umma_commit_elected(&s.s_full[1]);
      }
      if (more) umma_commit_elected(&s.k_empty[st1]);  // both QK^T of tile i+1 are issued
    }
    if (!ok) {
      report(p.status, kErrTimeout);
      s.abort_flag = 1;
      if (issued_any) {
        // wait for the tensor core to finish whatever was issued before freeing TMEM
        umma_commit_elected(&s.drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&s.drain, 0, &never);
      }
    }
    __syncwarp();
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax groups ---
    const int grp = warp >> 2;  // 0 = head A, 1 = head B
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + grp * 128;
    const uint32_t tO = tmem + lane_base + 256 + grp * 128;
    const int h = h0 + grp;
    if (grp == 0 || has_b) {
      const float* brow = p.bias + (size_t)h * p.R;
      const float bconst = __ldg(brow + p.R - 1);
      const int R = p.R, W = p.window;
      float m = -INFINITY;  // running max of the logits, natural units
      float2 l2 = make_float2(0.f, 0.f);
      const float2 sc2 = make_float2(p.scale, p.scale);
      const float2 lg2 = make_float2(kLog2e, kLog2e);
      bool ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int k0 = (kt_hi - i) * kTile;
        const int delta = P0 - k0;
        // the single clamped value serves only tiles with every distance past the table end
        // and attended; the others read the staged slice, which carries the mask as -inf
        const bool clamped = delta - 127 >= R - 1 && !(delta < 127 || (W > 0 && delta + 127 > W - 1));
        const float* bias_buf = &s.bias[i % kStages][grp][0];
        if (!clamped && !mbar_wait(&s.b_full[i % kStages], (i / kStages) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&s.s_full[grp], i & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        // S row in two halves: the second half's TMEM load overlaps work on the first
        uint32_t sr[128];
        tmem_ld32(tS + 0, sr);
        tmem_ld32(tS + 32, sr + 32);
        tmem_wait_ld();
        reg_fence<64>(sr);
        tmem_ld32(tS + 64, sr + 64);
        tmem_ld32(tS + 96, sr + 96);
        float2 x[64];  // logit * log2 e, pairs of columns
        // rb4[k] = bias at distance delta + r - c for columns c = 4k .. 4k+3 (16-byte aligned)
        const int bsh = (127 - r) & 3;
        const float4* rb4 =
            reinterpret_cast<const float4*>(bias_buf + bsh * kBiasCopyStride + (127 - r - bsh));
        const float2 bc2 = make_float2(bconst, bconst);
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
          const float2 sv0 = make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1]));
          const float2 sv1 = make_float2(__uint_as_float(sr[2 * k + 2]), __uint_as_float(sr[2 * k + 3]));
          if (clamped) {
            x[k] = __ffma2_rn(sv0, sc2, bc2);
            x[k + 1] = __ffma2_rn(sv1, sc2, bc2);
          } else {
            const float4 b4 = rb4[k >> 1];
            x[k] = __ffma2_rn(sv0, sc2, make_float2(b4.x, b4.y));
            x[k + 1] = __ffma2_rn(sv1, sc2, make_float2(b4.z, b4.w));
          }
        }
        tmem_wait_ld();
        reg_fence<64>(sr + 64);
#pragma unroll
        for (int k = 32; k < 64; k += 2) {
          const float2 sv0 = make_float2(__uint_as_float(sr[2 * k]), __uint_as_float(sr[2 * k + 1]));
          const float2 sv1 = make_float2(__uint_as_float(sr[2 * k + 2]), __uint_as_float(sr[2 * k + 3]));
          if (clamped) {
            x[k] = __ffma2_rn(sv0, sc2, bc2);
            x[k + 1] = __ffma2_rn(sv1, sc2, bc2);
          } else {
            const float4 b4 = rb4[k >> 1];
            x[k] = __ffma2_rn(sv0, sc2, make_float2(b4.x, b4.y));
            x[k + 1] = __ffma2_rn(sv1, sc2, make_float2(b4.z, b4.w));
          }
        }
        float mx0 = fmax3(x[0].x, x[0].y, x[1].x), mx1 = fmax3(x[1].y, x[2].x, x[2].y);
        float mx2 = fmax3(x[3].x, x[3].y, x[4].x), mx3 = fmax3(x[4].y, x[5].x, x[5].y);
#pragma unroll
        for (int k = 6; k < 62; k += 4) {
          mx0 = fmax3(mx0, x[k].x, x[k].y);
          mx1 = fmax3(mx1, x[k + 1].x, x[k + 1].y);
          mx2 = fmax3(mx2, x[k + 2].x, x[k + 2].y);
          mx3 = fmax3(mx3, x[k + 3].x, x[k + 3].y);
        }
        mx0 = fmax3(mx0, x[62].x, x[62].y);
        mx1 = fmax3(mx1, x[63].x, x[63].y);
        const float m_new = fmax3(m, fmaxf(mx0, mx1), fmaxf(mx2, mx3));
        const bool need = m_new > m + kRescaleThreshold || (m == -INFINITY && m_new > -INFINITY);
        const float alpha = need ? ex2((m - m_new) * kLog2e) : 1.f;
        if (need) {
          l2.x *= alpha;
          l2.y *= alpha;
          m = m_new;
        }
        const float nm = m == -INFINITY ? 0.f : -m * kLog2e;  // p = 2^(x log2 e - m log2 e)
        const float2 nm2 = make_float2(nm, nm);
        // P as bf16 pairs, reusing the S registers
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          const float2 d2 = __ffma2_rn(x[k], lg2, nm2);
          const float2 e2 = make_float2(ex2(d2.x), ex2(d2.y));
          l2 = __fadd2_rn(l2, e2);
          sr[k] = pack_bf16(e2.x, e2.y);
        }
        // rescale O (warp-wide, only when some row's max grew past the threshold)
        if (__any_sync(0xffffffffu, need) && i > 0) {
          // PV(i-1) was issued before S(i), so it is complete here
          uint32_t orr[32];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            tmem_ld32(tO + c * 32, orr);
            tmem_wait_ld();
            reg_fence<32>(orr);
#pragma unroll
            for (int j = 0; j < 32; ++j) orr[j] = __float_as_uint(__uint_as_float(orr[j]) * alpha);
            tmem_st32(tO + c * 32, orr);
          }
        }
        tmem_st32(tS + 0, sr);
        tmem_st32(tS + 32, sr + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[grp]);
      }
      const float l = l2.x + l2.y;
      if (ok) ok = mbar_wait(&s.o_full[grp], 0, abort_flag, p.status);
      if (!ok) {
        report(p.status, kErrTimeout);
        s.abort_flag = 1;
      } else {
        tc_fence_after();
        const float inv_l = p.out_scale / l;
        const int t = t_glob0 + r;
        const bool store = r < rows;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t orr[32];
          tmem_ld32(tO + c * 32, orr);
          tmem_wait_ld();
          reg_fence<32>(orr);
          if (store) {
            const size_t obase = ((size_t)t * p.Hq + h) * 128 + c * 32;
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
        if (store && p.lse != nullptr) p.lse[(size_t)t * p.Hq + h] = m + __log2f(l) * kLn2;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace prefill

cudaError_t launch_prefill(const AttnArgs& a, const AttnMaps& maps, cudaStream_t stream) {
  using namespace prefill;
  Params p;
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
  p.pairs_per_group = (p.G + 1) / 2;
  p.head_pairs = a.Hkv * p.pairs_per_group;
  p.q_tiles = (a.max_q_len + kTile - 1) / kTile;
  p.max_q_len = a.max_q_len;
  p.num_blocks = a.num_blocks;
  p.scale = a.scale;
  p.out_scale = a.out_scale;
  const long long grid = (long long)p.q_tiles * p.B * p.head_pairs;
  if (grid == 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const size_t smem = sizeof(Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_kernel);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;  // see kLaunchRegs
  return launch_pdl(prefill_kernel, dim3((unsigned)grid), dim3(kThreads), smem, stream, maps.q,
                    maps.k, maps.v, p);
}

}  // namespace ink
