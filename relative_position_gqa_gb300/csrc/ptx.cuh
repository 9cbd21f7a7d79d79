// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor), and the
// fifth-generation tensor core (tcgen05.alloc / mma / commit / ld / st) with its shared
// memory and instruction descriptors.  Every wait is bounded: a wait that runs out of
// its cycle budget returns false and the caller records an error and unwinds.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace ink {

// ------------------------------------------------------------------ status words ---
// Codes match inkling_status_t in include/inkling.h.
enum : int {
  kOk = 0, kErrInvalidArg = 1, kErrUnsupported = 2, kErrCuda = 3, kErrTimeout = 4,
  kErrBadBlock = 5, kErrBadInput = 6, kErrWorkspace = 7
};

// First writer wins: later errors never overwrite the first one.
__device__ __forceinline__ void report(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ~2 s at the boost clock: far beyond any legitimate wait inside one launch.
constexpr long long kWaitBudgetCycles = 4000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------- mbarrier ------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Programmatic dependent launch: every kernel of the library is launched so that it may
// start while the previous kernel on the stream is still finishing, and waits here for
// that kernel's completion (and the visibility of its memory) before it reads any input.
// The short conv kernels also release the next launch early, so the attention grid that
// follows them is resident when they finish; the attention kernels do not (measured:
// releasing early from them cost 1-2% on back-to-back decode steps).  Without a
// predecessor that allows it, both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase with the given parity to complete.  Gives up (returns false) when
// `abort_flag` is raised by another warp of the CTA, after kWaitBudgetCycles, or, once the
// wait has lasted kGlobalPollAfter cycles, when the launch's global status word
// (nullable) shows that some CTA has already failed.  The slow checks only run every few
// spins and global memory is not touched at all by a wait of normal length.
constexpr long long kGlobalPollAfter = 1000000LL;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag,
                                          const int* global_status = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 15u) != 0) continue;
    if (*abort_flag) return false;
    if ((spins & 255u) == 0) {
      const long long dt = clock64() - t0;
      if (dt > kWaitBudgetCycles) return false;
      if (dt > kGlobalPollAfter && global_status != nullptr &&
          *reinterpret_cast<const volatile int*>(global_status) != 0)
        return false;
    }
  }
  return true;
}

// 4-byte asynchronous global -> shared copy (no register round trip); pair with
// cp_async_mbar_arrive so an mbarrier tracks its completion.
// Bulk copy global -> shared (no tensor map): both addresses 16-byte aligned, bytes a
// multiple of 16; completion is counted on the mbarrier's transaction bytes.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst_smem)), "l"(src)
               : "memory");
}
// Arrive on `bar` once every cp.async issued so far by this thread has landed (the
// barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------------------------ TMA ------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled load into shared memory, completion counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map,
                                                 uint64_t* bar, int c0, int c1, int c2,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05 ------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Same with the A operand read from tensor memory (one row per lane, bf16 pairs packed
// in 32-bit columns).
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Eight-k-step MMA issue blocks: D[d] (+)= A B over the eight 16-wide k-steps of a
// 128-deep product, issued from the lane that elect.sync picks, with every lane of the
// warp executing the block (converged), in one asm statement that adds the k-step offsets
// itself.  Issued this way a warp keeps up one MMA every ~40 cycles while other warps on
// its sub-partition run FFMA/MUFU work; single-MMA statements under a lane-0 branch fell
// to one every 130-260 cycles under the same load.  The first k-step accumulates iff
// acc != 0, the others always.
//
// A k-step's descriptor is that of k-step 0 plus its start-address offset: the address
// field counts 16-byte units, and shared addresses plus the offsets stay below its 2^18 B,
// so the add never carries into the next field.  K-major operands are two 64-column
// 128-byte-swizzled atoms 16 KB apart, k-step ks starting (ks & 3) * 32 bytes into atom
// ks >> 2 (+2 and +1024 units); an MN-major B operand steps 16 rows = 2048 bytes (+128);
// a TMEM A operand steps 8 columns (16 bf16/f16 values packed in pairs).
#define INK_MMA_SS_STEP(off)                                  \
  "add.s64 ra, %1, " #off ";\n\tadd.s64 rb, %2, " #off ";\n\t" \
  "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], ra, rb, %3, pt;\n\t"
#define INK_MMA_TS_STEP(ao, bo)                                 \
  "add.s32 rt, %1, " #ao ";\n\tadd.s64 rb, %2, " #bo ";\n\t"    \
  "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [rt], rb, %3, pt;\n\t"
#define INK_MMA_HEAD                                                   \
  "setp.ne.b32 pa, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\t"             \
  "elect.sync _|pe, 0xffffffff;\n\t"
// A and B K-major in shared memory (S = Q K^T of the prefill).
template <uint32_t kIdesc>
__device__ __forceinline__ void mma8_ss_kmajor(uint32_t d, uint64_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred pe, pa, pt;\n\t.reg .b64 ra, rb;\n\t" INK_MMA_HEAD
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, pa;\n\t"
      INK_MMA_SS_STEP(2) INK_MMA_SS_STEP(4) INK_MMA_SS_STEP(6) INK_MMA_SS_STEP(1024)
      INK_MMA_SS_STEP(1026) INK_MMA_SS_STEP(1028) INK_MMA_SS_STEP(1030) "}" ::"r"(d),
      "l"(a), "l"(b), "n"(kIdesc), "r"(acc)
      : "memory");
}
// A in TMEM, B K-major in shared memory (S = K Q^T of the decode: Q resident in TMEM).
template <uint32_t kIdesc>
__device__ __forceinline__ void mma8_ts_kmajor(uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred pe, pa, pt;\n\t.reg .b64 rb;\n\t.reg .b32 rt;\n\t" INK_MMA_HEAD
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n\t"
      INK_MMA_TS_STEP(8, 2) INK_MMA_TS_STEP(16, 4) INK_MMA_TS_STEP(24, 6)
      INK_MMA_TS_STEP(32, 1024) INK_MMA_TS_STEP(40, 1026) INK_MMA_TS_STEP(48, 1028)
      INK_MMA_TS_STEP(56, 1030) "}" ::"r"(d),
      "r"(a), "l"(b), "n"(kIdesc), "r"(acc)
      : "memory");
}
// A in TMEM, B MN-major in shared memory (O += P V: P in TMEM, V rows = keys).
template <uint32_t kIdesc>
__device__ __forceinline__ void mma8_ts_mnmajor(uint32_t d, uint32_t a, uint64_t b, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred pe, pa, pt;\n\t.reg .b64 rb;\n\t.reg .b32 rt;\n\t" INK_MMA_HEAD
      "@pe tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, pa;\n\t"
      INK_MMA_TS_STEP(8, 128) INK_MMA_TS_STEP(16, 256) INK_MMA_TS_STEP(24, 384)
      INK_MMA_TS_STEP(32, 512) INK_MMA_TS_STEP(40, 640) INK_MMA_TS_STEP(48, 768)
      INK_MMA_TS_STEP(56, 896) "}" ::"r"(d),
      "r"(a), "l"(b), "n"(kIdesc), "r"(acc)
      : "memory");
}
#undef INK_MMA_SS_STEP
#undef INK_MMA_TS_STEP
#undef INK_MMA_HEAD
// The commit for MMAs issued by the lane that elect.sync picks in a converged warp (the
// issue blocks of the attention kernels): the same full-mask election picks the same lane,
// so the commit tracks those MMAs.  Called by every lane of the warp.
__device__ __forceinline__ void umma_commit_elected(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

#define INK_R8(o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), \
                  "=r"(r[o + 4]), "=r"(r[o + 5]), "=r"(r[o + 6]), "=r"(r[o + 7])
#define INK_W8(o) "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), \
                  "r"(r[o + 4]), "r"(r[o + 5]), "r"(r[o + 6]), "r"(r[o + 7])

// Warp-collective: thread i gets lane (taddr.lane + i), 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
      "[%32];"
      : INK_R8(0), INK_R8(8), INK_R8(16), INK_R8(24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      INK_W8(0), INK_W8(8), INK_W8(16), INK_W8(24)
      : "memory");
}
#undef INK_R8
#undef INK_W8

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Keeps the compiler from using registers written by tcgen05.ld before the wait::ld.
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i])::"memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout a TMA tiled load with
// CU_TENSOR_MAP_SWIZZLE_128B writes).  lbo/sbo in bytes.
//   K-major operand: rows of 128 B (64 bf16 along K), sbo = 1024 (8-row group stride);
//   MN-major operand: rows of 128 B (64 bf16 along M/N) per k, lbo = stride between
//   64-wide M/N blocks, sbo = 1024 (8-k group stride).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, dense.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn_major,
                                                  bool b_mn_major) {
  return (1u << 4)                                  // D = f32
         | (1u << 7)                                // A = bf16
         | (1u << 10)                               // B = bf16
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The same with f16 A and B (a_type = b_type = 0).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)  // D = f32
         | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three floats in one instruction (sm_100+)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Four floats to four E4M3 bytes (round to nearest even, saturating at +-448); a lands
// in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}
// Two E4M3 bytes (x's low byte first) to two f16 in one word, low half first; exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t x) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(x));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  // cvt packs its first source into the upper half
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }
__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }


// Keys at or past the end of a sequence live in cache slots nobody wrote: zero rows
// r0..127 of a staged 128-row K or V page (two 64-wide d halves of 128-byte rows, 16 KB
// apart) so that no stale NaN reaches an MMA.  One warp; the generic-proxy stores are
// fenced for the tensor core's async-proxy reads.
__device__ __forceinline__ void zero_tail_rows(uint8_t (*page)[16384], int r0, int lane) {
  const int chunks = (128 - r0) * 8;  // 16-byte chunks per d half
  for (int c = lane; c < 2 * chunks; c += 32) {
    const int half = c / chunks, cc = c % chunks;
    *reinterpret_cast<uint4*>(page[half] + (size_t)(r0 + cc / 8) * 128 + (cc % 8) * 16) =
        make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncwarp();
}

}  // namespace ink
