// Device-side building blocks shared by the kernels of libkaio_qkv:
// inline-PTX wrappers for mbarrier, TMA, tcgen05 (UMMA / TMEM) and
// mma.sync, bounded waits, and the INT4 -> f16 dequantisation primitives.
//
// Target: sm_103a only (tcgen05 and TMEM need the arch-specific 'a' target).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace kaio {

// ---------------------------------------------------------------------------
// Device error word. Each translation unit that launches kernels owns one
// (file-scope, internal linkage) and reports it through the host API. Bits:
constexpr unsigned kDevErrTimeout = 1u;      // a bounded wait gave up
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s per wait

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// First 1024-byte-aligned address at or after p (p in shared memory). The
// offset is added to p itself, so the compiler still knows the result points
// into shared memory and emits shared-memory loads and stores through it
// (rounding the address through an integer would make them generic accesses).
__device__ __forceinline__ unsigned char* align_smem_1024(unsigned char* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

__device__ __forceinline__ bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// ---------------------------------------------------------------------------
// mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking check of a phase (acquire when it reports completion). Used to
// look one stage ahead: its latency overlaps work issued after it.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: a thread whose phase has not completed is
// suspended (it stops taking issue slots from the warps doing work) until the
// phase completes or about `ns` nanoseconds pass.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete. Never waits forever: after
// kWaitLimitNs, or as soon as another warp of the CTA has raised `abort`, it
// records the failure and returns false so that the caller can wind down.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          unsigned* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    // The abort flag and the clock are looked at every 64th try only: a try
    // that fails costs the waiting warp a few instructions, and waiting warps
    // share their scheduler with warps doing the dequant arithmetic.
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, kDevErrTimeout);
        return false;
      }
    }
  }
}

// mbar_wait with a per-launch limit. At the normal limit (kWaitLimitNs) it is
// mbar_wait. A shorter limit (a test of the timeout path) polls without
// blocking, so that the limit, not the phase's completion, ends an unfinished
// wait: the first poll that finds the phase incomplete after `limit_ns` gives up.
__device__ __forceinline__ bool mbar_wait_lim(uint64_t* bar, uint32_t parity, volatile int* abort,
                                              unsigned* err, uint64_t limit_ns) {
  if (limit_ns >= kWaitLimitNs) return mbar_wait(bar, parity, abort, err);
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_test_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 >= limit_ns) {
      *abort = 1;
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// Wind-down wait: like mbar_wait but ignores the abort flag (used to let
// copies or MMAs already in flight finish before the CTA frees its resources).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, unsigned* err) {
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start before the previous kernel in its stream has
// finished; grid_dependency_wait() returns once that kernel has completed and
// its memory operations are visible, so every thread runs it before its first
// global-memory access. allow_dependents_launch() lets the next such kernel
// start its CTAs (on free SMs) once every CTA of this grid has signalled.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA (tiled tensor copies global -> shared, completion on an mbarrier)
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// Bring one 2-D box of a tensor into L2 (no shared memory, no barrier). A
// performance hint only: it loads nothing into the SM, so it may run before
// the dependency wait on a preceding kernel -- L2 is the point of coherence,
// and a later write by that kernel updates the cached line.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int c0, int c1) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(c0),
               "r"(c1)
               : "memory");
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// tcgen05.mma kind::f16, A from TMEM, B descriptor given as two 32-bit halves.
__device__ __forceinline__ void umma_ts_lohi(uint32_t d, uint32_t a, uint32_t lo, uint32_t hi,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\tsetp.ne.b32 p, %5, 0;\n\tmov.b64 bd, {%2, %3};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d),
      "r"(a), "r"(lo), "r"(hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns -> 32 registers per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// 32 lanes x 4 consecutive 32-bit columns -> 4 registers per thread.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
// 32 lanes x 8 consecutive 32-bit columns -> 8 registers per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 lanes x 8 consecutive 32-bit columns <- 8 registers per thread.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}
// 32 lanes x 16 consecutive 32-bit columns <- 16 registers per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns <- 32 registers per thread.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a tcgen05 operand stored with the
// 128-byte swizzle (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
// Fields: start address >> 4 [0,14), leading-dimension byte offset >> 4
// [16,30), stride-dimension byte offset >> 4 [32,46), descriptor version 1 at
// [46,48), base offset 0 (atoms are 1024-byte aligned), swizzle mode 2
// (128-byte) at [61,64).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16 with f16 A/B and f32 D.
// Bits: D format [4,6) = 1 (f32); A format [7,10) = 0 (f16); B format
// [10,13) = 0 (f16); A major [15] and B major [16] (0 = K-major, 1 = MN-major);
// N >> 3 at [17,23); M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn, bool b_mn) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// ---------------------------------------------------------------------------
// INT4 -> f16 dequantisation.
//
// Packed word P holds eight signed two's-complement nibbles; nibble i (bits
// 4i..4i+3) is K-row 8r+i. The dequantised weight is RN_f16(n * s): the
// nibble n is first built as an exact f16 integer, then one correctly-rounded
// f16 multiply by the group scale s gives RN_f16(n * s) bit for bit.
//
// Building n exactly without a conversion instruction: put the nibble, with
// its sign bit flipped (u' = n + 8 in 0..15), into the low mantissa bits of
// a constant f16 and subtract the constant's value plus 8:
//   nibble at mantissa bits 0..3 under exponent 2^10  -> 1024 + u'  (- 1032)
//   nibble at mantissa bits 4..7 under exponent 2^6   ->   64 + u'  (-   72)
// Mask, sign flip and exponent are one LOP3: (word & mask) ^ magic, where the
// magic holds the exponent bits and the flipped sign position.

// (a & kMask) ^ magic as one three-input logic instruction (truth table 0x6A).
// Written out because, left to itself, the compiler spends two logic
// instructions on this expression when both constants are literals.
template <uint32_t kMask>
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t magic) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "n"(kMask), "r"(magic));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_rn(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// f16 constants (bit patterns): 1032.0 = 0x6408, 72.0 = 0x5480.
constexpr uint32_t kLoMask = 0x000F000Fu, kLoMagic = 0x64086408u;  // (lo, hi) both bits 0..3
constexpr uint32_t kHiMask = 0x00F000F0u, kHiMagic = 0x54805480u;  // both bits 4..7
constexpr uint32_t kMixMask = 0x00F0000Fu, kMixMagic = 0x54806408u; // lo bits 0..3, hi bits 20..23

// "Paired" order, used by the register-fragment decode path: pair j (0..3)
// is the f16x2 {n_j, n_(j+4)} (low half = nibble j), scaled by s2 = {s, s}.
// Costs one shift per word plus three ops per pair.
struct PairedNibbles {
  uint32_t w, w8;
  __device__ __forceinline__ explicit PairedNibbles(uint32_t word) : w(word), w8(word >> 8) {}
  __device__ __forceinline__ uint32_t pair(int j, uint32_t s2) const {
    const uint32_t src = (j & 2) ? w8 : w;
    const uint32_t mag = (j & 1) ? kHiMagic : kLoMagic;
    const uint32_t v = (j & 1) ? and_xor<kHiMask>(src, kHiMagic) : and_xor<kLoMask>(src, kLoMagic);
    return hmul2_rn(hsub2_rn(v, mag), s2);
  }
};

// "Natural" order, used where the consumer wants K-rows in memory order
// (tensor-core operand tiles): output word c (0..3) is {n_2c, n_2c+1}.
// A byte permute puts byte c/... of the word into bytes 0 and 2 so that the
// even nibble sits at bits 0..3 and the odd one at bits 20..23.
__device__ __forceinline__ void dequant_natural(uint32_t word, uint32_t s2, uint32_t (&out)[4]) {
  const uint32_t b01 = prmt(word, 0u, 0x1010u);  // bytes {0,1,0,1}
  const uint32_t b10 = prmt(word, 0u, 0x0101u);  // bytes {1,0,1,0}
  const uint32_t b23 = prmt(word, 0u, 0x3232u);  // bytes {2,3,2,3}
  const uint32_t b32 = prmt(word, 0u, 0x2323u);  // bytes {3,2,3,2}
  out[0] = hmul2_rn(hsub2_rn(and_xor<kMixMask>(b01, kMixMagic), kMixMagic), s2);  // n0, n1
  out[1] = hmul2_rn(hsub2_rn(and_xor<kMixMask>(b10, kMixMagic), kMixMagic), s2);  // n2, n3
  out[2] = hmul2_rn(hsub2_rn(and_xor<kMixMask>(b23, kMixMagic), kMixMagic), s2);  // n4, n5
  out[3] = hmul2_rn(hsub2_rn(and_xor<kMixMask>(b32, kMixMagic), kMixMagic), s2);  // n6, n7
}

// K order inside a 16-byte chunk of staged f16 activations (8 K values) changed
// from (0..7) to (0,4,1,5,2,6,3,7), the order in which PairedNibbles yields a
// packed word's weights: a tensor-core operand pair and its activations must
// agree on the K order, and a chunk's 16 bytes stay together under the 128-byte
// swizzle, so the permutation is done in place wherever the chunk sits.
__device__ __forceinline__ void permute_x_chunk(unsigned char* p) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  uint4 o;
  o.x = __byte_perm(v.x, v.z, 0x5410);
  o.y = __byte_perm(v.x, v.z, 0x7632);
  o.z = __byte_perm(v.y, v.w, 0x5410);
  o.w = __byte_perm(v.y, v.w, 0x7632);
  *reinterpret_cast<uint4*>(p) = o;
}

// ---------------------------------------------------------------------------
// INT8 -> f16, exact (every int8 value is an f16 integer).
//
// Packed word P holds four signed two's-complement bytes; byte i (bits
// 8i..8i+7) is K-row 4r+i. Exponent-bias conversion: flip each byte's sign
// bit (u = b + 128 in 0..255), place u in the low mantissa bits of the f16
// 1024.0 with a byte permute (bit pattern 0x6400 | u, value 1024 + u) and
// subtract 1152 = 1024 + 128 (0x6480), an exact f16 subtraction here.
// lo = {row 4r, row 4r+1}, hi = {row 4r+2, row 4r+3} (K-rows in memory order).
__device__ __forceinline__ void int8x4_to_half2x2(uint32_t word, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = word ^ 0x80808080u;
  lo = hsub2_rn(prmt(u, 0x64646464u, 0x5140u), 0x64806480u);   // bytes {u0, 0x64, u1, 0x64}
  hi = hsub2_rn(prmt(u, 0x64646464u, 0x5342u), 0x64806480u);   // bytes {u2, 0x64, u3, 0x64}
}

__device__ __forceinline__ uint32_t half2_bits(uint16_t lo, uint16_t hi) {
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_map(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 dsmem_ld_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// ---------------------------------------------------------------------------
// CTA pairs on the tensor cores (tcgen05 .cta_group::2). The two CTAs of a
// cluster of two (ranks 0 and 1) issue one MMA of M = 256 rows from rank 0:
// each CTA holds its 128 rows of A and its half of B's N columns in its own
// shared memory, at the same offsets, and its 128 rows of D in its own tensor
// memory. Every tcgen05 allocation, MMA and commit of such a kernel is a pair
// operation; the allocation is made by one warp of each CTA together.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], M = 256 over the pair (rank 0 only).
__device__ __forceinline__ void umma_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once, when every pair MMA issued so far by this thread has completed,
// on the mbarrier at cluster shared-memory address `bar` (this CTA's or the peer's).
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// TMA load into this CTA's shared memory, its bytes counted on the mbarrier at
// cluster address `bar`, which may belong to either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}
// Arrivals on an mbarrier at a cluster address, ordered after this thread's
// earlier memory operations for the whole cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
// mbar_wait for a barrier that CTAs of the cluster arrive on: the acquire
// covers their writes, at cluster scope.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  unsigned* err) {
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicOr(err, kDevErrTimeout);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool mbar_wait_cluster_drain(uint64_t* bar, uint32_t parity, unsigned* err) {
  const uint64_t t0 = globaltimer();
  for (;;) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(err, kDevErrTimeout);
      return false;
    }
  }
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05 operand reads) before signalling the consumer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Named barrier over `count` threads (a multiple of 32), id 1..15.
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// cp.async (global -> shared, 16 bytes, L2 only); src_bytes < 16 zero-fills.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the arrival counts toward the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// Legacy warp-level MMA m16n8k16, f16 inputs, f32 accumulate (register operands).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 128-bit streaming load that does not allocate in L1 (read-once weights).
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace kaio
