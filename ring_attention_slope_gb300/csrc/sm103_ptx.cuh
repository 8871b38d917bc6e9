// Inline-PTX building blocks for sm_103a: mbarriers, TMA tensor loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM load/store) and the shared
// memory / instruction descriptors the tensor-core MMAs consume.
//
// Everything here is written from the public PTX ISA description of the
// sm_100-family instructions; no library headers are involved.
#pragma once

#include <cstdint>
#include <cuda.h>

namespace slope {

// ----------------------------------------------------------------- basics

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Like mbar_try_wait, but the thread sleeps in hardware (up to `hint_ns`) until
// the phase completes instead of returning at once: waiting warps stop taking
// issue slots from the warps that do the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// ----------------------------------------------------------------- programmatic dependent launch

// Lets the next kernel of the stream, when it is launched as a programmatic dependent, be
// scheduled as soon as every CTA of this grid has executed this (or exited).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until the grid this one was launched as a programmatic dependent of has completed and
// its memory writes are visible; returns at once for a kernel launched the ordinary way.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled tensor load global -> shared, completion counted in bytes on `bar`.
// Coordinates are in elements, innermost first; out-of-range elements read 0.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled tensor store shared -> global (bulk-group completion).  Coordinates in
// elements, innermost first; elements outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until every committed bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Same, but leaves the most recently committed bulk store pending.
__device__ __forceinline__ void bulk_wait_read_allbut1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Waits until every committed bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Orders this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- tcgen05

// TMEM allocation: executed by one whole warp; the base address lands in smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) = A * B [+ D] on the tensor cores (kind::f16: bf16 operands, fp32 accumulator),
// one instruction issued by one thread.  The 64-bit descriptors are given as (low, high)
// words, so that a caller can keep the high word fixed and step the start address in the
// low word.  mma_ss_lh: A and B in shared memory; mma_ts_lh: A in tensor memory.
__device__ __forceinline__ void mma_ss_lh(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %2};\n\t"
      "mov.b64 db, {%3, %4};\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_ts_lh(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Each thread of the warp reads 32 consecutive 32-bit columns of its own TMEM
// lane (lane = warp's 32-lane quarter + lane id).  Values are valid only after
// tmem_ld_wait(); pass them through reg_fence() after the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// tmem_ld32 that also returns the maximum of the 32 loaded fp32 values of the thread's
// lane (tcgen05.ld.red, max over the columns; -inf elements take part as -inf).  The
// maximum, like the values, is valid only after tmem_ld_wait() and reg_fence().
__device__ __forceinline__ float tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32]) {
  float m;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(m)
      : "r"(taddr)
      : "memory");
  return m;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Compiler-level dependency: values loaded by tcgen05.ld are only consumed
// after this point (place it after tmem_ld_wait()).
template <int N>
__device__ __forceinline__ void reg_fence(uint32_t (&r)[N]) {
#pragma unroll
  for (int i = 0; i < N; ++i) asm volatile("" : "+r"(r[i]));
}
__device__ __forceinline__ void reg_fence(float& x) { asm volatile("" : "+f"(x)); }

// ----------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor (tcgen05 form), kept as two 32-bit words: the start
// address (16-byte units, bits 0-13) and leading byte offset (16-byte units, bits 16-29)
// in the low word; the stride byte offset (bits 32-45), descriptor version 1 (bit 46)
// and the swizzle mode (bits 61-63, 2 = 128-byte swizzle) in the high word.  Tiles are
// 1024-byte aligned so the base-offset field stays 0.
constexpr uint32_t kSwizzle128B = 2;

// Low / high words of the descriptor: the start address lives in bits 0-13 of the low
// word, so adding (byte offset >> 4) to it steps through a tile as long as the address
// stays below 256 KB (always true for shared memory).
__device__ __forceinline__ uint32_t smem_desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t smem_desc_hi(uint32_t sbo_bytes, uint32_t swizzle_mode) {
  return ((sbo_bytes >> 4) & 0x3FFFu) | (1u << 14) | ((swizzle_mode & 7u) << 29);
}

// Instruction descriptor for kind::f16 with bf16 A/B and an fp32 accumulator.
// a_mn / b_mn select MN-major (1) or K-major (0) operands.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(a_mn) << 15)       // A major
         | (static_cast<uint32_t>(b_mn) << 16)       // B major
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ----------------------------------------------------------------- math

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// One pair of softmax elements: x = s * sl2 - m (packed FMA), p = 2^x (two MUFU ops),
// acc += p (packed add, accumulator kept as a 64-bit register pair), and p packed to
// bf16x2 (round to nearest even).  sl2_m holds {sl2, sl2} and neg_m {-m, -m}.
__device__ __forceinline__ uint32_t softmax_pair(float s0, float s1, uint64_t sl2_pair, uint64_t negm_pair,
                                                 uint64_t& acc) {
  uint32_t packed;
  asm("{\n\t.reg .b64 sp, xp, pp;\n\t.reg .f32 x0, x1, p0, p1;\n\t"
      "mov.b64 sp, {%2, %3};\n\t"
      "fma.rn.f32x2 xp, sp, %4, %5;\n\t"
      "mov.b64 {x0, x1}, xp;\n\t"
      "ex2.approx.ftz.f32 p0, x0;\n\t"
      "ex2.approx.ftz.f32 p1, x1;\n\t"
      "mov.b64 pp, {p0, p1};\n\t"
      "add.rn.f32x2 %1, %1, pp;\n\t"
      "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t}"
      : "=r"(packed), "+l"(acc)
      : "f"(s0), "f"(s1), "l"(sl2_pair), "l"(negm_pair));
  return packed;
}
// The same pair with 2^x on the FMA pipe instead of the MUFU unit, so that the kernel can
// move part of its exponentials off the MUFU unit, which bounds the softmax.  2^x is
// reduced Cody-Waite style to 2^n * 2^f: adding 1.5 * 2^23 rounds x to the integer n
// (left in the low mantissa bits of t), f = x - n lies in [-1/2, 1/2], 2^f is a cubic
// 1 + c1 f + c2 f^2 + c3 f^3 fitted for the smallest maximum relative error
// (exp2_poly_fit.py beside this file: 1.0e-4 in float32, far below the 2^-9 of the
// bf16 rounding that follows; c0 = 1, so an integer x gives 2^x exactly), and 2^n is
// added into the exponent field (t << 23 keeps n << 23 exactly, because every set bit
// of 1.5 * 2^23 lies at bit 22 or above).  x is clamped to >= -125 first, so the
// exponent cannot underflow: 2^x for x < -125 (and -inf) comes out as about 2^-125,
// not 0, and a NaN x as 2^-125 too.
// poly holds {c3, c2, c1, c0} as {c, c} pairs; magic is {1.5 * 2^23, 1.5 * 2^23}.
struct Exp2Poly {
  uint64_t magic, c3, c2, c1, c0;
};
__device__ __forceinline__ uint32_t softmax_pair_poly(float s0, float s1, uint64_t sl2_pair, uint64_t negm_pair,
                                                      uint64_t& acc, const Exp2Poly& k) {
  uint32_t packed;
  asm("{\n\t.reg .b64 sp, xp, tp, jp, fp, qp, pp;\n\t.reg .f32 x0, x1, p0, p1;\n\t"
      ".reg .b32 t0, t1, q0, q1, e0, e1;\n\t"
      "mov.b64 sp, {%2, %3};\n\t"
      "fma.rn.f32x2 xp, sp, %4, %5;\n\t"
      "mov.b64 {x0, x1}, xp;\n\t"
      "max.f32 x0, x0, 0fC2FA0000;\n\t"
      "max.f32 x1, x1, 0fC2FA0000;\n\t"
      "mov.b64 xp, {x0, x1};\n\t"
      "add.rn.f32x2 tp, xp, %6;\n\t"
      "sub.rn.f32x2 jp, tp, %6;\n\t"
      "sub.rn.f32x2 fp, xp, jp;\n\t"
      "fma.rn.f32x2 qp, %7, fp, %8;\n\t"
      "fma.rn.f32x2 qp, qp, fp, %9;\n\t"
      "fma.rn.f32x2 qp, qp, fp, %10;\n\t"
      "mov.b64 {t0, t1}, tp;\n\t"
      "mov.b64 {q0, q1}, qp;\n\t"
      "shl.b32 e0, t0, 23;\n\t"
      "shl.b32 e1, t1, 23;\n\t"
      "add.u32 e0, e0, q0;\n\t"
      "add.u32 e1, e1, q1;\n\t"
      "mov.b32 p0, e0;\n\t"
      "mov.b32 p1, e1;\n\t"
      "mov.b64 pp, {p0, p1};\n\t"
      "add.rn.f32x2 %1, %1, pp;\n\t"
      "cvt.rn.bf16x2.f32 %0, p1, p0;\n\t}"
      : "=r"(packed), "+l"(acc)
      : "f"(s0), "f"(s1), "l"(sl2_pair), "l"(negm_pair), "l"(k.magic), "l"(k.c3), "l"(k.c2), "l"(k.c1), "l"(k.c0));
  return packed;
}
// Coefficients printed by exp2_poly_fit.py (float32 bit patterns).
constexpr uint32_t kExp2PolyC0 = 0x3F800000u;  // exactly 1: integer x gives 2^x exactly
constexpr uint32_t kExp2PolyC1 = 0x3F317AFDu;
constexpr uint32_t kExp2PolyC2 = 0x3E780626u;
constexpr uint32_t kExp2PolyC3 = 0x3D61510Bu;
constexpr uint32_t kExp2PolyMagic = 0x4B400000u;  // 1.5 * 2^23
__host__ __device__ constexpr uint64_t splat_bits(uint32_t b) { return (static_cast<uint64_t>(b) << 32) | b; }
__device__ __forceinline__ Exp2Poly exp2_poly_consts() {
  return {splat_bits(kExp2PolyMagic), splat_bits(kExp2PolyC3), splat_bits(kExp2PolyC2), splat_bits(kExp2PolyC1),
          splat_bits(kExp2PolyC0)};
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace slope
