// Blackwell (sm_103a) tensor-core helpers: tcgen05.mma with operands in shared memory
// and accumulators in Tensor Memory (TMEM), mbarrier completion, TMEM allocation.
//
// Encodings used (checked on GB300 with exact-integer products before use):
//   * shared-memory operand descriptor: start address >> 4 (bits 0-13), leading byte
//     offset >> 4 (16-29), stride byte offset >> 4 (32-45), version 1 (bit 46),
//     swizzle mode 2 = 128-byte swizzle (bits 61-63).  Tiles are 64 rows of 128 bytes,
//     1024-byte aligned, with 16-byte unit u of row r stored at unit u ^ (r & 7).
//     K-major operands: stride byte offset 1024 (eight rows), K steps of 16 elements
//     advance the start address by 32 bytes.  MN-major operands (rows = K): leading and
//     stride byte offsets 1024, K steps advance by 16 rows = 2048 bytes.
//   * instruction descriptor (kind::f16): f32 accumulate (bit 4), bf16 A and B
//     (bits 7, 10), B MN-major (bit 16), N >> 3 at bit 17, M >> 4 at bit 24.
//   * M = 64 accumulator: row r lives in TMEM lane 32 * (r / 16) + r % 16, one 32-bit
//     column per output column; warp w reads its 16 rows with tcgen05.ld.16x256b, which
//     gives thread t rows t/4 and t/4 + 8, columns 2(t%4) and 2(t%4) + 1 of each
//     8-column block (the same fragment as mma.sync's accumulator).
//   * A operand in TMEM (K-major): row r in the same lane as the accumulator's row r for
//     that M (M = 128: lane r), two 16-bit elements per 32-bit column with the even K
//     index in the low half, so a K step of 16 advances the address by 8 columns.
//   * tcgen05.st.16x128b.x4: register 2i of thread t goes to (lane t/4, column
//     4i + t%4), register 2i + 1 to (lane t/4 + 8, column 4i + t%4); with the 16x256b
//     load fragment above, a thread's packed pair from 8-column block n of a row lands
//     in column 4n + t%4, the A-operand position of that pair.
//   * Issue cost: an MMA issued from a one-lane branch costs about 44 cycles of issue,
//     more than an M = 64, N = 64, K = 16 MMA takes in the pipe (about 35); issued by
//     an elected lane of a converged warp it costs less than the pipe time, unless other
//     warps keep the MMA warp's SM sub-partition busy (then about 59 cycles one by one,
//     39 four at a time from one elect: mma4_ss / mma4_ts).
#pragma once

#include <stdint.h>

namespace gca {
namespace tc {

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Descriptors with every field fixed except the start address: desc(addr) = base +
// (addr >> 4) for any shared-memory address (below 256 KB, so no carry leaves the
// 14-bit field).  K steps then add a constant: 2 (32 bytes) for K-major operands, 128
// (2048 bytes) for MN-major ones.
__device__ __forceinline__ uint64_t desc_km(uint32_t addr) { return sdesc(0, 16, 1024) + (addr >> 4); }
__device__ __forceinline__ uint64_t desc_mn(uint32_t addr) { return sdesc(0, 1024, 1024) + (addr >> 4); }
constexpr uint64_t kKStepKm = 2, kKStepMn = 128;

// K-major 64-row tile, K step ks (16 elements).
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t base, int ks) { return sdesc(base + 32 * ks, 16, 1024); }
// MN-major tile (rows = K), K step ks (16 rows).
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t base, int ks) { return sdesc(base + 2048 * ks, 1024, 1024); }

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major ? (1u << 16) : 0u) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// The same MMA issued by one elected lane of a converged warp: every lane of the warp
// executes the call with the same operands.
__device__ __forceinline__ void mma_warp(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// A operand from TMEM (address a_tmem, lane 0 of the operand), B from shared memory.
__device__ __forceinline__ void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
// tcgen05.commit by the same elected lane (elect.sync picks the lowest active lane, so
// the lane that issued the MMAs above).
__device__ __forceinline__ void commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(su32(bar)));
}

// Arrive on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar)));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;"); }

// Bounded wait for phase `parity` of `bar`.  Each try_wait may suspend the thread in
// hardware for a short, implementation-defined time until the phase completes, so a
// waiting thread does not keep re-issuing shared-memory requests.  Returns false if the
// limit ran out (the caller records the timeout and carries on, so that nothing hangs).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = 1u << 21) {
  uint32_t done = 0;
  for (uint32_t it = 0; it < limit; ++it) {
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(su32(bar)), "r"(parity));
    if (done) return true;
  }
  return false;
}

// One probe of phase `parity` of `bar` (try_wait without a suspend-time hint: the thread
// may wait in hardware for a short, implementation-defined time; measured faster to
// resume than with a 1 us hint when the phase completes).
__device__ __forceinline__ bool mbar_try(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(su32(bar)), "r"(parity));
  return done != 0;
}

// Non-blocking test of phase `parity` of `bar` (1 if it has completed).
__device__ __forceinline__ uint32_t mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done)
      : "r"(su32(bar)), "r"(parity));
  return done;
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;"); }
// Make generic-proxy shared-memory writes (st.shared, cp.async) visible to tcgen05.mma.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;"); }

// TMEM allocation by one full warp; the base address lands in *slot.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)), "r"(ncols));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}

// 16 lanes x 8 columns (32-bit) from lane base `taddr`: thread t gets lanes t/4, t/4+8,
// columns 2(t%4), 2(t%4)+1.
__device__ __forceinline__ void ld16x256(uint32_t taddr, float (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x1.b32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
               : "r"(taddr));
}
__device__ __forceinline__ void ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 16 lanes x 16 columns from lane base `taddr` (layout in the header comment).
__device__ __forceinline__ void st16x128_x4(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}
// Store in the 16x256b fragment layout (the inverse of ld16x256).
__device__ __forceinline__ void st16x256(uint32_t taddr, const float (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x1.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "f"(v[0]), "f"(v[1]),
               "f"(v[2]), "f"(v[3])
               : "memory");
}
// 16 lanes x 8 columns (registers 0-3 as in the x4 form, columns 0-7).
__device__ __forceinline__ void st16x128_x2(uint32_t taddr, const uint32_t (&v)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x2.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3])
               : "memory");
}
// Wait for outstanding tcgen05.ld, tied to 8 loaded registers.
__device__ __forceinline__ void ld_wait(float (&v)[2][4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0][0]), "+f"(v[0][1]), "+f"(v[0][2]), "+f"(v[0][3]), "+f"(v[1][0]), "+f"(v[1][1]),
                 "+f"(v[1][2]), "+f"(v[1][3]));
}
__device__ __forceinline__ void st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Wait for outstanding tcgen05.ld and tie the 32 loaded registers to the wait, so that
// the compiler cannot move a use of them above it.
__device__ __forceinline__ void ld_wait(float (&v)[8][4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0][0]),"+f"(v[0][1]),"+f"(v[0][2]),"+f"(v[0][3]),"+f"(v[1][0]),"+f"(v[1][1]),"+f"(v[1][2]),"+f"(v[1][3]),"+f"(v[2][0]),"+f"(v[2][1]),"+f"(v[2][2]),"+f"(v[2][3]),"+f"(v[3][0]),"+f"(v[3][1]),"+f"(v[3][2]),"+f"(v[3][3]),"+f"(v[4][0]),"+f"(v[4][1]),"+f"(v[4][2]),"+f"(v[4][3]),"+f"(v[5][0]),"+f"(v[5][1]),"+f"(v[5][2]),"+f"(v[5][3]),"+f"(v[6][0]),"+f"(v[6][1]),"+f"(v[6][2]),"+f"(v[6][3]),"+f"(v[7][0]),"+f"(v[7][1]),"+f"(v[7][2]),"+f"(v[7][3]));
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// mbarrier arrival that also announces `bytes` of incoming TMA data.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}

// TMA tile load of a 4-D tensor map (innermost coordinate first) into shared memory,
// completing `bytes` on `bar`.  The innermost coordinate must be a multiple of 16 bytes
// (here always 0).
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2, int c3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(su32(bar))
      : "memory");
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// Named CTA barriers (ids 1..15) between a producer and consumers: `arrive` does not
// block, `sync` blocks until `count` threads (a multiple of 32) have arrived.
__device__ __forceinline__ void named_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// 2^x with the hardware approximation (MUFU.EX2, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16), completing
// `bytes` on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// Wait for outstanding tcgen05.ld, tied to 16 loaded registers.
__device__ __forceinline__ void ld_wait(float (&v)[4][4]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0][0]),"+f"(v[0][1]),"+f"(v[0][2]),"+f"(v[0][3]),"+f"(v[1][0]),"+f"(v[1][1]),"+f"(v[1][2]),"+f"(v[1][3]),"+f"(v[2][0]),"+f"(v[2][1]),"+f"(v[2][2]),"+f"(v[2][3]),"+f"(v[3][0]),"+f"(v[3][1]),"+f"(v[3][2]),"+f"(v[3][3]));
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// Plain arrival (count 1) on an mbarrier.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}

}  // namespace tc
}  // namespace gca


namespace gca {
namespace tc {

// Packed pairs of f32 in one 64-bit register (x in the low half) and the paired
// arithmetic of sm_100-class GPUs: one instruction for both halves, each rounded as its
// scalar counterpart.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void uf2(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max(a, b, c) in one instruction.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Four 8 x 8 matrices of 16-bit pairs to shared memory: register i of thread t holds
// row t/4, columns 2(t%4), 2(t%4)+1 of matrix i (the mma.sync accumulator fragment, and
// the tcgen05.ld.16x256b one); thread t gives the address of row t%8 of matrix t/8.
__device__ __forceinline__ void stmatrix_x4(uint32_t saddr, const uint32_t (&r)[4]) {
  asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// ld16x256 repeated along the columns: repetition r reads columns 8r..8r+7 into v[r].
__device__ __forceinline__ void ld16x256_x4(uint32_t taddr, float (&v)[4][4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=f"(v[0][0]), "=f"(v[0][1]), "=f"(v[0][2]), "=f"(v[0][3]), "=f"(v[1][0]), "=f"(v[1][1]), "=f"(v[1][2]),
        "=f"(v[1][3]), "=f"(v[2][0]), "=f"(v[2][1]), "=f"(v[2][2]), "=f"(v[2][3]), "=f"(v[3][0]), "=f"(v[3][1]),
        "=f"(v[3][2]), "=f"(v[3][3])
      : "r"(taddr));
}
__device__ __forceinline__ void ld16x256_x8(uint32_t taddr, float (&v)[8][4]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=f"(v[0][0]), "=f"(v[0][1]), "=f"(v[0][2]), "=f"(v[0][3]), "=f"(v[1][0]), "=f"(v[1][1]), "=f"(v[1][2]),
        "=f"(v[1][3]), "=f"(v[2][0]), "=f"(v[2][1]), "=f"(v[2][2]), "=f"(v[2][3]), "=f"(v[3][0]), "=f"(v[3][1]),
        "=f"(v[3][2]), "=f"(v[3][3]), "=f"(v[4][0]), "=f"(v[4][1]), "=f"(v[4][2]), "=f"(v[4][3]), "=f"(v[5][0]),
        "=f"(v[5][1]), "=f"(v[5][2]), "=f"(v[5][3]), "=f"(v[6][0]), "=f"(v[6][1]), "=f"(v[6][2]), "=f"(v[6][3]),
        "=f"(v[7][0]), "=f"(v[7][1]), "=f"(v[7][2]), "=f"(v[7][3])
      : "r"(taddr));
}

}  // namespace tc
}  // namespace gca

namespace gca {
namespace tc {

// Four MMAs into one accumulator from a single elect.sync (the first takes the accumulate
// flag `acc`, the other three accumulate).  Issued per MMA, the elect, the predicate set-up
// and the 64-bit descriptor arithmetic compete for the issue slots of the MMA warp's SM
// sub-partition with the warps that share it; measured on this GPU with three busy warps
// there, 58.7 cycles per M=64 N=64 K=16 product one by one against 39.1 four at a time
// (34.2 either way on an idle sub-partition).  Descriptors advance by adding to their low
// 32-bit word: the start-address field (bits 0-13, address >> 4) cannot carry for shared-
// memory addresses below 256 KB with these steps.
// A and B from shared memory; MMA i uses a + i ASTEP and b + i BSTEP (units of 16 bytes).
template <uint32_t ASTEP, uint32_t BSTEP>
__device__ __forceinline__ void mma4_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p, t;\n .reg .b32 al, ah, bl, bh, a1, a2, a3, b1, b2, b3;\n"
      " .reg .b64 A1, A2, A3, B1, B2, B3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, 0, 0;\n"
      " mov.b64 {al, ah}, %1;\n mov.b64 {bl, bh}, %2;\n"
      " add.u32 a1, al, %5;\n add.u32 a2, al, %6;\n add.u32 a3, al, %7;\n"
      " add.u32 b1, bl, %8;\n add.u32 b2, bl, %9;\n add.u32 b3, bl, %10;\n"
      " mov.b64 A1, {a1, ah};\n mov.b64 A2, {a2, ah};\n mov.b64 A3, {a3, ah};\n"
      " mov.b64 B1, {b1, bh};\n mov.b64 B2, {b2, bh};\n mov.b64 B3, {b3, bh};\n"
      " elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], A1, B1, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], A2, B2, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], A3, B3, %3, t;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "n"(ASTEP), "n"(2 * ASTEP), "n"(3 * ASTEP), "n"(BSTEP),
      "n"(2 * BSTEP), "n"(3 * BSTEP));
}
// A from TMEM: MMA i reads A at column a + Ai (A0 = 0), B at b + i BSTEP.
template <uint32_t A1, uint32_t A2, uint32_t A3, uint32_t BSTEP>
__device__ __forceinline__ void mma4_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred e, p, t;\n .reg .b32 bl, bh, b1, b2, b3, x1, x2, x3;\n .reg .b64 B1, B2, B3;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, 0, 0;\n"
      " mov.b64 {bl, bh}, %2;\n"
      " add.u32 x1, %1, %5;\n add.u32 x2, %1, %6;\n add.u32 x3, %1, %7;\n"
      " add.u32 b1, bl, %8;\n add.u32 b2, bl, %9;\n add.u32 b3, bl, %10;\n"
      " mov.b64 B1, {b1, bh};\n mov.b64 B2, {b2, bh};\n mov.b64 B3, {b3, bh};\n"
      " elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [x1], B1, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [x2], B2, %3, t;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [x3], B3, %3, t;\n}\n" ::"r"(d),
      "r"(a), "l"(b), "r"(idesc), "r"(acc), "n"(A1), "n"(A2), "n"(A3), "n"(BSTEP), "n"(2 * BSTEP),
      "n"(3 * BSTEP));
}

}  // namespace tc
}  // namespace gca
