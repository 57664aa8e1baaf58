// kda_sm100.cuh -- inline-PTX building blocks for the sm_103a tensor-core path:
// mbarriers with bounded waits, 1-D bulk async copies, TMEM allocation and
// loads/stores, tcgen05.mma (kind::f16, bf16 operands, fp32 accumulate) and the
// shared-memory matrix descriptors of the 128-byte-swizzled K-major layout.
//
// Operand layout used throughout ("SW128 K-major"): a tile of R rows and K
// bf16 columns is stored as K/64 column blocks of R x 128 bytes; row r of a
// block starts at r*128 and its eight 16-byte chunks are permuted by
// chunk ^ (r % 8).  Tiles start 1024-byte aligned, so the swizzle phase equals
// r % 8.  A descriptor covers one K=16 step: start = block base + 32*step,
// stride between 8-row groups (SBO) = 1024 bytes.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_internal.cuh"

namespace kda {
namespace sm100 {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s: a bounded wait gives up after this

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// Waits for the phase with the given parity to complete.  Returns false (and
// records kDevErrTimeout in *err) if it has not after `timeout_ns`.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* err,
                                          uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > timeout_ns) {
      if (err) atomicExch(err, kDevErrTimeout);
      return false;
    }
  }
}

// mbar_wait for a CTA whose threads wait on different barriers: a wait also ends
// (returning false) as soon as another thread of the CTA has raised *abort_flag,
// and a wait that runs out raises it, so that every waiting thread of the CTA
// stops within a few polls of the first one that gives up.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, int* err,
                                              volatile int* abort_flag,
                                              uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        if (err) atomicExch(err, kDevErrTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

// --------------------------------------------------------------- bulk copies
// 1-D bulk copy global -> shared, completing `bytes` of transaction on `bar`.
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// 3-D tiled tensor copy global -> shared (TMA) described by `tmap` (a
// __grid_constant__ CUtensorMap kernel parameter) at coordinates (x, y, z),
// innermost first; completes the box's bytes on `bar`.  Out-of-range elements
// are filled with zeros.  x * element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// Warms L2 with the same box a tma_load_3d at these coordinates would copy.
__device__ __forceinline__ void tma_prefetch_l2_3d(const void* tmap, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// 1-D bulk copy shared -> global in the calling thread's bulk group.
// src, dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// The calling thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// All but the calling thread's most recently committed bulk group have finished
// reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_last() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// The calling thread's committed bulk stores are complete.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// L2 eviction priorities for the cache-hinted copies below: lines a copy touches
// with an evict-first policy are the first candidates for eviction (data read or
// written once), evict-last the last (data wanted again soon).
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// tma_load_3d, tma_prefetch_l2_3d and bulk_s2g with an L2 policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y,
                                                 int z, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d_hint(const void* tmap, int x, int y, int z,
                                                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.3d.L2.global.tile.L2::cache_hint [%0, {%1, %2, %3}], %4;" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_s2g_hint(void* dst, uint32_t src, uint32_t bytes,
                                              uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                   dst),
               "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}

// ------------------------------------------------------- named barriers
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Arrives at barrier `id` (over `nthreads` threads) without waiting: the producer
// half of a producer/consumer hand-off whose consumers call named_sync.
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier `id` over `nthreads` threads that also ANDs `p` across them.
__device__ __forceinline__ bool named_sync_and(uint32_t id, uint32_t nthreads, bool p) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred a, b;\n\t"
      "setp.ne.u32 a, %1, 0;\n\t"
      "bar.red.and.pred b, %2, %3, a;\n\t"
      "selp.u32 %0, 1, 0, b;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)p), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// ----------------------------------------------------------------- fences
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 32-byte global store (8 consecutive fp32; p must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(float* p, const float* v) {
  asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]),
               "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------- TMEM
// Warp-collective: allocates `ncols` (power of two >= 32) TMEM columns and writes
// the base address to shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// 32 lanes x 32 columns of 32-bit: thread i of the warp gets lane (base lane + i),
// columns col .. col+31.  Warp w may only address lanes 32*(w%4) .. +31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// -------------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, SW128 K-major (see the header comment).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);       // start address
  d |= (uint64_t)1 << 16;                         // leading byte offset (unused here): 16 B
  d |= (uint64_t)(1024u >> 4) << 32;              // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                         // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                         // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T for one K=16 step.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T for one K=16 step.  A (M=128 rows = lanes) holds
// bf16 pairs packed along K in 32-bit columns: 8 columns per K step.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor: kind::tf32 (fp32 operands used at tf32 precision, fp32 D),
// operand majorness as idesc_bf16_mn.
__host__ __device__ constexpr uint32_t idesc_tf32_mn(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T for one K=8 step of kind::tf32.  A (M=128 rows =
// lanes) holds one fp32 element per 32-bit column: 8 columns per K step.  B is a
// K-major SW128 tile of fp32 (32 elements per 128-byte row), so a K step is 32 bytes
// as for bf16.
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 lanes x 16 columns store (16 registers per thread).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}
// 32 lanes x 4 columns of 32-bit (one 16-byte piece per thread).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint4 v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ void tmem_st32u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
      "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
      "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Arrives (once) on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Issues the K/16 steps of D (+)= A * B^T where A (M rows) and B (N rows) are SW128
// K-major tiles with `a_rows` / `b_rows` rows per column block (the block stride is
// rows * 128 bytes) and the operands start at row offsets already folded into the
// base addresses.
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_base, int a_rows,
                                         uint32_t b_base, int b_rows, int K, uint32_t idesc,
                                         bool accumulate) {
#pragma unroll 1
  for (int s = 0; s < K / 16; ++s) {
    const uint32_t koff = (uint32_t)((s >> 2) * 0) + (uint32_t)((s & 3) * 32);
    const uint32_t a = a_base + (uint32_t)(s >> 2) * (uint32_t)a_rows * 128u + koff;
    const uint32_t b = b_base + (uint32_t)(s >> 2) * (uint32_t)b_rows * 128u + koff;
    mma_bf16(d_tmem, desc_sw128(a), desc_sw128(b), idesc, (accumulate || s > 0) ? 1u : 0u);
  }
}

// Byte offset of element (row, col) in an SW128 K-major tile with `rows` rows per
// column block.
__host__ __device__ __forceinline__ uint32_t sw128_offset(int rows, int row, int col) {
  const int kb = col >> 6, w = col & 63;
  return (uint32_t)(kb * rows * 128 + row * 128 + ((((w >> 3) ^ (row & 7)) << 4) | ((w & 7) << 1)));
}
// Byte offset of the 16-byte chunk holding columns 8*ch .. 8*ch+7 of `row`.
__host__ __device__ __forceinline__ uint32_t sw128_chunk(int rows, int row, int ch) {
  const int kb = ch >> 3, w = ch & 7;
  return (uint32_t)(kb * rows * 128 + row * 128 + ((w ^ (row & 7)) << 4));
}

// ---- MN-major SW128 tiles ------------------------------------------------
// A tile whose M (or N) extent X is a multiple of 64 and whose K extent is a
// multiple of 8: 1024-byte atoms of 8 K-rows x 64 X-elements (128 bytes per
// K-row, 16-byte chunks permuted by chunk ^ (k % 8)); atoms along X are 1024
// bytes apart (LBO), groups of 8 K-rows are (X/64)*1024 bytes apart (SBO).  A
// thread that owns one K index writes its run of X contiguously.
__host__ __device__ __forceinline__ uint32_t mn_sbo(int X) { return (uint32_t)(X >> 6) * 1024u; }
__host__ __device__ __forceinline__ uint32_t mn_offset(int X, int x, int k) {
  return (uint32_t)((x >> 6) * 1024) + (uint32_t)(k >> 3) * mn_sbo(X) + (uint32_t)((k & 7) * 128) +
         (uint32_t)(((((x & 63) >> 3) ^ (k & 7)) << 4) | ((x & 7) << 1));
}
// 16-byte chunk holding X elements 8*xc .. 8*xc+7 of K-row k.
__host__ __device__ __forceinline__ uint32_t mn_chunk(int X, int xc, int k) {
  return (uint32_t)((xc >> 3) * 1024) + (uint32_t)(k >> 3) * mn_sbo(X) + (uint32_t)((k & 7) * 128) +
         (uint32_t)(((xc & 7) ^ (k & 7)) << 4);
}

__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Descriptor of K step s (16 elements of K) of a K-major tile with `rows` rows per
// 64-column block, starting at `base`.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int rows, int s) {
  return make_desc(base + (uint32_t)(s >> 2) * (uint32_t)rows * 128u + (uint32_t)(s & 3) * 32u, 16u,
                   1024u);
}
// The descriptor `d` with its start address advanced by `bytes` (a multiple of 16
// that keeps the address inside shared memory, so the 14-bit field cannot carry).
__device__ __forceinline__ uint64_t desc_advance(uint64_t d, uint32_t bytes) {
  return d + (uint64_t)(bytes >> 4);
}
// Descriptor of K step s of an MN-major tile with SBO `sbo`, starting at `base`.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, uint32_t sbo, int s) {
  return make_desc(base + (uint32_t)s * 2u * sbo, 1024u, sbo);
}
// Same, with an explicit stride `lbo` between the 64-wide MN atoms.
__device__ __forceinline__ uint64_t mnmajor_desc_lbo(uint32_t base, uint32_t lbo, uint32_t sbo,
                                                     int s) {
  return make_desc(base + (uint32_t)s * 2u * sbo, lbo, sbo);
}
// Instruction descriptor with operand majorness (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t idesc_bf16_mn(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// 2^x with the hardware's approximate base-2 exponential (ex2.approx).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

}  // namespace sm100
}  // namespace kda
