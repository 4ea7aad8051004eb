// sm103_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100a/sm_103a) features the
// attention kernels use: mbarrier phases with bounded waits, TMA tiled loads, tensor memory
// (tcgen05.alloc/ld/st) and 5th-generation tensor-core MMAs (tcgen05.mma) with their shared-memory
// and instruction descriptors. Written from the PTX ISA descriptions of these instructions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace falp {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One non-blocking probe of the phase with parity `parity`: true once that phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking poll (never suspends): true once the phase with parity `parity` completed.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Probe with a suspend-time hint: a waiting thread is parked in hardware (it issues nothing) until
// the phase completes or about `hint_ns` nanoseconds pass, so waiting warps do not take issue
// slots from working warps on the same sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), tiled mode, completion on an mbarrier
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Warp-converged forms: every lane executes the call, one elected lane (lane 0) issues.
__device__ __forceinline__ void tma_load_3d_elect(uint32_t dst, const void* tmap, uint32_t bar,
                                                  int x, int y, int z) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar), "r"(bytes)
      : "memory");
}

// Plain (non-tensor) bulk copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on an mbarrier; one elected lane issues.
__device__ __forceinline__ void bulk_load_elect(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      "\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ------------------------------------------------------------------------------------------------
// Tensor memory
// ------------------------------------------------------------------------------------------------
// Whole warp: allocate `ncols` columns (power of two >= 32); the TMEM address is written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
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
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base_lane + i),
// registers r[c] = column (col + c).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// tcgen05.ld of 16 columns that also returns the maximum of the lane's 16 loaded values (f32).
__device__ __forceinline__ float tmem_ld16_max(uint32_t taddr, uint32_t (&r)[16]) {
  float mx;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15}, %16, [%17];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=f"(mx)
      : "r"(taddr)
      : "memory");
  return mx;
}

// tcgen05.ld of 32 columns that also returns the maximum of the lane's 32 loaded values (f32),
// a reduction the load unit performs (sm_103a); the maximum is valid after tcgen05.wait::ld.
__device__ __forceinline__ float tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32]) {
  float mx;
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=f"(mx)
      : "r"(taddr)
      : "memory");
  return mx;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy (TMA, MMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
      : "memory");
}

// 16x32bx2 shapes (two threads per tensor-memory lane): thread t of the warp accesses lane
// (taddr lane) + (t & 15); threads 0-15 use columns [col, col + n), threads 16-31 columns
// [col + kSplit, col + kSplit + n). Established by a GB300 probe for ld, ld.red and st.
#define FALP_OUT32(r)                                                                           \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), \
      "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),  \
      "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), \
      "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), \
      "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define FALP_IN32(r)                                                                            \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),         \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),          \
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),        \
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),        \
      "r"(r[29]), "r"(r[30]), "r"(r[31])
#define FALP_LIST32 \
  "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}"

// 32 columns per thread with, as the second result, this thread's maximum of the 32 values.
template <int kSplit>
__device__ __forceinline__ float tmem_ld32x2_max(uint32_t taddr, uint32_t (&r)[32]) {
  float mx;
  asm volatile("tcgen05.ld.red.sync.aligned.16x32bx2.x32.max.f32 " FALP_LIST32 ", %32, [%33], %34;"
               : FALP_OUT32(r), "=f"(mx)
               : "r"(taddr), "n"(kSplit)
               : "memory");
  return mx;
}
template <int kSplit>
__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x32.b32 " FALP_LIST32 ", [%32], %33;"
               : FALP_OUT32(r)
               : "r"(taddr), "n"(kSplit)
               : "memory");
}
template <int kSplit>
__device__ __forceinline__ void tmem_st32x2(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};"
      ::"r"(taddr), "n"(kSplit), FALP_IN32(r)
      : "memory");
}
template <int kSplit>
__device__ __forceinline__ void tmem_st8x2(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x32bx2.x8.b32 [%0], %1, {%2,%3,%4,%5,%6,%7,%8,%9};"
               ::"r"(taddr), "n"(kSplit), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),
               "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
template <int kSplit>
__device__ __forceinline__ float tmem_ld16x2_max(uint32_t taddr, uint32_t (&r)[16]) {
  float mx;
  asm volatile("tcgen05.ld.red.sync.aligned.16x32bx2.x16.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
               "%10,%11,%12,%13,%14,%15}, %16, [%17], %18;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=f"(mx)
               : "r"(taddr), "n"(kSplit)
               : "memory");
  return mx;
}
template <int kSplit>
__device__ __forceinline__ void tmem_ld8x2(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr), "n"(kSplit)
               : "memory");
}
template <int kSplit>
__device__ __forceinline__ uint32_t tmem_ld1x2(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x1.b32 {%0}, [%1], %2;"
               : "=r"(r)
               : "r"(taddr), "n"(kSplit)
               : "memory");
  return r;
}
template <int kSplit>
__device__ __forceinline__ void tmem_st4x2(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.16x32bx2.x4.b32 [%0], %1, {%2,%3,%4,%5};" ::"r"(taddr),
               "n"(kSplit), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
               : "memory");
}
template <int kSplit>
__device__ __forceinline__ void tmem_st1x2(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.16x32bx2.x1.b32 [%0], %1, {%2};" ::"r"(taddr),
               "n"(kSplit), "r"(v)
               : "memory");
}
#undef FALP_OUT32
#undef FALP_IN32
#undef FALP_LIST32

// tcgen05.cp of a 32-row x 128-bit matrix from shared memory (no-swizzle K-major descriptor:
// row i at byte 16 i when the stride byte offset is 128) into columns [col, col + 4) of lanes
// i, 32 + i, 64 + i and 96 + i (replicated into every lane quarter), as B-side scale factors
// need. Asynchronous, ordered before the issuing thread's later tcgen05.mma; completion is
// tracked by tcgen05.commit like an MMA.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// Warp-converged form: the whole warp executes the call, one elected lane (lane 0, the lane that
// issues the warp's MMAs and commits) issues the copy.
__device__ __forceinline__ void tmem_cp_32x128b_warpx4_elect(uint32_t taddr, uint64_t sdesc) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(sdesc)
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// tcgen05.mma descriptors
// ------------------------------------------------------------------------------------------------
// Shared-memory matrix descriptor, K-major operand staged by TMA with 128-byte swizzling:
// rows of 128 bytes, 8-row groups 1024 bytes apart (stride byte offset), tile base 1024-aligned.
// Fields: [0,14) start>>4, [16,30) leading byte offset>>4 (unused for swizzled K-major),
// [32,46) stride byte offset>>4, [46,49) fixed 0b001, [49,52) base offset, [52] LBO mode,
// [61,64) layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;                 // LBO (ignored): 16 bytes
  d |= static_cast<uint64_t>(1024 >> 4) << 32;         // SBO: 8 rows * 128 bytes
  d |= static_cast<uint64_t>(1) << 46;                 // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;                 // SWIZZLE_128B
  return d;
}

// Shared-memory descriptor, K-major operand without swizzle: core matrices of 8 rows x 16 bytes;
// lbo = byte distance between core matrices along K, sbo = along M/N (0 repeats one group of 8
// rows for every row group), layout code 0.
__device__ __forceinline__ uint64_t sdesc_kmajor_noswz(uint32_t smem_addr, uint32_t lbo,
                                                       uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor for kind::f16 / kind::tf32 / kind::f8f6f4 (dense):
// [4,6) D format (1 = f32), [7,10) A format, [10,13) B format (kind::f8f6f4: 0 = E4M3,
// 1 = E5M2, 5 = E2M1), [15] A major (0 = K), [16] B major (0 = K), [17,23) N>>3, [24,29) M>>4.
__host__ __device__ constexpr uint32_t idesc_f8f6f4(uint32_t M, uint32_t N, uint32_t afmt,
                                                    uint32_t bfmt) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f8f6f4, one CTA.
__device__ __forceinline__ void mma_f8f6f4_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f8f6f4, one CTA (A: lane = row, 4 E4M3 per column).
__device__ __forceinline__ void mma_f8f6f4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-converged forms: the whole warp executes the call with warp-uniform operands (so they
// live in uniform registers) and elect.sync lets exactly one lane (the lowest, lane 0) issue.
__device__ __forceinline__ void mma_f8f6f4_ss_elect(uint32_t d_tmem, uint64_t adesc,
                                                    uint64_t bdesc, uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (F16 or BF16 operands, F32 accumulate).
__device__ __forceinline__ void mma_f16_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f8f6f4_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                    uint64_t bdesc, uint32_t idesc,
                                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One elected lane issues a whole K = 128 contraction of E4M3 operands in shared memory (four
// K = 32 MMAs; each K step moves both K-major descriptors by 32 bytes = 2 in the start-address
// field), the first overwriting D, then the commit of the four to `bar`. One elect.sync per group
// keeps the issuing warp's instruction count (and its cost to the warps it shares a scheduler
// with) low.
__device__ __forceinline__ void mma_f8f6f4_ss_k128_commit_elect(uint32_t d_tmem, uint64_t adesc,
                                                                uint64_t bdesc, uint32_t idesc,
                                                                uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
      "setp.ne.b32 p0, 0, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
      "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a1, b1, %3, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a2, b2, %3, p1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], a3, b3, %3, p1;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%4];\n\t}"
      ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(bar)
      : "memory");
}

// Same for a K = 64 contraction with A (E4M3) in tensor memory: two K = 32 MMAs (A moves by 8
// columns = 32 bytes per row, B by 32 bytes), the first accumulating only if `accumulate`.
__device__ __forceinline__ void mma_f8f6f4_ts_k64_commit_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                               uint64_t bdesc, uint32_t idesc,
                                                               uint32_t accumulate, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b64 b1;\n\t.reg .b32 a1;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\t"
      "add.s32 a1, %1, 8;\n\tadd.s64 b1, %2, 2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %3, p1;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(bar)
      : "memory");
}

// The same, with a second commit to `bar2` when `second` is non-zero (one elect for the group).
__device__ __forceinline__ void mma_f8f6f4_ts_k64_commit2_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                                uint64_t bdesc, uint32_t idesc,
                                                                uint32_t accumulate, uint32_t bar,
                                                                uint32_t second, uint32_t bar2) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1, r;\n\t.reg .b64 b1;\n\t.reg .b32 a1;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 p1, 0, 0;\n\tsetp.ne.b32 r, %6, 0;\n\t"
      "add.s32 a1, %1, 8;\n\tadd.s64 b1, %2, 2;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [a1], b1, %3, p1;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t"
      "and.pred r, r, e;\n\t"
      "@r tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(bar), "r"(second),
        "r"(bar2)
      : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

// Shared-memory descriptor, K-major operand with 64-byte rows staged by TMA with 64-byte
// swizzling: 8-row groups 512 bytes apart, tile base 512-aligned, layout code 4 (SWIZZLE_64B).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw64(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFF) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(512 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(4) << 61;
  return d;
}

// Instruction descriptor for kind::mxf4nvf4 (block-scaled FP4): A and B E2M1 (format code 1),
// scale factors UE4M3 (bit 23 = 0), scale-factor ids 0 (all four 16-element blocks of a K=64
// step), both operands K-major.
__host__ __device__ constexpr uint32_t idesc_mxf4nvf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A B^T with one UE4M3 scale per 16 elements of K (scale_vec::4X). The scale
// factors of one K=64 step occupy 4 tensor-memory columns: row 32c + i in column c; A's in the
// row's own lane quarter (lane 32c + i), B's repeated in every lane quarter (lane i + 32q).
__device__ __forceinline__ void mma_mxf4_ss_elect(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

__device__ __forceinline__ void mma_mxf4_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                                  uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], [%1], %2, %3, "
      "[%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 async operation issued so far by this thread
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ------------------------------------------------------------------------------------------------
// Numeric conversions used by the softmax / quantizers
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 -> two E4M3 (round to nearest even, saturate to +-448); `lo` lands in the low byte.
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two E4M3 (low byte first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t cvt_e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr),
               "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

// One byte of two E2M1 codes (low nibble first) -> f16x2 (exact).
__device__ __forceinline__ uint32_t cvt_e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// Two fp32 -> two E2M1 codes in one byte (round to nearest even, saturate to +-6);
// `lo` lands in the low nibble.
__device__ __forceinline__ uint8_t cvt_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u16.u8 %0, t;\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return static_cast<uint8_t>(r);
}

// Two fp32 -> two E2M1 codes (round to nearest even, saturate to +-6): the code byte (`lo` in the
// low nibble) and the two quantized values back in f16x2 (exact).
__device__ __forceinline__ uint32_t cvt_e2m1x2_and_f16x2(float lo, float hi, uint32_t& h2) {
  uint32_t b;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %2, %3;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, t;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(b), "=r"(h2)
      : "f"(hi), "f"(lo));
  return b;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Three-input maximum (sm_100+).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Row maximum of 64 values: four independent 3-input-max chains, then a combine.
__device__ __forceinline__ float row_max64(const float (&s)[64]) {
  float acc[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    acc[k] = max3f(s[k], s[k + 4], s[k + 8]);
#pragma unroll
    for (int i = 3; i < 15; i += 2) acc[k] = max3f(acc[k], s[k + 4 * i], s[k + 4 * (i + 1)]);
    acc[k] = fmaxf(acc[k], s[k + 60]);
  }
  return fmaxf(max3f(acc[0], acc[1], acc[2]), acc[3]);
}

// (d0, d1) = (a0, a1) * b + c on the packed fp32x2 FMA (one issue slot for two results).
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %4};\n\t"
      "mov.b64 z, {%5, %5};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\t"
      "mov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1) on the packed fp32x2 FMA.
__device__ __forceinline__ void fma2v(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                      float c0, float c1) {
  asm("{\n\t.reg .b64 x, y, z, w;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "mov.b64 z, {%6, %7};\n\t"
      "fma.rn.f32x2 w, x, y, z;\n\t"
      "mov.b64 {%0, %1}, w;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Packed f16x2 fused multiply-add on raw 32-bit registers.
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Packed f16x2 addition on raw 32-bit registers.
__device__ __forceinline__ uint32_t hadd2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

}  // namespace falp
