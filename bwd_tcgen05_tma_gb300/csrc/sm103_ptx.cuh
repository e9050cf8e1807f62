// Inline-PTX building blocks for sm_103a: mbarriers, TMA tensor loads,
// tcgen05 tensor-memory allocation, MMA issue/commit and TMEM load/store.
//
// Everything here is a thin wrapper over one PTX instruction (or a short fixed
// sequence); the attention kernels compose them.  Every wait is bounded: a
// wait that runs past its limit reports failure to the caller, which records
// an error status and unwinds instead of spinning forever.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#define SM103_DEV __device__ __forceinline__

namespace sm103 {

SM103_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SM103_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
SM103_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

SM103_DEV void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

SM103_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

SM103_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

SM103_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
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

// Non-blocking test of the same condition (try_wait may suspend the thread
// for a while when the phase is not complete; test_wait returns at once).
SM103_DEV bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false
// once `limit_ns` of wall time has passed without completion (the caller then
// records a timeout status and unwinds).  The limit is far above any
// legitimate wait of these kernels.
SM103_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) reads of the same memory.
SM103_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

SM103_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- TMA loads
// Tiled tensor loads into shared memory, completing on an mbarrier
// (transaction bytes).  Coordinates are element indices, innermost first.
SM103_DEV void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}

SM103_DEV void tma_load_3d(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Bulk tensor reduce-add (fp32) from shared memory into global memory, tracked
// by the issuing thread's bulk-async group.
SM103_DEV void tma_reduce_add_3d(const void* map, const void* src, int x, int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(map),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// Bulk tensor store from shared memory (a box in the map's swizzled layout);
// rows past the tensor's extent are not written.  Tracked by the issuing
// thread's bulk-async group.
SM103_DEV void tma_store_4d(const void* map, const void* src, int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(map),
      "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
SM103_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group has finished reading its shared-memory source.
SM103_DEV void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group has completed (global writes done).
SM103_DEV void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

SM103_DEV void prefetch_tensormap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// ---------------------------------------------------------------- TMEM
// Allocation is a whole-warp operation; the base address lands in shared memory.
SM103_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
SM103_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SM103_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SM103_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
SM103_DEV void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- MMA
// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B).  Byte offsets: `lbo` is the stride between
// swizzle atoms along the leading (MN, for MN-major operands) dimension, `sbo`
// the stride between 8-row groups.  Tiles must be 1024-byte aligned.
SM103_DEV uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // swizzle mode: 128-byte
  return d;
}

// Instruction descriptor for kind::f16 with fp32 accumulation; ab_fmt is the
// format of both A and B (0 fp16, 1 bf16; the two are always the same).
// a_mn / b_mn select MN-major (transposed) shared-memory operands.
__host__ __device__ constexpr uint32_t idesc_f32acc(uint32_t ab_fmt, int M, int N, bool a_mn,
                                                    bool b_mn) {
  return (1u << 4)           // D: f32
         | (ab_fmt << 7)     // A
         | (ab_fmt << 10)    // B
         | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- warp-collective MMA issue
// The issuing warp runs its loop converged, on warp-uniform values, and one
// elected lane issues.  All K slices of one GEMM (K = 16 * NK) go out from one
// asm statement whose per-slice operand steps are immediates, so an MMA costs
// a handful of instructions.  With a lone lane issuing one asm per MMA, the
// operands are per-thread values that have to be moved into the uniform
// registers the MMA reads, and next to arithmetic-bound warps on the same
// scheduler that issue slowed to 150-170 clk per 128x128x16 MMA (a probe on
// this GPU); issued this way it stays at the tensor core's 64 clk.
//
// Steps (16-byte units for descriptors, columns for tensor-memory addresses)
// from slice k-1 to slice k, with the period JP of the jumps:
//   K-major 128-byte-swizzled tile of R rows, 64-column chunks R*128 B apart:
//                                          JP 4, S 2, J (R*128 - 96) / 16
//   MN-major 128-byte-swizzled tile (16 rows of 128 B per slice): S = J = 128
//   packed 16-bit pairs in tensor memory, contiguous:              S = J = 8
//   the same in 32-column halves 64 columns apart:   JP 4, S 8, J 40
#define SM103_MMA_F16 "@e tcgen05.mma.cta_group::1.kind::f16 "

// Operand step before K slice k: J when k is a multiple of the period JP
// (a jump to the next 64-column chunk or tensor-memory half), S otherwise.
template <int K, int JP, int S, int J>
__host__ __device__ constexpr int step() {
  return (K % JP == 0) ? J : S;
}

// D[tmem] (+)= A[smem] B[smem] over NK K-slices; the first slice accumulates
// iff `accumulate`, the others always.  Steps: see step().
template <int NK, int JP, int AS, int AJ, int BS, int BJ>
SM103_DEV void mma_ss_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  static_assert(NK == 4 || NK == 8 || NK == 12, "K slices per GEMM");
  if constexpr (NK == 4) {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 alo, ahi, blo, bhi;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b64 {alo, ahi}, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], %1, %2, %3, p0;\n\t"
        "add.u32 alo, alo, %6;\n\tadd.u32 blo, blo, %9;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %7;\n\tadd.u32 blo, blo, %10;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %8;\n\tadd.u32 blo, blo, %11;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>())
        : "memory");
  } else if constexpr (NK == 8) {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 alo, ahi, blo, bhi;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b64 {alo, ahi}, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], %1, %2, %3, p0;\n\t"
        "add.u32 alo, alo, %6;\n\tadd.u32 blo, blo, %13;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %7;\n\tadd.u32 blo, blo, %14;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %8;\n\tadd.u32 blo, blo, %15;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %9;\n\tadd.u32 blo, blo, %16;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %10;\n\tadd.u32 blo, blo, %17;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %11;\n\tadd.u32 blo, blo, %18;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %12;\n\tadd.u32 blo, blo, %19;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()), "n"(step<4, JP, AS, AJ>()), "n"(step<5, JP, AS, AJ>()), "n"(step<6, JP, AS, AJ>()), "n"(step<7, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>()), "n"(step<4, JP, BS, BJ>()), "n"(step<5, JP, BS, BJ>()), "n"(step<6, JP, BS, BJ>()), "n"(step<7, JP, BS, BJ>())
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 alo, ahi, blo, bhi;\n\t.reg .b64 ad, bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b64 {alo, ahi}, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], %1, %2, %3, p0;\n\t"
        "add.u32 alo, alo, %6;\n\tadd.u32 blo, blo, %17;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %7;\n\tadd.u32 blo, blo, %18;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %8;\n\tadd.u32 blo, blo, %19;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %9;\n\tadd.u32 blo, blo, %20;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %10;\n\tadd.u32 blo, blo, %21;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %11;\n\tadd.u32 blo, blo, %22;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %12;\n\tadd.u32 blo, blo, %23;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %13;\n\tadd.u32 blo, blo, %24;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %14;\n\tadd.u32 blo, blo, %25;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %15;\n\tadd.u32 blo, blo, %26;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "add.u32 alo, alo, %16;\n\tadd.u32 blo, blo, %27;\n\t"
        "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], ad, bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()), "n"(step<4, JP, AS, AJ>()), "n"(step<5, JP, AS, AJ>()), "n"(step<6, JP, AS, AJ>()), "n"(step<7, JP, AS, AJ>()), "n"(step<8, JP, AS, AJ>()), "n"(step<9, JP, AS, AJ>()), "n"(step<10, JP, AS, AJ>()), "n"(step<11, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>()), "n"(step<4, JP, BS, BJ>()), "n"(step<5, JP, BS, BJ>()), "n"(step<6, JP, BS, BJ>()), "n"(step<7, JP, BS, BJ>()), "n"(step<8, JP, BS, BJ>()), "n"(step<9, JP, BS, BJ>()), "n"(step<10, JP, BS, BJ>()), "n"(step<11, JP, BS, BJ>())
        : "memory");
  }
}

// kind::f8f6f4 with both operands one 128-byte-swizzled K-major row of 128
// one-byte elements per M / N row: four K slices of 32, 32 bytes apart.
SM103_DEV void mma_f8_ss4_warp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 alo, ahi, blo, bhi;\n\t.reg .b64 ad, bd;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
      "mov.b64 {alo, ahi}, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p0;\n\t"
      "add.u32 alo, alo, 2;\n\tadd.u32 blo, blo, 2;\n\t"
      "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %3, p1;\n\t"
      "add.u32 alo, alo, 2;\n\tadd.u32 blo, blo, 2;\n\t"
      "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %3, p1;\n\t"
      "add.u32 alo, alo, 2;\n\tadd.u32 blo, blo, 2;\n\t"
      "mov.b64 ad, {alo, ahi};\n\tmov.b64 bd, {blo, bhi};\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], ad, bd, %3, p1;\n\t"
      "}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u)
      : "memory");
}

// D[tmem] (+)= A[tmem] B[smem] over NK K-slices (A: packed 16-bit pairs).
template <int NK, int JP, int AS, int AJ, int BS, int BJ>
SM103_DEV void mma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  static_assert(NK == 4 || NK == 8 || NK == 12, "K slices per GEMM");
  if constexpr (NK == 4) {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 at, blo, bhi;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b32 at, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], [%1], %2, %3, p0;\n\t"
        "add.u32 at, at, %6;\n\tadd.u32 blo, blo, %9;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %7;\n\tadd.u32 blo, blo, %10;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %8;\n\tadd.u32 blo, blo, %11;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>())
        : "memory");
  } else if constexpr (NK == 8) {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 at, blo, bhi;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b32 at, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], [%1], %2, %3, p0;\n\t"
        "add.u32 at, at, %6;\n\tadd.u32 blo, blo, %13;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %7;\n\tadd.u32 blo, blo, %14;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %8;\n\tadd.u32 blo, blo, %15;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %9;\n\tadd.u32 blo, blo, %16;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %10;\n\tadd.u32 blo, blo, %17;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %11;\n\tadd.u32 blo, blo, %18;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %12;\n\tadd.u32 blo, blo, %19;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()), "n"(step<4, JP, AS, AJ>()), "n"(step<5, JP, AS, AJ>()), "n"(step<6, JP, AS, AJ>()), "n"(step<7, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>()), "n"(step<4, JP, BS, BJ>()), "n"(step<5, JP, BS, BJ>()), "n"(step<6, JP, BS, BJ>()), "n"(step<7, JP, BS, BJ>())
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred e, p0, p1;\n\t.reg .b32 at, blo, bhi;\n\t.reg .b64 bd;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.ne.b32 p1, %5, 0;\n\t"
        "mov.b32 at, %1;\n\tmov.b64 {blo, bhi}, %2;\n\t"
        SM103_MMA_F16 "[%0], [%1], %2, %3, p0;\n\t"
        "add.u32 at, at, %6;\n\tadd.u32 blo, blo, %17;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %7;\n\tadd.u32 blo, blo, %18;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %8;\n\tadd.u32 blo, blo, %19;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %9;\n\tadd.u32 blo, blo, %20;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %10;\n\tadd.u32 blo, blo, %21;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %11;\n\tadd.u32 blo, blo, %22;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %12;\n\tadd.u32 blo, blo, %23;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %13;\n\tadd.u32 blo, blo, %24;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %14;\n\tadd.u32 blo, blo, %25;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %15;\n\tadd.u32 blo, blo, %26;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "add.u32 at, at, %16;\n\tadd.u32 blo, blo, %27;\n\t"
        "mov.b64 bd, {blo, bhi};\n\t" SM103_MMA_F16 "[%0], [at], bd, %3, p1;\n\t"
        "}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(1u),
        "n"(step<1, JP, AS, AJ>()), "n"(step<2, JP, AS, AJ>()), "n"(step<3, JP, AS, AJ>()), "n"(step<4, JP, AS, AJ>()), "n"(step<5, JP, AS, AJ>()), "n"(step<6, JP, AS, AJ>()), "n"(step<7, JP, AS, AJ>()), "n"(step<8, JP, AS, AJ>()), "n"(step<9, JP, AS, AJ>()), "n"(step<10, JP, AS, AJ>()), "n"(step<11, JP, AS, AJ>()),
        "n"(step<1, JP, BS, BJ>()), "n"(step<2, JP, BS, BJ>()), "n"(step<3, JP, BS, BJ>()), "n"(step<4, JP, BS, BJ>()), "n"(step<5, JP, BS, BJ>()), "n"(step<6, JP, BS, BJ>()), "n"(step<7, JP, BS, BJ>()), "n"(step<8, JP, BS, BJ>()), "n"(step<9, JP, BS, BJ>()), "n"(step<10, JP, BS, BJ>()), "n"(step<11, JP, BS, BJ>())
        : "memory");
  }
}

// Arrive on `bar` once every tcgen05 op issued so far by the warp is done;
// issued by the elected lane of a converged warp.
SM103_DEV void mma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Lane 0's value, known to the compiler to be the same in every lane.
SM103_DEV int warp_uniform(int v) { return __shfl_sync(0xffffffffu, v, 0); }
SM103_DEV uint32_t warp_uniform(uint32_t v) { return __shfl_sync(0xffffffffu, v, 0); }

// ---------------------------------------------------------------- TMEM ld/st
// 32x32b shape: thread t of a warp accesses TMEM lane (32 * (warp % 4) + t);
// register k holds column (col + k).
#define SM103_R8(a, o) "=r"(a[o + 0]), "=r"(a[o + 1]), "=r"(a[o + 2]), "=r"(a[o + 3]), \
                       "=r"(a[o + 4]), "=r"(a[o + 5]), "=r"(a[o + 6]), "=r"(a[o + 7])
#define SM103_W8(a, o) "r"(a[o + 0]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), \
                       "r"(a[o + 4]), "r"(a[o + 5]), "r"(a[o + 6]), "r"(a[o + 7])

SM103_DEV void tmem_ld32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : SM103_R8(r, 0), SM103_R8(r, 8)
      : "r"(taddr)
      : "memory");
}

SM103_DEV void tmem_ld32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SM103_R8(r, 0), SM103_R8(r, 8), SM103_R8(r, 16), SM103_R8(r, 24)
      : "r"(taddr)
      : "memory");
}

// tcgen05.ld fills its registers asynchronously: they hold the loaded values
// once tcgen05.wait::ld has returned, but the compiler sees them as set by
// the load itself and is free to move their uses above a wait that does not
// name them.  So the wait takes the loaded registers as operands ("+r"): every
// later use then depends on it.  Further arrays loaded before the same wait
// pass through an empty statement placed after it (volatile statements keep
// their order).
#define SM103_RW8(a, o) "+r"(a[o + 0]), "+r"(a[o + 1]), "+r"(a[o + 2]), "+r"(a[o + 3]), \
                        "+r"(a[o + 4]), "+r"(a[o + 5]), "+r"(a[o + 6]), "+r"(a[o + 7])
SM103_DEV void tmem_ld_wait(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : SM103_RW8(r, 0), SM103_RW8(r, 8)::"memory");
}
SM103_DEV void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : SM103_RW8(r, 0), SM103_RW8(r, 8), SM103_RW8(r, 16), SM103_RW8(r, 24)::"memory");
}
SM103_DEV void tmem_ld_after_wait(uint32_t (&r)[32]) {
  asm volatile("" : SM103_RW8(r, 0), SM103_RW8(r, 8), SM103_RW8(r, 16), SM103_RW8(r, 24)::"memory");
}
SM103_DEV void tmem_ld_wait(uint32_t (&r0)[32], uint32_t (&r1)[32]) {
  tmem_ld_wait(r0);
  tmem_ld_after_wait(r1);
}
template <int N>
SM103_DEV void tmem_ld_wait(uint32_t (&r)[N][32]) {
  tmem_ld_wait(r[0]);
#pragma unroll
  for (int i = 1; i < N; ++i) tmem_ld_after_wait(r[i]);
}

SM103_DEV void tmem_st32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      SM103_W8(r, 0), SM103_W8(r, 8)
      : "memory");
}

SM103_DEV void tmem_st32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      SM103_W8(r, 0), SM103_W8(r, 8), SM103_W8(r, 16), SM103_W8(r, 24)
      : "memory");
}

SM103_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- misc
SM103_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

SM103_DEV void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Warp-uniform bounded wait: every lane waits, and the warp agrees on failure
// so that later .sync.aligned instructions stay convergent.
SM103_DEV bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait(bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// fp16 counterparts of the two above.
SM103_DEV uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
SM103_DEV uint32_t mul_f16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Elementwise product of two packed bf16 pairs, rounded to nearest even.
SM103_DEV uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Per-warpgroup register budgets.  Every warp of a warpgroup executes the
// same call, at the top of its role's code.  A raise waits until lowered
// budgets elsewhere in the CTA have returned enough registers, so callers keep
// the sum of all budgets within the launch's registers per CTA.
template <uint32_t N>
SM103_DEV void regs_lower() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
SM103_DEV void regs_raise() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Programmatic dependent launch.  grid_dep_wait holds the calling thread until
// every grid this one was launched behind has completed and its memory writes
// are visible (a no-op for a grid launched without the attribute);
// grid_dep_launch lets the next grid on the stream be scheduled early.
SM103_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SM103_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Paired fp32 arithmetic: one instruction computes both lanes of a pair, each
// lane rounded exactly as the scalar operation would be.
SM103_DEV float2 fma_f32x2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
SM103_DEV float2 add_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
SM103_DEV float2 sub_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
SM103_DEV float2 mul_f32x2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
// Largest of three values (NaN inputs ignored, as fmaxf does).
SM103_DEV float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

SM103_DEV uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// 32-byte global store (the address must be 32-byte aligned).
SM103_DEV void st_global_v8(void* p, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                            uint32_t a4, uint32_t a5, uint32_t a6, uint32_t a7) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a0),
               "r"(a1), "r"(a2), "r"(a3), "r"(a4), "r"(a5), "r"(a6), "r"(a7)
               : "memory");
}

SM103_DEV void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

SM103_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace sm103
