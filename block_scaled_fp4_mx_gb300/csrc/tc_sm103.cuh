// tc_sm103.cuh -- small wrappers over the sm_103a tensor-core (tcgen05), TMA and
// mbarrier instructions used by the GEMM kernels (inline PTX).
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cuda_runtime.h>

namespace fp4mx {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle: start address / 16 in bits 0-13, the
// stride between groups of 8 rows (1024 bytes) / 16 in bits 32-45, descriptor
// version 1 in bits 46-47, swizzle mode 2 (128 B) in bits 61-63. The leading
// byte offset is unused for this layout (one swizzle atom along K).
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
           (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B
// bf16 (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N / 8 in bits 17-22, M / 16 in bits 24-28.
template <int M, int N>
__host__ __device__ constexpr uint32_t instr_desc_bf16() {
    static_assert(M == 64 || M == 128, "cta_group::1 M");
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `phase` of the mbarrier (polling); false once about
// 2^29 SM cycles (~0.3 s) have passed without the phase completing. The clock is
// read only after a first poll fails.
constexpr long long kWaitCycles = 1ll << 29;
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase) {
    if (mbar_try_wait(bar, phase)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, phase))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Bounded wait that lets the thread sleep: try_wait with a suspend-time hint
// (1 ms), so a waiting warp does not take issue slots from the warps beside it
// until the phase completes; false after about 2^29 SM cycles (~0.3 s).
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t phase) {
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(phase), "r"(0x100000u)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > kWaitCycles) return false;
    }
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One K slice of MMAs with A in tensor memory, then a commit to `empty_bar`, with
// a non-blocking probe of the next stage's barrier (`next_bar`, phase
// `next_phase`) issued ahead of them so that its latency hides behind the MMA
// issue. Four K = 16 steps: A advances 8 columns and the B descriptor 32 bytes
// (2 in its address field) per step. `accumulate` = 0 overwrites D with the
// first step. Returns whether the probed phase had already completed.
__device__ __forceinline__ uint32_t mma_slice_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                     uint32_t idesc, uint32_t accumulate,
                                                     uint32_t empty_bar, uint32_t next_bar,
                                                     uint32_t next_phase) {
    uint32_t ready;
    asm volatile(
        "{\n\t.reg .pred pr, p0, pt;\n\t.reg .b64 b1, b2, b3;\n\t.reg .b32 a1, a2, a3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 pr, [%7], %8;\n\t"
        "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pt, %5, %5;\n\t"
        "add.u64 b1, %3, 2;\n\tadd.u64 b2, %3, 4;\n\tadd.u64 b3, %3, 6;\n\t"
        "add.u32 a1, %2, 8;\n\tadd.u32 a2, %2, 16;\n\tadd.u32 a3, %2, 24;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a1], b1, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a2], b2, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a3], b3, %4, pt;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(ready)
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(empty_bar),
          "r"(next_bar), "r"(next_phase)
        : "memory");
    return ready;
}

// mma_slice_tmem_a over two 64-wide K sub-slices: eight K = 16 steps, A advancing 8
// columns per step across both, B taking each sub-slice's four steps from its own
// descriptor (b_desc, b2_desc); the same probe of the next stage's barrier and one
// commit to `empty_bar`.
__device__ __forceinline__ uint32_t mma_slice2_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                      uint64_t b2_desc, uint32_t idesc,
                                                      uint32_t accumulate, uint32_t empty_bar,
                                                      uint32_t next_bar, uint32_t next_phase) {
    uint32_t ready;
    asm volatile(
        "{\n\t.reg .pred pr, p0, pt;\n\t.reg .b64 b1, b2, b3, c1, c2, c3;\n\t"
        ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 pr, [%8], %9;\n\t"
        "setp.ne.b32 p0, %6, 0;\n\tsetp.eq.b32 pt, %6, %6;\n\t"
        "add.u64 b1, %3, 2;\n\tadd.u64 b2, %3, 4;\n\tadd.u64 b3, %3, 6;\n\t"
        "add.u64 c1, %4, 2;\n\tadd.u64 c2, %4, 4;\n\tadd.u64 c3, %4, 6;\n\t"
        "add.u32 a1, %2, 8;\n\tadd.u32 a2, %2, 16;\n\tadd.u32 a3, %2, 24;\n\t"
        "add.u32 a4, %2, 32;\n\tadd.u32 a5, %2, 40;\n\tadd.u32 a6, %2, 48;\n\t"
        "add.u32 a7, %2, 56;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %5, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a1], b1, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a2], b2, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a3], b3, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a4], %4, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a5], c1, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a6], c2, %5, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a7], c3, %5, pt;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(ready)
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "l"(b2_desc), "r"(idesc), "r"(accumulate),
          "r"(empty_bar), "r"(next_bar), "r"(next_phase)
        : "memory");
    return ready;
}

// One K slice of MMAs with A in tensor memory (four K = 16 steps: A advances 8
// columns and the B descriptor 32 bytes per step) and a commit to `empty_bar`.
// `accumulate` = 0 overwrites D with the first step.
__device__ __forceinline__ void mma_slice_tmem_a_commit(uint32_t d_tmem, uint32_t a_tmem,
                                                        uint64_t b_desc, uint32_t idesc,
                                                        uint32_t accumulate, uint32_t empty_bar) {
    asm volatile(
        "{\n\t.reg .pred p0, pt;\n\t.reg .b64 b1, b2, b3;\n\t.reg .b32 a1, a2, a3;\n\t"
        "setp.ne.b32 p0, %4, 0;\n\tsetp.eq.b32 pt, %4, %4;\n\t"
        "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, pt;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];\n\t}"
        :
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(empty_bar)
        : "memory");
}

// Two 64-wide K sub-slices of MMAs with A in tensor memory (eight K = 16 steps: A
// advances 8 columns per step across both sub-slices; B takes the four steps of each
// sub-slice from its own descriptor, b_desc and b2_desc) and one commit to
// `empty_bar`. `accumulate` = 0 overwrites D with the first step.
__device__ __forceinline__ void mma_slice2_tmem_a_commit(uint32_t d_tmem, uint32_t a_tmem,
                                                         uint64_t b_desc, uint64_t b2_desc,
                                                         uint32_t idesc, uint32_t accumulate,
                                                         uint32_t empty_bar) {
    asm volatile(
        "{\n\t.reg .pred p0, pt;\n\t.reg .b64 b1, b2, b3, c1, c2, c3;\n\t"
        ".reg .b32 a1, a2, a3, a4, a5, a6, a7;\n\t"
        "setp.ne.b32 p0, %5, 0;\n\tsetp.eq.b32 pt, %5, %5;\n\t"
        "add.u64 b1, %2, 2;\n\tadd.u64 b2, %2, 4;\n\tadd.u64 b3, %2, 6;\n\t"
        "add.u64 c1, %3, 2;\n\tadd.u64 c2, %3, 4;\n\tadd.u64 c3, %3, 6;\n\t"
        "add.u32 a1, %1, 8;\n\tadd.u32 a2, %1, 16;\n\tadd.u32 a3, %1, 24;\n\t"
        "add.u32 a4, %1, 32;\n\tadd.u32 a5, %1, 40;\n\tadd.u32 a6, %1, 48;\n\t"
        "add.u32 a7, %1, 56;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], %3, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], c1, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], c2, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], c3, %4, pt;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
        :
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "l"(b2_desc), "r"(idesc), "r"(accumulate),
          "r"(empty_bar)
        : "memory");
}

// The single-tile slice of mma_slice_tmem_a with a second accumulator: each K step
// also multiplies the same A columns with a second B operand (`b2_desc`, e.g. the
// activation rows past the first N) into `d2_tmem` with its own instruction
// descriptor `idesc2` (a smaller N).
__device__ __forceinline__ uint32_t mma_slice_tmem_a_ext(uint32_t d_tmem, uint32_t a_tmem,
                                                         uint64_t b_desc, uint32_t idesc,
                                                         uint32_t d2_tmem, uint64_t b2_desc,
                                                         uint32_t idesc2, uint32_t accumulate,
                                                         uint32_t empty_bar, uint32_t next_bar,
                                                         uint32_t next_phase) {
    uint32_t ready;
    asm volatile(
        "{\n\t.reg .pred pr, p0, pt;\n\t.reg .b64 b1, b2, b3, c1, c2, c3;\n\t.reg .b32 a1, a2, a3;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 pr, [%10], %11;\n\t"
        "setp.ne.b32 p0, %8, 0;\n\tsetp.eq.b32 pt, %8, %8;\n\t"
        "add.u64 b1, %3, 2;\n\tadd.u64 b2, %3, 4;\n\tadd.u64 b3, %3, 6;\n\t"
        "add.u64 c1, %6, 2;\n\tadd.u64 c2, %6, 4;\n\tadd.u64 c3, %6, 6;\n\t"
        "add.u32 a1, %2, 8;\n\tadd.u32 a2, %2, 16;\n\tadd.u32 a3, %2, 24;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [%2], %3, %4, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%5], [%2], %6, %7, p0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a1], b1, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%5], [a1], c1, %7, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a2], b2, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%5], [a2], c2, %7, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%1], [a3], b3, %4, pt;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%5], [a3], c3, %7, pt;\n\t"
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%9];\n\t"
        "selp.u32 %0, 1, 0, pr;\n\t}"
        : "=r"(ready)
        : "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(d2_tmem), "l"(b2_desc),
          "r"(idesc2), "r"(accumulate), "r"(empty_bar), "r"(next_bar), "r"(next_phase)
        : "memory");
    return ready;
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     bar)
                 : "memory");
}

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 16 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from registers; the
// stores are complete once tmem_wait_st() returns.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Read-only global loads issued where they stand in the program (volatile asm
// keeps them ahead of the work that follows), so that prefetched slices really
// are in flight while earlier slices are decoded.
__device__ __forceinline__ uint32_t ldg_early_u8(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// 16-byte store to a shared-memory address.
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// TMA: 2-D tile (x = innermost coordinate in elements, y = row) of the tensor map into shared
// memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}


__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched once through the runtime (no link to libcuda).
inline EncodeTiled tensor_map_encoder() {
    static EncodeTiled fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiled) nullptr;
        return reinterpret_cast<EncodeTiled>(ptr);
    }();
    return fn;
}

}  // namespace fp4mx
