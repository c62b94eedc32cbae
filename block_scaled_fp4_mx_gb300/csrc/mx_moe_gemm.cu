// mx_moe_gemm.cu -- MoE expert GEMM with MXFP4 weights decoded into the tensor-core
// B operand (tcgen05, sm_103a).
//
// The consumer the pages' unpack serves: "vllm-project/vllm pull 51583",
// "Motivation" and the comments on the unpack_B loop -- the CPU MoE GEMM
// (ops.fused_experts_cpu with CPUQuantMethod.MXFP4) unpacks a tile of MXFP4
// weights to bf16 and multiplies it with bf16 activations. Here one CTA owns a
// 128 x 128 output tile of one expert: for every 64-wide slice of K it decodes
// the expert's 128 x 64 weight tile (MXFP4 rule of fp4_mx_unpack, in registers)
// straight into shared memory in the 128-byte-swizzled K-major layout the
// tensor core reads, stages the matching 128 x 64 bf16 activation tile beside
// it, and one thread issues four tcgen05.mma kind::f16 (M = 128, N = 128,
// K = 16 each) accumulating in fp32 in tensor memory. The bf16 weights never
// reach HBM: 0.53 bytes per weight are read instead of 2.
//
// Every wait on an mbarrier is bounded: if the tensor core does not signal
// completion within kWaitLimit polls the kernel records FP4_ERR_TIMEOUT in the
// caller's status word, stops issuing work, frees its tensor memory and returns.
#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kThreads = 128;  // 4 warps: one per 32-lane quarter of tensor memory
constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kTileK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr uint32_t kTmemCols = 128;  // fp32 accumulator: one column per output column
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kTileBytes = kTileM * kTileK * 2;  // 16 KiB per operand tile
// shared memory: A tile, B tile, then the mbarrier, tensor-memory address and
// abort flag; +1 KiB to align the tiles to the 1024-byte swizzle atom, padded so
// that at most 4 CTAs (4 x 128 tensor-memory columns) share an SM.
constexpr int kSmemBytes = 56 * 1024;

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
constexpr uint32_t kInstrDesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                ((uint32_t)(kTileN >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);

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

// Bounded wait for phase `phase` of the mbarrier; false when the limit ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, phase)) return true;
    return false;
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kInstrDesc), "r"(accumulate)
        : "memory");
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

// Byte offset of 16-byte chunk `kc` (8 bf16 along K) of row `r` in a tile of
// 128-byte rows with the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t kc) {
    return r * 128u + ((kc ^ (r & 7u)) << 4);
}

__global__ void __launch_bounds__(kThreads)
mx_moe_gemm_kernel(const uint16_t *__restrict__ a, const int64_t *__restrict__ expert_offsets,
                   const uint8_t *__restrict__ w_packed, const uint8_t *__restrict__ w_scales,
                   int64_t max_rows, int64_t total_rows, int32_t n, int32_t k,
                   uint16_t *__restrict__ out, int32_t *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t *tile_a = smem;
    uint8_t *tile_b = smem + kTileBytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + 2 * kTileBytes);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + 2 * kTileBytes + 8);
    volatile uint32_t *abort_flag = reinterpret_cast<uint32_t *>(smem + 2 * kTileBytes + 12);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int expert = blockIdx.z;
    const int n0 = blockIdx.x * kTileN;
    const int64_t m0 = (int64_t)blockIdx.y * kTileM;
    const int64_t row_begin = expert_offsets[expert];
    const int64_t rows = expert_offsets[expert + 1] - row_begin;
    // offsets live on the device: check them here, never read or write past the buffers
    if (row_begin < 0 || rows < 0 || rows > max_rows || row_begin + rows > total_rows) {
        if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicExch(status, FP4_ERR_SHAPE);
        return;
    }
    if (m0 >= rows) return;  // this expert has fewer row tiles than the grid

    const uint8_t *wp = w_packed + (int64_t)expert * n * (k / 2);
    const uint8_t *ws = w_scales + (int64_t)expert * n * (k / 32);
    const uint16_t *ap = a + row_begin * k;

    if (tid == 0) {
        mbar_init(smem_addr(bar), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const uint32_t a_base = smem_addr(tile_a);
    const uint32_t b_base = smem_addr(tile_b);
    uint32_t phase = 0;
    bool ok = true;
    for (int k0 = 0; k0 < k && ok; k0 += kTileK) {
        // activations: 128 rows x 8 chunks of 16 bytes
#pragma unroll
        for (int i = 0; i < (kTileM * 8) / kThreads; ++i) {
            const uint32_t c = tid + i * kThreads;
            const uint32_t r = c >> 3, kc = c & 7u;
            const int64_t gm = m0 + r;
            const int gk = k0 + (int)kc * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (gm < rows && gk < k) v = __ldg(reinterpret_cast<const uint4 *>(ap + gm * k + gk));
            *reinterpret_cast<uint4 *>(tile_a + sw128_offset(r, kc)) = v;
        }
        // weights: 128 rows x 8 words of packed codes, decoded to 8 bf16 each
#pragma unroll
        for (int i = 0; i < (kTileN * 8) / kThreads; ++i) {
            const uint32_t c = tid + i * kThreads;
            const uint32_t r = c >> 3, kc = c & 7u;
            const int gn = n0 + (int)r;
            const int gk = k0 + (int)kc * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (gn < n && gk < k) {
                const uint32_t w =
                    __ldg(reinterpret_cast<const uint32_t *>(wp + (int64_t)gn * (k / 2) + gk / 2));
                const uint32_t e = __ldg(ws + (int64_t)gn * (k / 32) + gk / 32);
                v = mx_decode_word(w, mx_scaled_table(e));
            }
            *reinterpret_cast<uint4 *>(tile_b + sw128_offset(r, kc)) = v;
        }
        // make the generic-proxy shared-memory writes visible to the tensor core
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
                mma_bf16(tmem, kmajor_sw128_desc(a_base + kk * 32),
                         kmajor_sw128_desc(b_base + kk * 32), (k0 > 0 || kk > 0) ? 1u : 0u);
            mma_commit(smem_addr(bar));
        }
        // every thread waits until the tensor core has consumed the tiles
        if (!mbar_wait_bounded(smem_addr(bar), phase)) *abort_flag = 1;
        phase ^= 1u;
        __syncthreads();
        ok = (*abort_flag == 0);
    }
    tc_fence_after();

    if (ok) {
        const int64_t row = m0 + warp * 32 + lane;
        uint16_t *orow = out + (row_begin + row) * n;
#pragma unroll 1
        for (int c0 = 0; c0 < kTileN; c0 += 32) {
            uint32_t acc[32];
            tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c0, acc);
            if (row < rows && n0 + c0 < n) {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + n0 + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 o;
                    o.x = pack_bf16x2_rn(__uint_as_float(acc[8 * q + 0]), __uint_as_float(acc[8 * q + 1]));
                    o.y = pack_bf16x2_rn(__uint_as_float(acc[8 * q + 2]), __uint_as_float(acc[8 * q + 3]));
                    o.z = pack_bf16x2_rn(__uint_as_float(acc[8 * q + 4]), __uint_as_float(acc[8 * q + 5]));
                    o.w = pack_bf16x2_rn(__uint_as_float(acc[8 * q + 6]), __uint_as_float(acc[8 * q + 7]));
                    dst[q] = o;
                }
            }
        }
    } else if (tid == 0) {
        atomicExch(status, FP4_ERR_TIMEOUT);
        // give in-flight tensor-core work a last bounded chance to finish
        mbar_wait_bounded(smem_addr(bar), phase);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

}  // namespace

cudaError_t launch_mx_moe_gemm(const uint16_t *a, const int64_t *expert_offsets, int64_t experts,
                               int64_t max_rows, int64_t total_rows, const uint8_t *w_packed,
                               const uint8_t *w_scales, int64_t n, int64_t k, uint16_t *out,
                               int32_t *status, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (configured_device != device) {
        err = cudaFuncSetAttribute(mx_moe_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   kSmemBytes);
        if (err != cudaSuccess) return err;
        configured_device = device;
    }
    const dim3 grid((unsigned)((n + kTileN - 1) / kTileN),
                    (unsigned)((max_rows + kTileM - 1) / kTileM), (unsigned)experts);
    mx_moe_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
        a, expert_offsets, w_packed, w_scales, max_rows, total_rows, (int32_t)n, (int32_t)k, out,
        status);
    return cudaGetLastError();
}

}  // namespace fp4mx
