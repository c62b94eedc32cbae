// mx_moe_gemm.cu -- MoE expert GEMM with MXFP4 weights decoded into the tensor-core
// B operand (tcgen05, sm_103a).
//
// The consumer the pages' unpack serves: "vllm-project/vllm pull 51583",
// "Motivation" and the comments on the unpack_B loop -- the CPU MoE GEMM
// (ops.fused_experts_cpu with CPUQuantMethod.MXFP4) unpacks a tile of MXFP4
// weights to bf16 and multiplies it with bf16 activations. Here the bf16 weights
// never reach HBM: 0.53 bytes per weight are read instead of 2.
//
// One CTA owns a 128 x 128 output tile of one expert. The activation tiles and
// the decoded weight tiles run in two separate shared-memory rings over 64-wide
// slices of K, each with full/empty mbarriers:
//   - one thread of the TMA warp keeps kStagesA activation tiles (128 x 64 bf16,
//     cp.async.bulk.tensor with the 128-byte swizzle the tensor core reads) in
//     flight ahead of the tensor core;
//   - 8 decoder warps turn the expert's 128 x 64 MXFP4 weight tile into bf16 in
//     the same swizzled K-major layout: each thread takes one row's 32 codes of a
//     slice (one 16-byte load, one E8M0 byte, one scaled table), with the raw
//     words of its next kAhead slices already in flight in registers; it decodes
//     into registers before waiting for a free weight stage, so only the stores
//     sit between the wait and the warp's single arrival;
//   - one thread of the MMA warp waits for both tiles of a slice, issues four
//     tcgen05.mma kind::f16 (M = 128, N = 128, K = 16) into the fp32 accumulator
//     in tensor memory and commits both stages back to their "empty" barriers.
// The decoder warps then read the accumulator with tcgen05.ld, round to bf16
// and store the tile.
//
// Every wait on an mbarrier is bounded: a wait that runs out records
// FP4_ERR_TIMEOUT in the caller's status word and sets a shared abort flag; all
// roles then stop issuing work, the tensor memory is freed and the CTA returns.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)

#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"

namespace fp4mx {
namespace {

constexpr int kTileM = 128;
constexpr int kTileN = 128;
constexpr int kTileK = 64;  // one 128-byte swizzle atom of bf16 along K
constexpr int kStagesA = 4;      // activation tiles in flight (TMA)
constexpr int kStagesB = 2;      // decoded weight tiles (the raw words run further ahead)
constexpr int kDecodeWarps = 8;  // 2 threads per weight row: 256 threads
constexpr int kTmaWarp = kDecodeWarps;
constexpr int kMmaWarp = kDecodeWarps + 1;
constexpr int kThreads = (kDecodeWarps + 2) * 32;
constexpr int kAhead = 5;        // raw weight slices in flight per decoder thread
constexpr int kRing = kAhead + 1;
constexpr uint32_t kTmemCols = 128;  // fp32 accumulator: one column per output column
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr int kTileBytes = kTileM * kTileK * 2;  // 16 KiB per operand tile and stage
// shared memory: 1 KiB to align the tiles to the 1024-byte swizzle atom, the A
// and B rings, then barriers, the tensor-memory address and the abort flag.
// Two CTAs (2 x 128 tensor-memory columns) fit on an SM.
constexpr int kBarrierOffset = (kStagesA + kStagesB) * kTileBytes;
constexpr int kSmemBytes = 1024 + kBarrierOffset + 256;

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

// Read-only global loads issued where they stand in the program (volatile asm
// keeps them ahead of the work that follows), so that prefetched slices really
// are in flight while earlier slices are decoded.
__device__ __forceinline__ uint4 ldg_early_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_early_u8(const void *p) {
    uint32_t v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// 16-byte store to a shared-memory address (always the shared-state space).
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Byte offset of 16-byte chunk `kc` (8 bf16 along K) of row `r` in a tile of
// 128-byte rows with the 128-byte swizzle (chunk index XOR row mod 8).
__device__ __forceinline__ uint32_t sw128_offset(uint32_t r, uint32_t kc) {
    return r * 128u + ((kc ^ (r & 7u)) << 4);
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// TMA: 2-D tile (x = K offset in elements, y = row) of the tensor map into shared
// memory, completing `bytes` of transaction count on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

struct RawSlice {
    uint4 words;  // 32 packed codes of one weight row (4 words)
    uint32_t e8m0;
};

__global__ void __launch_bounds__(kThreads, 2)
mx_moe_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const int64_t *__restrict__ expert_offsets,
                   const uint8_t *__restrict__ w_packed, const uint8_t *__restrict__ w_scales,
                   int64_t max_rows, int64_t total_rows, int32_t n, int32_t k,
                   uint16_t *__restrict__ out, int32_t *__restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t a_ring = smem_addr(smem);
    const uint32_t b_ring = a_ring + kStagesA * kTileBytes;
    // barriers: full/empty of each A stage, full/empty of each B stage, accumulator
    const uint32_t bars = a_ring + kBarrierOffset;
    auto full_a = [&](int s) { return bars + 8u * s; };
    auto empty_a = [&](int s) { return bars + 8u * (kStagesA + s); };
    auto full_b = [&](int s) { return bars + 8u * (2 * kStagesA + s); };
    auto empty_b = [&](int s) { return bars + 8u * (2 * kStagesA + kStagesB + s); };
    const uint32_t acc_bar = bars + 8u * (2 * kStagesA + 2 * kStagesB);
    uint32_t *tmem_slot =
        reinterpret_cast<uint32_t *>(smem + kBarrierOffset + 8 * (2 * kStagesA + 2 * kStagesB + 1));
    volatile uint32_t *abort_flag = tmem_slot + 1;

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
    const int nk = (k + kTileK - 1) / kTileK;

    if (tid == 0) {
        for (int s = 0; s < kStagesA; ++s) {
            mbar_init(full_a(s), 1);   // the TMA thread's expect_tx arrival
            mbar_init(empty_a(s), 1);  // the MMA commit
        }
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(full_b(s), kDecodeWarps);  // one arrival per decoder warp
            mbar_init(empty_b(s), 1);            // the MMA commit
        }
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
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

    if (warp < kDecodeWarps) {
        // ---- decoder warps: the expert's weights, one K slice after another ----
        const uint32_t r = (uint32_t)tid >> 1;  // weight row of the tile
        const uint32_t h = (uint32_t)tid & 1u;  // which 32 codes of the 64-wide slice
        const int gn = n0 + (int)r;
        const bool row_ok = gn < n;
        const uint8_t *wrow = w_packed + ((int64_t)expert * n + (row_ok ? gn : 0)) * (k / 2) + h * 16;
        const uint8_t *srow = w_scales + ((int64_t)expert * n + (row_ok ? gn : 0)) * (k / 32) + h;
        auto load_raw = [&](int kt) {
            RawSlice raw{make_uint4(0, 0, 0, 0), 127u};
            if (kt < nk && row_ok && kt * kTileK + (int)h * 32 < k) {
                raw.words = ldg_early_v4(wrow + kt * (kTileK / 2));
                raw.e8m0 = ldg_early_u8(srow + kt * (kTileK / 32));
            }
            return raw;
        };
        uint32_t st_off[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) st_off[j] = sw128_offset(r, h * 4 + j);
        RawSlice ring[kRing];
#pragma unroll
        for (int i = 0; i < kAhead; ++i) ring[i] = load_raw(i);
        bool stop = false;
        for (int base = 0; base < nk && !stop; base += kRing) {
#pragma unroll
            for (int j = 0; j < kRing; ++j) {
                const int kt = base + j;
                if (kt >= nk) break;
                const int s = kt % kStagesB;
                const uint32_t use = (uint32_t)(kt / kStagesB);
                ring[(j + kAhead) % kRing] = load_raw(kt + kAhead);
                // decode into registers first: the arithmetic stays off the wait
                const RawSlice cur = ring[j % kRing];
                const ByteTable t = mx_scaled_table(cur.e8m0);
                const uint4 d0 = mx_decode_word(cur.words.x, t);
                const uint4 d1 = mx_decode_word(cur.words.y, t);
                const uint4 d2 = mx_decode_word(cur.words.z, t);
                const uint4 d3 = mx_decode_word(cur.words.w, t);
                // one lane polls for the stage to be free; the warp follows via the vote
                if (kt >= kStagesB && lane == 0 &&
                    !mbar_wait_bounded(empty_b(s), (use - 1u) & 1u))
                    *abort_flag = 1;
                if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) {  // warp-uniform
                    stop = true;
                    break;
                }
                const uint32_t b_tile = b_ring + s * kTileBytes;
                st_shared_v4(b_tile + st_off[0], d0);
                st_shared_v4(b_tile + st_off[1], d1);
                st_shared_v4(b_tile + st_off[2], d2);
                st_shared_v4(b_tile + st_off[3], d3);
                // make this thread's generic-proxy writes visible to the tensor core;
                // after the warp has converged one lane arrives for all 32
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(full_b(s));
            }
        }
    } else if (warp == kTmaWarp && lane == 0) {
        // ---- TMA: activation tiles, kStagesA ahead of the tensor core ----
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kStagesA;
            const uint32_t use = (uint32_t)(kt / kStagesA);
            if (kt >= kStagesA && !mbar_wait_bounded(empty_a(s), (use - 1u) & 1u)) *abort_flag = 1;
            if (*abort_flag) break;
            mbar_arrive_expect_tx(full_a(s), kTileBytes);
            tma_load_2d(a_ring + s * kTileBytes, &map_a, kt * kTileK, (int)(row_begin + m0),
                        full_a(s));
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ---- MMA issue: one thread ----
        for (int kt = 0; kt < nk; ++kt) {
            const int sa = kt % kStagesA, sb = kt % kStagesB;
            if (!mbar_wait_bounded(full_a(sa), (uint32_t)(kt / kStagesA) & 1u) ||
                !mbar_wait_bounded(full_b(sb), (uint32_t)(kt / kStagesB) & 1u))
                *abort_flag = 1;
            if (*abort_flag) break;
            tc_fence_after();
            const uint32_t a_s = a_ring + sa * kTileBytes, b_s = b_ring + sb * kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
                mma_bf16(tmem, kmajor_sw128_desc(a_s + kk * 32), kmajor_sw128_desc(b_s + kk * 32),
                         (kt > 0 || kk > 0) ? 1u : 0u);
            // both stages are free once these MMAs have read them
            mma_commit(empty_a(sa));
            mma_commit(empty_b(sb));
        }
        mma_commit(acc_bar);  // fires when every MMA issued above has completed
    }

    // ---- epilogue: decoder warps read the accumulator ----
    if (warp < kDecodeWarps) {
        if (lane == 0 && !mbar_wait_bounded(acc_bar, 0)) *abort_flag = 1;
        const bool done = !__any_sync(0xFFFFFFFFu, *abort_flag != 0);  // warp-uniform
        tc_fence_after();
        if (done && *abort_flag == 0) {
            const uint32_t quarter = (uint32_t)warp & 3u;  // TMEM lanes this warp may read
            constexpr int kCols = kTileN / (kDecodeWarps / 4);  // columns per warp (64)
            const int c_begin = (warp >> 2) * kCols;
            const int64_t row = m0 + quarter * 32 + lane;
            uint16_t *orow = out + (row_begin + row) * n;
#pragma unroll 1
            for (int c0 = c_begin; c0 < c_begin + kCols; c0 += 32) {
                uint32_t acc[32];
                tmem_ld32(tmem + ((quarter * 32u) << 16) + (uint32_t)c0, acc);
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
        }
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            atomicExch(status, FP4_ERR_TIMEOUT);
            // give in-flight tensor-core work a last bounded chance to finish
            mbar_wait_bounded(acc_bar, 0);
        }
        __syncthreads();
    }
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(kTmemCols)
                     : "memory");
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled tensor_map_encoder() {
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
    // TMA descriptor of the activations [total_rows, k] bf16: 64 x 128 boxes with the
    // 128-byte swizzle; rows past total_rows and columns past k read as zero.
    EncodeTiled encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    CUtensorMap map;
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)(total_rows > 0 ? total_rows : 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
    const cuuint32_t box[2] = {kTileK, kTileM};
    const cuuint32_t elem_strides[2] = {1, 1};
    if (encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a), dims, strides,
               box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((n + kTileN - 1) / kTileN),
                    (unsigned)((max_rows + kTileM - 1) / kTileM), (unsigned)experts);
    mx_moe_gemm_kernel<<<grid, kThreads, kSmemBytes, stream>>>(
        map, expert_offsets, w_packed, w_scales, max_rows, total_rows, (int32_t)n, (int32_t)k, out,
        status);
    return cudaGetLastError();
}

}  // namespace fp4mx
