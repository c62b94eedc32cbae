// mx_moe_gemm_wide.cu -- the MoE GEMM's main kernel: 128 x 256 output tiles, every
// operand brought in by TMA (sm_103a).
//
// Same computation as mx_moe_gemm.cu (bf16 activations x MXFP4 expert weights
// decoded into the tensor-core operand, fp32 accumulation in tensor memory), laid
// out so that no thread waits on global memory:
//   - one TMA thread streams the 128 x 64 bf16 activation tiles (128-byte swizzle)
//     through a kStagesA ring;
//   - another TMA thread first bulk-copies the tile's E8M0 scales (256 rows x k/32
//     bytes, contiguous in memory) into shared memory, then streams the packed
//     codes of the 256 x 64 weight slices (256 rows x 32 bytes, a 2-D uint8 tensor
//     map) through a deep kStagesRaw ring;
//   - 16 decoder warps in two groups that own alternating K slices read a
//     slice's packed codes and scale
//     bytes from shared memory (one thread per weight row: 64 codes, two E8M0
//     blocks), release the raw stage, decode in registers and store the bf16 tile
//     in the swizzled K-major layout of the tensor core's B operand;
//   - one thread issues four tcgen05.mma kind::f16 (M = 128, N = 256, K = 16) per
//     slice into a 256-column fp32 accumulator and commits the stages back.
// A 256-wide tile halves the re-reads of the activations against 128-wide
// tiles, and every global read is a bulk copy that the copy engine overlaps.
//
// When an expert can have more than 128 rows, each CTA owns two 128-row tiles of
// the expert (two 256-column accumulators, all 512 tensor-memory columns) that
// share every decoded weight tile, halving the decode work per FLOP.
//
// Used when k <= 4096 (the scale block fits in shared memory) and the weight and
// scale buffers are 16-byte aligned; other calls take the general kernel.
// Every mbarrier wait is bounded, as in the general kernel.
#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"
#include "tc_sm103.cuh"

namespace fp4mx {
namespace {

constexpr int kM = 128;   // rows of one accumulator (one tensor-core M)
constexpr int kN = 256;
constexpr int kK = 64;
constexpr int kStagesRaw = 4;
constexpr int kGroups = 2;        // decoder groups owning alternating K slices
constexpr int kDecodeWarps = 16;  // two groups of 256 threads, one thread per weight row
constexpr int kGroupWarps = kDecodeWarps / kGroups;
constexpr int kTmaAWarp = kDecodeWarps;
constexpr int kTmaWWarp = kDecodeWarps + 1;
constexpr int kMmaWarp = kDecodeWarps + 2;
constexpr int kThreads = (kDecodeWarps + 3) * 32;
constexpr int kTileABytes = kM * kK * 2;  // 16 KiB: one 128 x 64 activation tile
constexpr int kRawBytes = kN * kK / 2;    // 8 KiB
constexpr int kBBytes = kN * kK * 2;      // 32 KiB
constexpr int kScaleBytes = 32 * 1024;    // 256 rows x k/32 bytes: k <= 4096

// kMT row tiles of 128 per CTA share every decoded weight tile: one accumulator
// of 256 tensor-memory columns each (kMT = 2 fills the 512 columns).
template <int kMT>
struct WideCfg {
    static constexpr int kRows = kM * kMT;
    static constexpr int kStagesA = 3;
    static constexpr int kStagesB = kMT == 1 ? 3 : 2;
    static constexpr uint32_t kTmemCols = 256u * kMT;
    static constexpr int kABytes = kMT * kTileABytes;
    // shared-memory layout from a 1024-byte aligned base
    static constexpr int kOffA = 0;
    static constexpr int kOffB = kOffA + kStagesA * kABytes;
    static constexpr int kOffRaw = kOffB + kStagesB * kBBytes;
    static constexpr int kOffScale = kOffRaw + kStagesRaw * kRawBytes;
    static constexpr int kOffBar = kOffScale + kScaleBytes;
    static constexpr int kSmemBytes = 1024 + kOffBar + 256;
    static_assert(kSmemBytes <= 232448, "shared memory per block");
};

template <int kMT>
__global__ void __launch_bounds__(kThreads, 1)
mx_moe_gemm_wide_kernel(const __grid_constant__ CUtensorMap map_a,
                        const __grid_constant__ CUtensorMap map_w,
                        const int64_t *__restrict__ expert_offsets,
                        const uint8_t *__restrict__ w_scales, int64_t max_rows,
                        int64_t total_rows, int32_t n, int32_t k, uint16_t *__restrict__ out,
                        int32_t *__restrict__ status) {
    using C = WideCfg<kMT>;
    constexpr int kStagesA = C::kStagesA, kStagesB = C::kStagesB, kABytes = C::kABytes;
    constexpr int kOffA = C::kOffA, kOffB = C::kOffB, kOffRaw = C::kOffRaw;
    constexpr int kOffScale = C::kOffScale, kOffBar = C::kOffBar;
    constexpr uint32_t kTmemCols = C::kTmemCols;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t base = smem_addr(smem);
    const uint32_t a_ring = base + kOffA, b_ring = base + kOffB, raw_ring = base + kOffRaw;
    const uint32_t scale_smem = base + kOffScale;
    const uint32_t bars = base + kOffBar;
    auto full_a = [&](int s) { return bars + 8u * s; };
    auto empty_a = [&](int s) { return bars + 8u * (kStagesA + s); };
    auto full_raw = [&](int s) { return bars + 8u * (2 * kStagesA + s); };
    auto empty_raw = [&](int s) { return bars + 8u * (2 * kStagesA + kStagesRaw + s); };
    auto full_b = [&](int s) { return bars + 8u * (2 * kStagesA + 2 * kStagesRaw + s); };
    auto empty_b = [&](int s) { return bars + 8u * (2 * kStagesA + 2 * kStagesRaw + kStagesB + s); };
    constexpr int kNumBars = 2 * kStagesA + 2 * kStagesRaw + 2 * kStagesB + 2;
    const uint32_t scale_bar = bars + 8u * (kNumBars - 2);
    const uint32_t acc_bar = bars + 8u * (kNumBars - 1);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + 8 * kNumBars);
    volatile uint32_t *abort_flag = tmem_slot + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int expert = blockIdx.z;
    const int n0 = blockIdx.x * kN;
    const int64_t m0 = (int64_t)blockIdx.y * C::kRows;
    const int64_t row_begin = expert_offsets[expert];
    const int64_t rows = expert_offsets[expert + 1] - row_begin;
    // offsets live on the device: check them here, never read or write past the buffers
    if (row_begin < 0 || rows < 0 || rows > max_rows || row_begin + rows > total_rows) {
        if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicExch(status, FP4_ERR_SHAPE);
        return;
    }
    if (m0 >= rows) return;  // this expert has fewer row tiles than the grid
    // row tiles of this CTA that hold rows of the expert (the rest is neither loaded nor computed)
    const int mt_live = (rows - m0 > (int64_t)kM) ? kMT : 1;
    const int nk = (k + kK - 1) / kK;
    const int scale_pitch = k / 32;

    if (tid == 0) {
        for (int s = 0; s < kStagesA; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(empty_a(s), 1);
        }
        for (int s = 0; s < kStagesRaw; ++s) {
            mbar_init(full_raw(s), 1);
            mbar_init(empty_raw(s), kGroupWarps);  // the warps of the group owning the slice
        }
        for (int s = 0; s < kStagesB; ++s) {
            mbar_init(full_b(s), kGroupWarps);  // one arrival per warp of the owning group
            mbar_init(empty_b(s), 1);
        }
        mbar_init(scale_bar, 1);
        mbar_init(acc_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
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
        // ---- decoder warps: two groups of 8 warps own alternating K slices (group
        // g takes kt = g, g + 2, ...); each thread decodes one whole row of its
        // slices: 64 codes, two E8M0 blocks ----
        const int group = warp / kGroupWarps;
        const uint32_t r = (uint32_t)(tid - group * kGroupWarps * 32);  // 0..255
        uint32_t st_off[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) st_off[j] = sw128_offset(r, (uint32_t)j);
        const uint32_t raw_off = r * 32u;
        const uint32_t scale_row = scale_smem + r * (uint32_t)scale_pitch;
        if (lane == 0 && !mbar_wait_bounded(scale_bar, 0)) *abort_flag = 1;
        bool stop = __any_sync(0xFFFFFFFFu, *abort_flag != 0);
        for (int kt = group; kt < nk && !stop; kt += kGroups) {
            const int sr = kt % kStagesRaw, sb = kt % kStagesB;
            const uint32_t use_b = (uint32_t)(kt / kStagesB);
            const uint32_t b_tile = b_ring + sb * kBBytes;
            if (lane == 0 && !mbar_wait_bounded(full_raw(sr), (uint32_t)(kt / kStagesRaw) & 1u))
                *abort_flag = 1;
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;  // warp-uniform
            const uint4 w0 = lds_v4(raw_ring + sr * kRawBytes + raw_off);
            const uint4 w1 = lds_v4(raw_ring + sr * kRawBytes + raw_off + 16u);
            const uint32_t e0 = (2 * kt < scale_pitch) ? lds_u8(scale_row + 2u * (uint32_t)kt) : 127u;
            const uint32_t e1 =
                (2 * kt + 1 < scale_pitch) ? lds_u8(scale_row + 2u * (uint32_t)kt + 1u) : 127u;
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_raw(sr));  // the slice's raw bytes are in registers
            const ByteTable t0 = mx_scaled_table(e0);
            const ByteTable t1 = mx_scaled_table(e1);
            uint4 d[8];
            d[0] = mx_decode_word(w0.x, t0);
            d[1] = mx_decode_word(w0.y, t0);
            d[2] = mx_decode_word(w0.z, t0);
            d[3] = mx_decode_word(w0.w, t0);
            d[4] = mx_decode_word(w1.x, t1);
            d[5] = mx_decode_word(w1.y, t1);
            d[6] = mx_decode_word(w1.z, t1);
            d[7] = mx_decode_word(w1.w, t1);
            if (use_b > 0 && lane == 0 && !mbar_wait_bounded(empty_b(sb), (use_b - 1u) & 1u))
                *abort_flag = 1;
            if (__any_sync(0xFFFFFFFFu, *abort_flag != 0)) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) st_shared_v4(b_tile + st_off[j], d[j]);
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(full_b(sb));
        }
    } else if (warp == kTmaAWarp && lane == 0) {
        // ---- TMA: activation tiles ----
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kStagesA;
            if (kt >= kStagesA && !mbar_wait_bounded(empty_a(s), (uint32_t)(kt / kStagesA - 1) & 1u))
                *abort_flag = 1;
            if (*abort_flag) break;
            mbar_arrive_expect_tx(full_a(s), (uint32_t)(mt_live * kTileABytes));
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
                if (mt < mt_live)
                        tma_load_2d(a_ring + s * kABytes + mt * kTileABytes, &map_a, kt * kK,
                                (int)(row_begin + m0 + mt * kM), full_a(s));
        }
    } else if (warp == kTmaWWarp && lane == 0) {
        // ---- TMA: the tile's scales once, then the packed weight slices ----
        const int rows_n = (n - n0 < kN) ? n - n0 : kN;
        const uint32_t scale_bytes = (uint32_t)rows_n * (uint32_t)scale_pitch;
        mbar_arrive_expect_tx(scale_bar, scale_bytes);
        bulk_load(scale_smem, w_scales + ((int64_t)expert * n + n0) * scale_pitch, scale_bytes,
                  scale_bar);
        const int w_row = expert * n + n0;
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kStagesRaw;
            if (kt >= kStagesRaw &&
                !mbar_wait_bounded(empty_raw(s), (uint32_t)(kt / kStagesRaw - 1) & 1u))
                *abort_flag = 1;
            if (*abort_flag) break;
            mbar_arrive_expect_tx(full_raw(s), kRawBytes);
            tma_load_2d(raw_ring + s * kRawBytes, &map_w, kt * (kK / 2), w_row, full_raw(s));
        }
    } else if (warp == kMmaWarp && lane == 0) {
        // ---- MMA issue ----
        constexpr uint32_t idesc = instr_desc_bf16<kM, kN>();
        for (int kt = 0; kt < nk; ++kt) {
            const int sa = kt % kStagesA, sb = kt % kStagesB;
            if (!mbar_wait_bounded(full_a(sa), (uint32_t)(kt / kStagesA) & 1u) ||
                !mbar_wait_bounded(full_b(sb), (uint32_t)(kt / kStagesB) & 1u))
                *abort_flag = 1;
            if (*abort_flag) break;
            tc_fence_after();
            const uint32_t a_s = a_ring + sa * kABytes, b_s = b_ring + sb * kBBytes;
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt)
#pragma unroll
                for (int kk = 0; kk < kK / 16; ++kk)
                    if (mt < mt_live)
                        mma_bf16(tmem + mt * kN, kmajor_sw128_desc(a_s + mt * kTileABytes + kk * 32),
                                 kmajor_sw128_desc(b_s + kk * 32), idesc, (kt > 0 || kk > 0) ? 1u : 0u);
            mma_commit(empty_a(sa));
            mma_commit(empty_b(sb));
        }
        mma_commit(acc_bar);
    }

    // ---- epilogue: decoder warps read the accumulator ----
    if (warp < kDecodeWarps) {
        if (lane == 0 && !mbar_wait_bounded(acc_bar, 0)) *abort_flag = 1;
        const bool done = !__any_sync(0xFFFFFFFFu, *abort_flag != 0);
        tc_fence_after();
        if (done) {
            const uint32_t quarter = (uint32_t)warp & 3u;  // TMEM lanes this warp may read
            constexpr int kCols = kN / (kDecodeWarps / 4);  // 64 columns per warp
            const int c_begin = (warp >> 2) * kCols;
#pragma unroll 1
            for (int mt = 0; mt < mt_live; ++mt) {
                const int64_t row = m0 + mt * kM + quarter * 32 + lane;
                uint16_t *orow = out + (row_begin + row) * n;
#pragma unroll 1
                for (int c0 = c_begin; c0 < c_begin + kCols; c0 += 32) {
                    uint32_t acc[32];
                    tmem_ld32(tmem + ((quarter * 32u) << 16) + (uint32_t)(mt * kN + c0), acc);
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
    }
    tc_fence_before();
    __syncthreads();
    if (*abort_flag) {
        if (tid == 0) {
            atomicExch(status, FP4_ERR_TIMEOUT);
            mbar_wait_bounded(acc_bar, 0);  // a last bounded chance for in-flight MMAs
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

}  // namespace

bool mx_moe_gemm_wide_eligible(const uint8_t *w_packed, const uint8_t *w_scales, int64_t n,
                               int64_t k) {
    return k <= 4096 && (int64_t)kN * (k / 32) <= kScaleBytes &&
           reinterpret_cast<uintptr_t>(w_packed) % 16 == 0 &&
           reinterpret_cast<uintptr_t>(w_scales) % 16 == 0 && n % 32 == 0 && k % 32 == 0;
}

cudaError_t launch_mx_moe_gemm_wide(const uint16_t *a, const int64_t *expert_offsets,
                                    int64_t experts, int64_t max_rows, int64_t total_rows,
                                    const uint8_t *w_packed, const uint8_t *w_scales, int64_t n,
                                    int64_t k, uint16_t *out, int32_t *status,
                                    cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int device = 0;
    cudaError_t err = cudaGetDevice(&device);
    if (err != cudaSuccess) return err;
    if (configured_device != device) {
        err = cudaFuncSetAttribute(mx_moe_gemm_wide_kernel<1>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   WideCfg<1>::kSmemBytes);
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(mx_moe_gemm_wide_kernel<2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       WideCfg<2>::kSmemBytes);
        if (err != cudaSuccess) return err;
        configured_device = device;
    }
    EncodeTiled encode = tensor_map_encoder();
    if (encode == nullptr) return cudaErrorNotSupported;
    const cuuint32_t elem_strides[2] = {1, 1};
    // activations [total_rows, k] bf16: 64 x 128 boxes, 128-byte swizzle
    CUtensorMap map_a;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)(total_rows > 0 ? total_rows : 1)};
        const cuuint64_t strides[1] = {(cuuint64_t)k * 2};
        const cuuint32_t box[2] = {kK, kM};  // one 128-row tile per TMA load
        if (encode(&map_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a), dims,
                   strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // packed weights [experts * n rows, k / 2 bytes] uint8: 32 x 256 boxes, no swizzle
    CUtensorMap map_w;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(k / 2), (cuuint64_t)(experts * n)};
        const cuuint64_t strides[1] = {(cuuint64_t)(k / 2)};
        const cuuint32_t box[2] = {kK / 2, kN};
        if (encode(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w_packed), dims,
                   strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // two 128-row tiles per CTA (sharing each decoded weight tile) once an expert
    // can have more than 128 rows
    if (max_rows > kM) {
        const dim3 grid((unsigned)((n + kN - 1) / kN),
                        (unsigned)((max_rows + WideCfg<2>::kRows - 1) / WideCfg<2>::kRows),
                        (unsigned)experts);
        mx_moe_gemm_wide_kernel<2><<<grid, kThreads, WideCfg<2>::kSmemBytes, stream>>>(
            map_a, map_w, expert_offsets, w_scales, max_rows, total_rows, (int32_t)n, (int32_t)k,
            out, status);
    } else {
        const dim3 grid((unsigned)((n + kN - 1) / kN), (unsigned)((max_rows + kM - 1) / kM),
                        (unsigned)experts);
        mx_moe_gemm_wide_kernel<1><<<grid, kThreads, WideCfg<1>::kSmemBytes, stream>>>(
            map_a, map_w, expert_offsets, w_scales, max_rows, total_rows, (int32_t)n, (int32_t)k,
            out, status);
    }
    return cudaGetLastError();
}

}  // namespace fp4mx
