// mx_moe_gemm.cu -- MoE expert GEMM with MXFP4 weights decoded into the tensor-core
// B operand (tcgen05, sm_103a): the general kernel (any k that is a multiple of
// 32, 16-byte aligned weights, any scale alignment) and the dispatch; calls with
// k <= 4096 and 16-byte aligned scales go to mx_moe_gemm_wide.cu.
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

#include "fp4_decode.cuh"
#include "fp4mx.h"
#include "launch.h"
#include "tc_sm103.cuh"

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
constexpr int kTileBytes = kTileM * kTileK * 2;  // 16 KiB per operand tile and stage
// shared memory: 1 KiB to align the tiles to the 1024-byte swizzle atom, the A
// and B rings, then barriers, the tensor-memory address and the abort flag.
// Two CTAs (2 x 128 tensor-memory columns) fit on an SM.
constexpr int kBarrierOffset = (kStagesA + kStagesB) * kTileBytes;
constexpr int kSmemBytes = 1024 + kBarrierOffset + 256;

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
                         instr_desc_bf16<kTileM, kTileN>(), (kt > 0 || kk > 0) ? 1u : 0u);
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


}  // namespace

cudaError_t launch_mx_moe_gemm(const uint16_t *a, const int64_t *expert_offsets, int64_t experts,
                               int64_t max_rows, int64_t total_rows, const uint8_t *w_packed,
                               const uint8_t *w_scales, int64_t n, int64_t k, uint16_t *out,
                               int32_t *status, cudaStream_t stream) {
    if (mx_moe_gemm_wide_eligible(w_packed, w_scales, n, k))
        return launch_mx_moe_gemm_wide(a, expert_offsets, experts, max_rows, total_rows, w_packed,
                                       w_scales, n, k, out, status, stream);
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
