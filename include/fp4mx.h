/*
 * fp4mx.h -- C ABI of a GB300 (sm_103a) library that decodes block-scaled FP4
 * (E2M1) data into bf16.
 *
 * The operations below; each is one CUDA kernel launch on the caller's stream,
 * except the MoE layer (one memset and five launches, the last four of which may
 * start while the one before them finishes):
 *
 *   fp4_mx_unpack             MXFP4: one E8M0 scale byte per 32 codes, applied as
 *                             a wrapping 16-bit integer add into the bf16 exponent
 *                             field; both zero codes become +0.0.
 *   fp4_nv_embedding_gather   NVFP4 embedding lookup: token ids pick rows of packed
 *                             codes and of e4m3 scales (one per 16 codes); each
 *                             value is multiplied by (block scale * global scale)
 *                             in fp32 and rounded to bf16 (nearest, ties to even).
 *   fp4_nv_dequant            the same NVFP4 decode over every row of a table.
 *   fp4_mx_unpack_pages       the MXFP4 unpack of pages picked from a pool by id
 *                             (a paged FP4 KV cache).
 *   fp4_mx_quantize           bf16 to MXFP4 (the inverse direction of the unpack).
 *   fp4_mx_moe_gemm           grouped MoE GEMM, MXFP4 weights decoded into the
 *                             tensor-core operand (tcgen05), bf16 activations.
 *   fp4_mx_moe_forward        the whole MoE layer: top-k routing, gate/up GEMM
 *                             with silu(gate) * up, down GEMM, weighted top-k sum,
 *                             scratch in a caller-owned workspace
 *                             (fp4_mx_moe_workspace_bytes).
 *   fp4_mx_moe_forward_noalloc  the same layer on the library's static device
 *                             scratch (fp4_mx_moe_static_scratch_bytes).
 *
 * Conventions shared by every entry point:
 *   - Pointers named "device" must be device-accessible CUDA allocations
 *     (cudaMalloc / PyTorch CUDA tensors, or managed memory). Host pointers that
 *     CUDA does not know return FP4_ERR_POINTER before anything is launched.
 *   - bf16 values are passed as their 16-bit patterns (uint16_t).
 *   - Element order inside a byte: the even element is the low nibble, the odd
 *     element the high nibble.
 *   - The caller owns every buffer. The library allocates, frees and
 *     synchronises nothing; a call only enqueues work on `stream` (NULL = the
 *     legacy default stream) and returns. Kernel faults surface at the caller's
 *     next synchronisation, as with any CUDA launch.
 *   - Arguments are checked on the host before any launch. On any error status
 *     nothing is launched and the outputs are untouched. A call with zero
 *     elements returns FP4_OK without launching.
 *   - Outputs must not overlap inputs (FP4_ERR_ALIAS).
 *   - Byte buffers may have any alignment; bf16 (uint16_t), int32, int64 and
 *     float buffers must be aligned to their element size (else FP4_ERR_ALIGN).
 *     16-byte aligned bf16 buffers with 4-byte aligned packed buffers take the
 *     vectorised kernels, others a scalar kernel with the same results.
 *   - Calls are thread-safe and may be captured into CUDA graphs (no host
 *     synchronisation, no allocation, no host-to-device copy).
 */
#ifndef FP4MX_H
#define FP4MX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st *fp4_stream_t;

typedef enum fp4_status {
    FP4_OK = 0,
    FP4_ERR_NULL_PTR = 1,    /* a required pointer is NULL                          */
    FP4_ERR_SHAPE = 2,       /* negative size, k % 32 != 0, or size overflow        */
    FP4_ERR_GROUP = 3,       /* hidden % group_size != 0                            */
    FP4_ERR_UNSUPPORTED = 4, /* group_size other than 16                           */
    FP4_ERR_INDEX = 5,       /* value written to err_flag when an id is out of range */
    FP4_ERR_CUDA = 6,        /* the CUDA runtime reported an error (see fp4_last_error) */
    FP4_ERR_POINTER = 7,     /* a pointer is not device-accessible memory           */
    FP4_ERR_ALIAS = 8,       /* an output range overlaps an input range             */
    FP4_ERR_ALIGN = 9,       /* a pointer not aligned as its entry point requires   */
    FP4_ERR_TIMEOUT = 10     /* written to a status word: a bounded device wait ran out */
} fp4_status;

/*
 * fp4_mx_unpack -- MXFP4 (E2M1 codes, E8M0 per-32 scale) to bf16.
 *
 * Defined by "vllm-project/vllm pull 51583" (prhub digest), sections
 * "Motivation" and "Implementation breakdown": the E8M0 block scale is applied
 * as an integer add into the bf16 exponent field, and the two zero codes (+0.0,
 * -0.0) are forced to +0.0 lane by lane. With E the scale byte of element j's
 * block (j / 32) and L the bf16 pattern of the code's E2M1 value:
 *     out[j] = (L & 0x7FFF) != 0 ? (L + ((E - 127) << 7)) mod 2^16 : 0x0000
 * The add wraps: every E in 0..255 is a plain exponent (255 is not NaN), and
 * exponents that leave the bf16 range give the wrapped bit pattern.
 *
 *   packed       device, uint8[rows * k / 2], row-major [rows, k/2]
 *   scales_e8m0  device, uint8[rows * k / 32], row-major [rows, k/32]
 *   out_bf16     device, uint16[rows * k], row-major [rows, k]
 *   rows, k      rows >= 0, k >= 0, k % 32 == 0 (else FP4_ERR_SHAPE)
 *   stream       CUDA stream the kernel is enqueued on
 *
 * Rows are contiguous, so the data is one stream of rows * k codes; element j
 * reads byte j / 2 and scale byte j / 32.
 */
fp4_status fp4_mx_unpack(const uint8_t *packed, const uint8_t *scales_e8m0, uint16_t *out_bf16,
                         int64_t rows, int64_t k, fp4_stream_t stream);

/*
 * fp4_nv_embedding_gather -- NVFP4 token-embedding lookup, dequantised while
 * gathering.
 *
 * Defined by "sgl-project/sglang pull 34222" (prhub digest), sections
 * "Implementation breakdown" (items 1-2) and "Key source snippets"
 * (ModelOptNvFp4EmbeddingMethod.embedding, create_weights, reference_dequant):
 * for token t with id = ids[t] and column c,
 *     code = nibble c of weight[id]           (even c: low nibble, odd c: high)
 *     v    = (code & 8 ? -1 : +1) * {0, 0.5, 1, 1.5, 2, 3, 4, 6}[code & 7]
 *     eff  = fp32(e4m3 block_scale[id][c / 16]) * global_scale      (fp32, RNE)
 *     out[t][c] = bf16_rne(v * eff)                                  (fp32, RNE)
 * No fused multiply-add; code 8 gives -0.0 * eff (a signed zero is kept).
 *
 *   ids              device, int64[num_ids] (any logical shape, flattened)
 *   num_ids          >= 0
 *   weight           device, uint8[vocab * hidden / 2], row-major [vocab, hidden/2]
 *   block_scale_e4m3 device, uint8[vocab * hidden / 16] float8 e4m3fn bit patterns,
 *                    row-major [vocab, hidden/16]
 *   global_scale     device, one fp32 (a device pointer so that no host read or
 *                    synchronisation is needed and the call can be graph-captured)
 *   vocab            >= 1 when num_ids > 0
 *   hidden           > 0, hidden % group_size == 0 (else FP4_ERR_GROUP, the check
 *                    the pages' create_weights performs), hidden <= 2^31 (else
 *                    FP4_ERR_SHAPE: a row's word and segment counts are 32-bit)
 *   group_size       must be 16 (NVFP4); other positive values: FP4_ERR_UNSUPPORTED
 *   out_bf16         device, uint16[num_ids * hidden], row-major [num_ids, hidden]
 *   err_flag         device int32 or NULL. An id outside [0, vocab) never faults:
 *                    its output row is written as +0.0 and, when err_flag is not
 *                    NULL, *err_flag is set to FP4_ERR_INDEX (never cleared by the
 *                    library; the caller zeroes it and reads it when it syncs).
 *   stream           CUDA stream the kernel is enqueued on
 */
fp4_status fp4_nv_embedding_gather(const int64_t *ids, int64_t num_ids, const uint8_t *weight,
                                   const uint8_t *block_scale_e4m3, const float *global_scale,
                                   int64_t vocab, int64_t hidden, int64_t group_size,
                                   uint16_t *out_bf16, int32_t *err_flag, fp4_stream_t stream);

/*
 * fp4_mx_unpack_pages -- batched (paged) MXFP4 dequant, e.g. of an FP4 KV cache.
 *
 * "sgl-project/sglang pull 34222" (prhub digest), "Risks" item 3: the KV-cache
 * path scales FP4 codes by E8M0 powers of two (batched_dequantize), unlike the
 * NVFP4 embedding. A page table picks pages of an MXFP4 pool and each page is
 * decoded by the fp4_mx_unpack rule:
 *     out[i][:] = fp4_mx_unpack(pool page page_ids[i])
 *
 *   page_ids          device, int64[num_pages] (any logical shape, flattened)
 *   num_pages         >= 0
 *   packed_pool       device, uint8[pool_pages * page_elems / 2], [pool_pages, page_elems/2]
 *   scales_pool_e8m0  device, uint8[pool_pages * page_elems / 32]
 *   pool_pages        >= 1 when num_pages > 0
 *   page_elems        codes per page, a positive multiple of 32, at most 2^31 (else
 *                     FP4_ERR_SHAPE: a page's word and segment counts are 32-bit)
 *   out_bf16          device, uint16[num_pages * page_elems], row-major
 *   err_flag          device int32 or NULL: a page id outside [0, pool_pages) gives a
 *                     +0.0 row and sets *err_flag to FP4_ERR_INDEX (never cleared)
 *   stream            CUDA stream the kernel is enqueued on
 */
fp4_status fp4_mx_unpack_pages(const int64_t *page_ids, int64_t num_pages,
                               const uint8_t *packed_pool, const uint8_t *scales_pool_e8m0,
                               int64_t pool_pages, int64_t page_elems, uint16_t *out_bf16,
                               int32_t *err_flag, fp4_stream_t stream);

/*
 * fp4_mx_quantize -- bf16 to MXFP4: E2M1 codes plus one E8M0 scale per 32.
 *
 * The inverse direction of fp4_mx_unpack. "vllm-project/vllm pull 51583"
 * (prhub digest), "Key source snippets": the test quantises bf16 weights with
 * MXFP4QuantizeUtil.quantize into packed codes and per-32 scales, the format
 * fp4_mx_unpack reads; the pages do not print the rule. The rule used is the
 * OCP Microscaling (MX) v1.0 conversion, per block of 32 consecutive values:
 *     s    = floor(log2(max |x_i|)) - 2, clamped below at -127  (E8M0 = s + 127;
 *            an all-zero block gets E8M0 = 0)
 *     code = x_i / 2^s rounded to the nearest of {0, 0.5, 1, 1.5, 2, 3, 4, 6}, a tie
 *            to the even code, magnitudes above 6 saturated to 6; the sign bit of
 *            x_i is kept (so -0.0 and negatives that round to zero give code 8)
 *     a block holding Inf or NaN gets E8M0 = 0xFF (the MX NaN scale), codes 0.
 * For every block with E8M0 in [2, 252], fp4_mx_unpack(fp4_mx_quantize(x))
 * returns the nearest MXFP4 values; on values it produced itself it is exact.
 *
 *   in_bf16          device, uint16[rows * k] bf16 bits, row-major [rows, k], 2-byte aligned
 *   packed_out       device, uint8[rows * k / 2] (even element in the low nibble)
 *   scales_e8m0_out  device, uint8[rows * k / 32]
 *   rows, k          rows >= 0, k >= 0, k % 32 == 0 (else FP4_ERR_SHAPE)
 *   stream           CUDA stream the kernel is enqueued on
 */
fp4_status fp4_mx_quantize(const uint16_t *in_bf16, uint8_t *packed_out, uint8_t *scales_e8m0_out,
                           int64_t rows, int64_t k, fp4_stream_t stream);

/*
 * fp4_mx_moe_gemm -- grouped MoE expert GEMM with MXFP4 weights, the decode fused
 * into the tensor-core operand (tcgen05 on sm_103a).
 *
 * The consumer of the MXFP4 unpack on the pages: "vllm-project/vllm pull 51583"
 * (prhub digest), "Motivation" and the comments on the unpack_B loop -- the CPU
 * MoE GEMM unpacks each tile of MXFP4 expert weights to bf16 before multiplying.
 * For expert e with activation rows [offsets[e], offsets[e+1]):
 *     out[r][j] = sum_k a[r][k] * W_e[j][k]        (r in expert e's rows, j < n)
 * where W_e[j][k] is the bf16 value fp4_mx_unpack gives for row j of expert e's
 * packed weights. Products and sums are accumulated in fp32 by the tensor core
 * (summation order unspecified), then rounded to bf16 (nearest, ties to even).
 * (The zero code with the sign bit set enters the products as -0.0 rather than
 * +0.0: the same value, so only the sign of an all-zero sum can differ.)
 *
 *   a_bf16               device, uint16[total_rows * k] bf16 bits, row-major, the rows
 *                        of each expert contiguous; 16-byte aligned
 *   expert_offsets       device, int64[experts + 1], non-decreasing, offsets[0] = 0,
 *                        offsets[experts] = total_rows
 *   experts              number of experts (<= 65535)
 *   max_rows_per_expert  upper bound on offsets[e+1] - offsets[e] (sets the grid; an
 *                        expert with more rows is not computed and status is set to
 *                        FP4_ERR_SHAPE)
 *   w_packed             device, uint8[experts * n * k / 2]: expert e's [n, k/2] codes
 *                        (as fp4_mx_unpack reads them); 16-byte aligned
 *   w_scales_e8m0        device, uint8[experts * n * k / 32]
 *   n, k                 output columns and reduction length, both multiples of 32;
 *                        experts * n <= 2^31 - 1024 (the weight loads, too, address
 *                        rows with 32-bit coordinates; else FP4_ERR_SHAPE)
 *   total_rows           rows of a and out, below 2^31 - 1024 (the tensor-core
 *                        loads address rows with 32-bit coordinates; else
 *                        FP4_ERR_SHAPE); an expert whose rows fall outside
 *                        [0, total_rows) is not computed and status is set to
 *                        FP4_ERR_SHAPE (the offsets are checked on the device)
 *   out_bf16             device, uint16[total_rows * n], row-major; 16-byte aligned
 *   status               device int32, required. Set to FP4_ERR_TIMEOUT if a bounded
 *                        wait on the tensor core ran out (the kernel then stops, frees
 *                        its tensor memory and returns) or FP4_ERR_SHAPE as above;
 *                        never cleared by the library.
 *   stream               CUDA stream the kernel is enqueued on
 */
fp4_status fp4_mx_moe_gemm(const uint16_t *a_bf16, const int64_t *expert_offsets, int64_t experts,
                           int64_t max_rows_per_expert, const uint8_t *w_packed,
                           const uint8_t *w_scales_e8m0, int64_t n, int64_t k, int64_t total_rows,
                           uint16_t *out_bf16, int32_t *status, fp4_stream_t stream);

/*
 * fp4_mx_moe_forward -- the MoE layer with MXFP4 experts: routing, gate/up GEMM,
 * silu(gate) * up, down GEMM and the top-k weighted sum, all on the device.
 *
 * The layer the pages' unpack feeds: "vllm-project/vllm pull 51583" (prhub
 * digest), the CPU test that runs ops.fused_experts_cpu with MXFP4 experts and
 * the zero-code test whose comment notes that silu(0) * 0 = 0 collapses the
 * layer to exact zeros. For token m and each slot j < topk with expert
 * e = topk_ids[m][j] and weight w = topk_weights[m][j]:
 *     h   = a[m] @ W1_e^T               W1_e [2n, k]: rows 0..n-1 gate, n..2n-1 up
 *     act = bf16(silu(h[:n]) * h[n:])   silu(x) = x / (1 + exp(-x)), fp32
 *     y   = bf16(act @ W2_e^T)          W2_e [k, n]
 *     out[m] = bf16(sum_j w * y)        fp32, slots in order j = 0, 1, ...
 * where W1_e and W2_e are what fp4_mx_unpack gives for the expert's packed rows
 * (as values: a zero code may enter a product as -0.0), and the GEMMs accumulate
 * in fp32 on the tensor core (order unspecified).
 *
 *   a_bf16               device, uint16[tokens * k] bf16 bits, row-major; 16-byte aligned
 *   topk_ids             device, int32[tokens * topk]; an id outside [0, experts)
 *                        contributes nothing and status is set to FP4_ERR_INDEX
 *   topk_weights         device, fp32[tokens * topk]
 *   tokens, topk         tokens >= 0 (0: nothing is launched), 1 <= topk <= 1024,
 *                        tokens * topk <= 2^31 - 1024
 *   experts              1 .. 65535
 *   max_rows_per_expert  capacity of one expert (values above tokens * topk are
 *                        treated as tokens * topk); the slots of an expert that
 *                        holds more rows contribute nothing and status is set to
 *                        FP4_ERR_SHAPE. When no token repeats an expert among its
 *                        slots, tokens is always enough.
 *   w1_packed            device, uint8[experts * 2n * k / 2]; 16-byte aligned
 *   w1_scales_e8m0       device, uint8[experts * 2n * k / 32]
 *   w2_packed            device, uint8[experts * k * n / 2]; 16-byte aligned
 *   w2_scales_e8m0       device, uint8[experts * k * n / 32]
 *   n, k                 intermediate and hidden sizes: multiples of 32, 32 .. 2^20,
 *                        with experts * 2n and experts * k <= 2^31 - 1024 (weight rows
 *                        of the two GEMMs, addressed with 32-bit coordinates)
 *   workspace            device scratch of workspace_bytes >= fp4_mx_moe_workspace_bytes(),
 *                        256-byte aligned; owned by the caller, overwritten by the call,
 *                        not read afterwards
 *   out_bf16             device, uint16[tokens * k], row-major; 16-byte aligned
 *   status               device int32, required; FP4_ERR_INDEX / FP4_ERR_SHAPE as
 *                        above or FP4_ERR_TIMEOUT from a GEMM; never cleared
 *   stream               CUDA stream every kernel is enqueued on
 * Returns FP4_ERR_SHAPE for bad sizes or a short workspace, FP4_ERR_ALIAS when the
 * output or the workspace overlaps an input or each other.
 */
fp4_status fp4_mx_moe_forward(const uint16_t *a_bf16, const int32_t *topk_ids,
                              const float *topk_weights, int64_t tokens, int64_t topk,
                              int64_t experts, int64_t max_rows_per_expert,
                              const uint8_t *w1_packed, const uint8_t *w1_scales_e8m0,
                              const uint8_t *w2_packed, const uint8_t *w2_scales_e8m0, int64_t n,
                              int64_t k, void *workspace, int64_t workspace_bytes,
                              uint16_t *out_bf16, int32_t *status, fp4_stream_t stream);

/* Bytes of workspace fp4_mx_moe_forward needs for these sizes (about
 * tokens * topk * (4k + 2n) bytes), or -1 when the sizes are invalid. */
int64_t fp4_mx_moe_workspace_bytes(int64_t tokens, int64_t topk, int64_t experts, int64_t n,
                                   int64_t k);

/*
 * fp4_mx_moe_forward_noalloc -- fp4_mx_moe_forward with the library's own static
 * scratch instead of a caller workspace. The paper has no counterpart: this entry
 * point exists for callers that cannot call cudaMalloc -- code running inside a
 * host application that owns all device memory and hands out no allocator, code
 * on a path where a device allocation (which may synchronise the device) is not
 * allowed, or code that must not change the process's memory footprint per call.
 *
 * Same arguments, semantics and errors as fp4_mx_moe_forward (above) minus the
 * workspace; nothing on this path calls cudaMalloc, cudaFree or an allocating
 * library routine. The scratch is a static __device__ array of
 * fp4_mx_moe_static_scratch_bytes() bytes (288 MiB: the 4,096-token, top-4,
 * 2880 x 2880 layer fits) in a module of its own. Under lazy module loading
 * (CUDA_MODULE_LOADING=LAZY, the CUDA 12+ default) the driver loads that module,
 * and reserves and zero-fills the array, on the first call on a device; make that
 * first call before any stream capture begins. Under eager loading every process
 * that loads this library reserves the 288 MiB on every device it uses, whether
 * or not it ever calls this function. Every GPU that loads the module holds the
 * array until the process exits. The array's address is looked up on every call
 * (a host-side lookup), so it follows the current context, also after a reset.
 * A layer whose workspace would exceed the array is rejected with FP4_ERR_SHAPE
 * before anything is launched (the reason is in fp4_last_error()). Each call
 * clears the counters it needs at zero itself. Every call on a device shares the
 * one array and finds the previous call's contents in it: calls must be ordered
 * (one stream, or events between streams); two calls that overlap on the GPU race
 * and overwrite each other's scratch. Thread-safe on the host.
 */
fp4_status fp4_mx_moe_forward_noalloc(const uint16_t *a_bf16, const int32_t *topk_ids,
                                      const float *topk_weights, int64_t tokens, int64_t topk,
                                      int64_t experts, int64_t max_rows_per_expert,
                                      const uint8_t *w1_packed, const uint8_t *w1_scales_e8m0,
                                      const uint8_t *w2_packed, const uint8_t *w2_scales_e8m0,
                                      int64_t n, int64_t k, uint16_t *out_bf16, int32_t *status,
                                      fp4_stream_t stream);

/* Bytes of the static scratch fp4_mx_moe_forward_noalloc uses (per device). */
int64_t fp4_mx_moe_static_scratch_bytes(void);

/*
 * fp4_wait_selftest -- check of the bounded waits that guard the tensor-core
 * kernels (fp4_mx_moe_gemm, fp4_mx_moe_forward): every mbarrier wait in them
 * gives up after a limit, and the launch then writes FP4_ERR_TIMEOUT to its
 * status word instead of hanging. This call runs one such wait on a barrier that
 * nothing arrives on, so that a test can see the limit run out without a fault.
 *
 *   mode    0: the polling wait (gives up after about 2^29 SM cycles, ~0.3 s);
 *           1: the sleeping wait (gives up after about 2^29 SM cycles, ~0.3 s);
 *           2: control, the phase completes first and *status is left alone;
 *           other values: FP4_ERR_SHAPE
 *   status  device, one int32; set to FP4_ERR_TIMEOUT when the wait gives up
 *           (never cleared by the library)
 *   stream  CUDA stream the one-warp kernel is enqueued on
 * Returns FP4_ERR_NULL_PTR / FP4_ERR_ALIGN / FP4_ERR_POINTER for a bad status
 * pointer, else FP4_OK once the kernel is enqueued.
 */
fp4_status fp4_wait_selftest(int32_t mode, int32_t *status, fp4_stream_t stream);

/*
 * fp4_nv_dequant -- dequantise a whole NVFP4 table (every row, in order).
 *
 * The dense counterpart of fp4_nv_embedding_gather: out[r][c] is what the
 * gather writes for id = r. "sgl-project/sglang pull 34222" (prhub digest),
 * sections "Comments" and "Risks": with tied word embeddings the lm_head is the
 * embedding table, and the gather-only method's apply() cannot serve it; the
 * table dequantised to bf16 is what that use needs. Same element rule, op order
 * and rounding as the gather (see above).
 *
 *   weight           device, uint8[rows * hidden / 2], row-major [rows, hidden/2]
 *   block_scale_e4m3 device, uint8[rows * hidden / 16] e4m3fn bits, [rows, hidden/16]
 *   global_scale     device, one fp32
 *   rows             >= 0 (0: nothing is launched)
 *   hidden           > 0, hidden % group_size == 0 (else FP4_ERR_GROUP), hidden <= 2^31
 *                    (else FP4_ERR_SHAPE)
 *   group_size       must be 16; other positive values: FP4_ERR_UNSUPPORTED
 *   out_bf16         device, uint16[rows * hidden], row-major [rows, hidden]
 *   stream           CUDA stream the kernel is enqueued on
 */
fp4_status fp4_nv_dequant(const uint8_t *weight, const uint8_t *block_scale_e4m3,
                          const float *global_scale, int64_t rows, int64_t hidden,
                          int64_t group_size, uint16_t *out_bf16, fp4_stream_t stream);

/* Static English text for a status code ("unknown status" for other values). */
const char *fp4_status_string(fp4_status status);

/* Text of the last CUDA error this thread's calls met ("" if none). Valid
 * until this thread's next call into the library. */
const char *fp4_last_error(void);

/* Version of this ABI (major * 100 + minor): 101 adds fp4_nv_dequant, 102 adds
 * fp4_mx_quantize and FP4_ERR_ALIGN, 103 adds fp4_mx_moe_gemm and FP4_ERR_TIMEOUT,
 * 104 adds fp4_mx_unpack_pages, 105 adds fp4_mx_moe_forward and
 * fp4_mx_moe_workspace_bytes, 106 adds fp4_mx_moe_forward_noalloc and
 * fp4_mx_moe_static_scratch_bytes, 107 adds fp4_wait_selftest, 108 bounds hidden
 * (NVFP4 gather and dequant) and page_elems (paged unpack) at 2^31 and the MoE
 * weight rows (experts * n, experts * 2n, experts * k) at 2^31 - 1024. */
int fp4_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FP4MX_H */
