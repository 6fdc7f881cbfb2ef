/*
 * rocmfp4.h -- C ABI of the GB300 (sm_103a) ROCmFP4 library.
 *
 * ROCmFP4 is the 4-bit block format defined on the page "Feasibility Report:
 * Porting ROCmFP4 to Atlas", section "What is ROCmFP4?":
 *   - subsection "Block Layout": a block holds 32 weights as qs[16] (32 packed
 *     4-bit codes) followed by e[2] (dual-scale, 18 bytes, one scale per
 *     16-weight half, type Q4_0_ROCMFP4) or by e (single-scale "fast" block,
 *     17 bytes, type Q4_0_ROCMFP4_FAST);
 *   - subsection "Codebook10 Value Table": code q maps to
 *     {0,1,2,3,4,6,8,10,0,-1,-2,-3,-4,-6,-8,-10}[q];
 *   - subsection "Scale Format": scale bytes are finite unsigned E4M3 values
 *     used as half-scales.
 * This library reads them as follows (the same readings the test oracle
 * takes):
 *   - byte j of qs holds weight j in its low nibble and weight j+16 in its
 *     high nibble; the first scale covers weights 0..15, the second 16..31;
 *   - weight = Codebook10[q] * hs(e), hs(e) = one half of the unsigned E4M3
 *     value of e (exponent bits 6..3 with bias 7, mantissa bits 2..0,
 *     exponent 0 subnormal); code 8 is +0;
 *   - a scale byte is finite iff it is below 0x7F;
 *   - a matrix of N rows and K columns (K a multiple of 32) is N rows of K/32
 *     blocks, rows and blocks back to back with no padding
 *     (row_bytes = K/32 * block_bytes).
 *
 * Conventions shared by every entry point
 *   - Every pointer to matrix, activation or output data is DEVICE memory
 *     owned by the caller.  Calls do not allocate per call; a per-device
 *     workspace (split-reduction partials and counters: about 0.18 MiB per
 *     SM, 27 MiB on a 152-SM GPU) is allocated once, on first use, and
 *     released by rocmfp4_shutdown().
 *   - Calls on one device share that workspace: calls that overlap on the GPU
 *     (unordered streams, or graphs replayed concurrently) race and give wrong
 *     results.  Calls ordered on one stream are safe.
 *   - Calls are asynchronous on the given CUDA stream (NULL = legacy default
 *     stream) except rocmfp4_validate, which waits for its own result.
 *   - Arguments are checked on the host: a NULL pointer with a non-empty
 *     shape, a negative size, K not a multiple of 32 or an unknown enum value
 *     returns ROCMFP4_ERR_INVALID_ARG and launches nothing.  A failed launch
 *     returns ROCMFP4_ERR_CUDA (rocmfp4_last_error() gives the CUDA message).
 *   - Weights are assumed validated (rocmfp4_validate): outputs computed from
 *     a non-finite scale byte are unspecified, but no access ever leaves the
 *     caller's buffers.
 *   - Outputs must not overlap inputs.  Results are bitwise identical from
 *     run to run for the same shapes on the same device (fixed reduction
 *     order, no floating-point atomics).
 *   - Empty shapes (N == 0, M == 0 or K == 0) are valid; K == 0 writes zeros.
 */
#ifndef ROCMFP4_H_
#define ROCMFP4_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA headers. */
typedef struct CUstream_st *rocmfp4_stream_t;

typedef enum {
  ROCMFP4_DUAL = 0, /* 18-byte block, two half-scales (Q4_0_ROCMFP4)        */
  ROCMFP4_FAST = 1  /* 17-byte block, one scale (Q4_0_ROCMFP4_FAST)          */
} rocmfp4_variant;

typedef enum {
  ROCMFP4_ACT_F16 = 0, /* activations are IEEE binary16                     */
  ROCMFP4_ACT_BF16 = 1 /* activations are bfloat16                          */
} rocmfp4_act;

typedef enum {
  ROCMFP4_OUT_F32 = 0,
  ROCMFP4_OUT_BF16 = 1,
  ROCMFP4_OUT_F16 = 2
} rocmfp4_out_dtype;

typedef enum {
  ROCMFP4_OK = 0,
  ROCMFP4_ERR_INVALID_ARG = 1,   /* bad pointer, size or enum value          */
  ROCMFP4_ERR_UNSUPPORTED = 2,   /* valid request this build cannot serve    */
  ROCMFP4_ERR_INVALID_SCALE = 3, /* rocmfp4_validate found a non-finite scale */
  ROCMFP4_ERR_CUDA = 4           /* a CUDA call failed                        */
} rocmfp4_status;

/* Bytes of one block: 18 (ROCMFP4_DUAL), 17 (ROCMFP4_FAST), 0 otherwise.
 * ("Block Layout": 4.50 and 4.25 bits per weight.) */
size_t rocmfp4_block_bytes(rocmfp4_variant variant);

/* Bytes of one packed row of K weights (K/32 blocks); 0 on a bad argument. */
size_t rocmfp4_row_bytes(int64_t K, rocmfp4_variant variant);

/* Batch-1 decode product y = W . x.
 *   W: N x K packed ROCmFP4 matrix (N * row_bytes bytes).
 *   x: K activations, fp16.        y: N fp32 outputs, overwritten.
 * Same as rocmfp4_gemv_ex(..., ROCMFP4_ACT_F16, NULL). */
rocmfp4_status rocmfp4_gemv(const void *W, const void *x, float *y, int64_t N, int64_t K,
                            rocmfp4_variant variant);

/* y = W . x with the activation type and stream given.  x is K elements of
 * type act; y is N fp32, overwritten.  Accumulation is fp32. */
rocmfp4_status rocmfp4_gemv_ex(const void *W, const void *x, float *y, int64_t N, int64_t K,
                               rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream);

/* Y = X . W^T: X is M x K activations (row-major), W is N x K packed,
 * Y is M x N fp32 (row-major), overwritten.  Plain form: X is bf16, default
 * stream.  M <= 8 runs the small-batch streaming kernel (each weight byte read
 * once for all M vectors); larger M runs the tensor-core prefill kernel. */
rocmfp4_status rocmfp4_gemm(const void *W, const void *X, float *Y, int64_t M, int64_t N, int64_t K,
                            rocmfp4_variant variant);

rocmfp4_status rocmfp4_gemm_ex(const void *W, const void *X, float *Y, int64_t M, int64_t N,
                               int64_t K, rocmfp4_variant variant, rocmfp4_act act,
                               rocmfp4_stream_t stream);

/* Fused gate/up decode product (the "gemv_gate_up" decode matvec kernel type
 * named in "Feasibility Report: Porting ROCmFP4 to Atlas", section "Kernel
 * System"; the pages give no definition, and this is the plain reading for a
 * gated MLP):
 *
 *   Y[m][i] = SiLU(g) * u,  g = sum_k Wg[i][k] X[m][k],  u = sum_k Wu[i][k] X[m][k],
 *   SiLU(g) = g / (1 + exp(-g)),
 *
 * for i < I and m < M.  W is one packed matrix of 2I rows and K columns: rows
 * 0 .. I-1 are the gate rows Wg, rows I .. 2I-1 the up rows Wu (each row
 * K/32 blocks, as for every entry point).  X is M x K of type act
 * (row-major), Y is M x I fp32 (row-major), overwritten; g and u accumulate in
 * fp32 and never leave the kernel.
 *   - M at most 8 (decode); M > 8 returns ROCMFP4_ERR_UNSUPPORTED.
 *   - K a multiple of 256 (dual) or 512 (single-scale) and W and X 16-byte
 *     aligned, else ROCMFP4_ERR_UNSUPPORTED; K == 0 writes zeros.
 *   - Asynchronous on `stream`; arguments checked as for every entry point. */
rocmfp4_status rocmfp4_gemv_gate_up(const void *W, const void *X, float *Y, int64_t M, int64_t I,
                                    int64_t K, rocmfp4_variant variant, rocmfp4_act act,
                                    rocmfp4_stream_t stream);

/* Decode attention over a ROCmFP4 K/V cache (one query token per sequence):
 * the "FlashAttention K/V cache optimization" item of "Feasibility Report:
 * Porting ROCmFP4 to Atlas" (sections "Why AMD is Different from NVIDIA" and
 * "Option 2"), which gives no formula; this is the plain reading:
 *
 *   s_t = scale * sum_d q[b][h][d] K[b][hk][t][d],   0 <= t < lens[b],
 *   out[b][h][d] = sum_t exp(s_t - max s) V[b][hk][t][d] / sum_t exp(s_t - max s),
 *   hk = h / (H / Hkv)  (grouped-query attention; Hkv = H is plain MHA).
 *
 *   - q     [B][H][D] of type act (row-major), device;
 *   - K, V  [B][Hkv][Tmax] rows, each D/32 packed blocks of `variant`
 *           (row_bytes = D/32 * block_bytes), device, 16-byte aligned;
 *   - lens  [B] int32 on the device: tokens held by sequence b; values are
 *           clamped to [0, Tmax]; rows at or past lens[b] are never used
 *           (they need not hold valid blocks); a sequence with no token gives
 *           zeros;
 *   - out   [B][H][D] fp32, overwritten.
 *   - D must be 64 or 128, H / Hkv at most 8, Tmax a multiple of 32, else
 *     ROCMFP4_ERR_UNSUPPORTED.  Scores, softmax and the weighted sum are fp32;
 *     results are bitwise repeatable for the same shapes on the same device.
 *   - One or two kernel launches on `stream` (a combine launch when the cache
 *     is split across CTAs); the split partials use the per-device workspace. */
rocmfp4_status rocmfp4_decode_attention(const void *q, const void *K, const void *V,
                                        const int32_t *lens, float *out, int64_t B, int64_t H,
                                        int64_t Hkv, int64_t D, int64_t Tmax, float scale,
                                        rocmfp4_variant variant, rocmfp4_act act,
                                        rocmfp4_stream_t stream);

/* One product of a chain: Y = X . W^T with the layouts of rocmfp4_gemm_ex
 * (X is M x K of the chain's activation type, Y is M x N fp32). */
typedef struct rocmfp4_gemv_op {
  const void *W;
  const void *X;
  float *Y;
  int64_t N;
  int64_t K;
} rocmfp4_gemv_op;

/* Runs the products ops[0 .. count-1] in order on one stream, all with the
 * same M, variant and activation type: the result is that of calling
 * rocmfp4_gemm_ex for each in turn, and product i may read (through X)
 * memory that products 0 .. i-1 write.
 *
 * This is the decode-step form: one call for a list of products.  Each
 * product is one launch, the launch rocmfp4_gemm_ex would make, in order on
 * `stream`; streaming launches (M <= 8) are programmatic dependent launches,
 * so a product's weights, which never depend on earlier products, stream
 * while the previous product finishes, and its activations are read only
 * once the previous launch has completed.
 *   - ops is host memory read during the call; count == 0 does nothing.
 *   - Y of a product must not overlap any W, nor the X or Y of another
 *     product of the chain, except that X of a later product may be (part
 *     of) Y of an earlier one.
 *   - Errors as rocmfp4_gemm_ex, checked for every product before any
 *     launch; a launch error leaves the products before it done. */
rocmfp4_status rocmfp4_gemv_chain(const rocmfp4_gemv_op *ops, int count, int64_t M,
                                  rocmfp4_variant variant, rocmfp4_act act, rocmfp4_stream_t stream);

/* rocmfp4_gemv_chain over products whose weights have different block
 * layouts: product i's W is in layout variants[i].
 *
 * ("Tensor-Aware Presets": a model quantised with a preset mixes the 18- and
 * 17-byte layouts across tensor roles, so the engine picks the layout per
 * tensor.  The pages name six presets but list none of their contents: the
 * caller maps its tensors to layouts.)
 *   - variants is host memory of `count` entries, read during the call.
 *   - The result is that of calling rocmfp4_gemm_ex for each product in turn
 *     with its own layout, bit for bit: one launch per product, as in
 *     rocmfp4_gemv_chain.
 *   - Every product is checked (shape, layout, pointers) before any launch;
 *     otherwise arguments, aliasing rules and errors as rocmfp4_gemv_chain. */
rocmfp4_status rocmfp4_gemv_chain_mixed(const rocmfp4_gemv_op *ops, const rocmfp4_variant *variants,
                                        int count, int64_t M, rocmfp4_act act,
                                        rocmfp4_stream_t stream);

/* Y = X . W^T for M <= 8 without allocating device memory.
 *
 * For callers that cannot call cudaMalloc where they run the product: an
 * inference engine that hands all device memory to its own pool at start-up
 * (a cudaMalloc behind its back could fail, or fragment the memory it
 * planned), a host with a real-time or certification rule against
 * allocating after initialisation (allocation time is unbounded), or a
 * plug-in loaded into a process whose allocator it must not touch.  The
 * format definition has no counterpart; this is a deployment convenience.
 *
 * Same arguments, layouts and results as rocmfp4_gemm_ex (fp32 Y, fp16 or
 * bf16 X), computed by the same streaming kernel, whose scratch (split-tile
 * partial sums, hand-off counters, error word) is a fixed array of about
 * 2 MiB inside the library (every GPU that loads the library holds it until
 * the process exits) instead of a workspace allocated on first use.
 *   - M > 8 returns ROCMFP4_ERR_UNSUPPORTED (the scratch keeps partial sums
 *     for at most 8 activation rows), as do K not a multiple of 256 (dual)
 *     or 512 (single-scale), and W or X not 16-byte aligned.  K == 0 writes
 *     zeros.
 *   - The first call on a device looks up the array's device address and
 *     zeroes its counters (a cudaMemset and a device synchronisation, no
 *     allocation); make that first call before any stream capture.
 *   - Every call shares the one array per device and finds it as the last
 *     call left it: calls that overlap on the GPU (for instance on two
 *     unordered streams) race and give wrong results.  Calls ordered on one
 *     stream are safe.
 *   - A kernel that gave up waiting records it in the array's own error word;
 *     rocmfp4_device_error_bits reports and clears it (and the array's
 *     counters) without allocating. */
rocmfp4_status rocmfp4_gemm_noalloc(const void *W, const void *X, float *Y, int64_t M, int64_t N,
                                    int64_t K, rocmfp4_variant variant, rocmfp4_act act,
                                    rocmfp4_stream_t stream);

/* Quantiser: packs src (N x K values of type src_type, row-major, device)
 * into ROCmFP4 blocks W (N rows of K/32 blocks, device), the inverse of
 * rocmfp4_dequant.  "Feasibility Report: Porting ROCmFP4 to Atlas", section
 * "What is ROCmFP4?", defines the format but no scale selection or rounding;
 * the rule used (a reading):
 *   - scale groups: the two 16-weight halves of a dual block, the whole
 *     block for single-scale;
 *   - a group's scale byte e is the smallest of 0x00 .. 0x7E whose half-scale
 *     covers the group's largest magnitude (5 * E4M3(e) >= amax); larger
 *     magnitudes use 0x7E and saturate at code +-10; a group of zeros gets 0;
 *   - each value takes the nearest Codebook10 magnitude times the half-scale,
 *     a tie going to the smaller magnitude; zero is code 0; non-finite inputs
 *     count as 0.
 * Every decision is exact, so the result does not depend on the device.
 * Values already of the form Codebook10[q] * hs(e) with a code of magnitude
 * 10 in every group come back bit for bit.  Asynchronous on `stream`. */
rocmfp4_status rocmfp4_quantize(const void *src, rocmfp4_act src_type, void *W, int64_t N, int64_t K,
                                rocmfp4_variant variant, rocmfp4_stream_t stream);

/* Dense weights: out[n*K + k] = Codebook10[q] * hs(e) for every weight,
 * written as fp32, bf16 or fp16.  Every value is exactly representable in
 * all three types, so the result is exact; code 8 gives +0. */
rocmfp4_status rocmfp4_dequant(const void *W, void *out, rocmfp4_out_dtype out_dtype, int64_t N,
                               int64_t K, rocmfp4_variant variant, rocmfp4_stream_t stream);

/* Row validation ("Scale Format": non-finite scale bytes are rejected).
 * Scans every scale byte; returns ROCMFP4_OK when all are finite, else
 * ROCMFP4_ERR_INVALID_SCALE.  *first_bad_block (may be NULL) receives the
 * row-major block index n*(K/32)+b of the first offending block, or -1.
 * Synchronises with the stream before returning. */
rocmfp4_status rocmfp4_validate(const void *W, int64_t N, int64_t K, rocmfp4_variant variant,
                                int64_t *first_bad_block, rocmfp4_stream_t stream);

/* Staging copy of a decode step's inputs or outputs: copies `bytes` bytes
 * from src to dst in stream order, by a kernel.  No counterpart in the
 * format definition; it serves the single-stream decode step that the
 * products are for ("Feasibility Report: Porting ROCmFP4 to Atlas", section
 * "Kernel System", the decode matvec): a step's activations come in from the
 * host and its results go back out without a copy-engine transfer that would
 * break the chain of dependent launches.
 *   - dst and src: memory of the current device, managed memory, or pinned
 *     host memory (cudaHostAlloc, cudaMallocHost, cudaHostRegister), which
 *     the kernel reaches through its device pointer; pageable host memory
 *     and another device's memory are refused.
 *     Both are owned by the caller; the ranges must not overlap.
 *   - The kernel is a programmatic dependent launch: the next kernel on the
 *     stream may begin launching at once (a following product's weights then
 *     stream while the copy runs), and the copy reads and writes nothing
 *     before the preceding kernel on the stream has completed.
 *   - 16-byte vectors when both pointers are 16-byte aligned, else bytes.
 * bytes == 0 is a no-op.  bytes < 0, a NULL pointer, overlapping ranges,
 * pageable host memory or another device's memory give
 * ROCMFP4_ERR_INVALID_ARG; a failed pointer query or launch gives
 * ROCMFP4_ERR_CUDA.  Asynchronous on `stream`. */
rocmfp4_status rocmfp4_copy(void *dst, const void *src, int64_t bytes, rocmfp4_stream_t stream);

/* Error bits recorded by kernels on the current device since the last query
 * (bit 0: a kernel gave up waiting for its own bulk copies, so its outputs
 * are invalid), from the workspace of the allocating entry points and from
 * the fixed array of rocmfp4_gemm_noalloc, whichever exist on the device.
 * Synchronises with the stream, clears the bits, and on a non-zero result
 * also clears the split-reduction counters.  Allocates nothing: a device on
 * which no allocating entry point has run yet keeps no workspace.  Returns
 * 0xFFFFFFFF if the query itself failed. */
uint32_t rocmfp4_device_error_bits(rocmfp4_stream_t stream);

/* Static name of a status code. */
const char *rocmfp4_status_string(rocmfp4_status status);

/* Message of the last failure seen by this thread ("" if none). */
const char *rocmfp4_last_error(void);

/* Number of device kernels this library has launched in this process
 * (a counter kept by the host wrappers; used by the benchmark). */
uint64_t rocmfp4_launch_count(void);

/* Free the per-device workspaces.  Calls made afterwards recreate them. */
void rocmfp4_shutdown(void);

#ifdef __cplusplus
}
#endif

#endif /* ROCMFP4_H_ */
