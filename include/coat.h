/*
 * coat.h -- C ABI of libcoat_gb300: the fused FP8 AdamW step with Dynamic
 * Range Expansion (DRE), and the standalone DRE quantizer / dequantizer, for
 * NVIDIA GB300 (sm_103a).
 *
 * The method is COAT's ("COAT: Compressing Optimizer States and Activation
 * for Memory-Efficient FP8 Training", paper-review page on the xllm-io blog):
 *   - FP8 quantization (section 3, core formulas, "FP8量化"):
 *       X_FP8 = round(X / S),  S = max|X| / 448         (448 = E4M3 max finite)
 *   - AdamW (section 3, core formulas, "AdamW优化器更新规则"):
 *       m_t = b1 m_{t-1} + (1-b1) g_t,   v_t = b2 v_{t-1} + (1-b2) g_t^2
 *       mhat = m_t / (1-b1^t),           vhat = v_t / (1-b2^t)
 *       w_{t+1} = w_t - lr (mhat / (sqrt(vhat) + eps) + wd w_t)
 *   - Dynamic Range Expansion (section 3, "动态范围扩展"):
 *       f(x) = sign(x)|x|^k,  R_X = max|X| / min|X|,  k = log_{R_X}(R_E4M3)
 *   - the fused optimizer kernel (section 4 table, "融合优化器内核" row) and
 *     per-shard statistics with no cross-GPU sync (section 4 table, FSDP row).
 *
 * Quantized state layout (all buffers flat, owned by the caller):
 *   a tensor of n values is split into groups of G contiguous elements
 *   (the last group may be shorter).  Each value is one E4M3 byte; each group
 *   has a scale S and an exponent k.  A code q stands for
 *       x = sign(q) * (|E4M3(q)| * S)^(1/k).
 *   Quantization picks, per group, k = min(log(R_E4M3)/log(R_X), 8) with
 *   min|X| taken over the non-zero elements, lowers k further if needed so
 *   that S stays a normal float in [2^-125, 2^126], rounds k to float, sets
 *   S = max|X|^k / 448 and encodes y = 448 sign(x) (|x|/max|X|)^k with
 *   round-to-nearest-even onto the E4M3 grid, saturating at +-448 (0x7E /
 *   0xFE); a value that rounds to zero, of either sign, encodes as 0x00
 *   (never 0x80), here and in every quantizer below.  An all-zero group has S = 0, k = 1; a group
 *   with one non-zero magnitude has k = 1.  R_E4M3 = 448 / 2^-9 = 229376
 *   (see coat_r_e4m3()).
 *
 * Conventions for every entry point below:
 *   - Data pointers are DEVICE pointers (cudaMalloc / torch CUDA tensors) on
 *     the current device, 16-byte aligned -- except the state buffers of
 *     coat_fp8_adamw_step_host and coat_fp8_adamw_step_host_static, which
 *     are host pointers.  The library allocates no memory and keeps no state
 *     between calls (coat_fp8_adamw_step_host creates and destroys its three
 *     streams and one event within the call; coat_fp8_adamw_step_host_static
 *     uses a fixed device array of the library as its scratch).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call is asynchronous on that stream, except
 *     coat_fp8_adamw_step_host and coat_fp8_adamw_step_host_static, which
 *     return when their result is in host memory.
 *   - G must be a power of two in [1, 256]; 1 <= n <= COAT_MAX_N (2^40
 *     elements: far more than one device holds, and small enough that every
 *     launch's grid stays within the hardware's limits).
 *   - Argument errors return a status and launch nothing.  A failed launch
 *     returns COAT_ERR_CUDA (the CUDA error is left for the caller to query
 *     with cudaGetLastError()).  Nothing aborts, traps or prints.
 *   - Inputs must be finite; NaN/Inf inputs and the E4M3 NaN codes (0x7F,
 *     0xFF) are outside the contract.
 */
#ifndef COAT_H_
#define COAT_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    COAT_OK = 0,
    COAT_ERR_INVALID_ARG = 1,   /* null pointer, n outside [1, COAT_MAX_N], step < 1, bad hyper-parameter, aliasing */
    COAT_ERR_MISALIGNED = 2,    /* a pointer is not 16-byte aligned */
    COAT_ERR_UNSUPPORTED_G = 3, /* G not a power of two in [1, 256] */
    COAT_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed */
    COAT_ERR_NOT_DEVICE = 5,    /* a device pointer is neither memory of the current device nor managed memory */
    COAT_ERR_SCRATCH_LIMIT = 6  /* the request needs more than COAT_STATIC_SCRATCH_BYTES */
} coat_status;

/* Largest element count n any entry point accepts. */
#define COAT_MAX_N ((int64_t)1 << 40)

/* Size of the fixed device scratch buffer of coat_fp8_adamw_step_host_static. */
#define COAT_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* Per-group record of the quantized optimizer state: 16 bytes, one per group,
 * scale and exponent of the first moment, then of the second moment. */
typedef struct {
    float m_scale;
    float m_k;
    float v_scale;
    float v_k;
} coat_group_meta;

/*
 * One fused AdamW + DRE step over a flat parameter buffer, in one pass over
 * HBM (COAT review page, section 3 core formulas and section 4 "fused
 * optimizer kernel").  For every group of G elements it dequantizes m and v,
 * undoes the expansion, applies the AdamW update above to w from the bf16
 * gradient g, recomputes the group's k and S for both moments from the new
 * fp32 moments and re-quantizes them.
 *
 *   w       [n] float32, in/out: master weights, updated in place.
 *   g       [n] bfloat16 (raw 16-bit patterns), in: gradient of this step.
 *   m_q,v_q [n] uint8, in/out: E4M3 codes of the first / second moment.
 *   meta    [ceil(n/G)] coat_group_meta, in/out.
 *   n, G    element count and group size.
 *   beta1, beta2 in [0,1); lr >= 0; eps > 0; weight_decay >= 0; all finite.
 *   step    t >= 1, the index of this update (bias correction uses b^t).
 *
 * First use: m_q = v_q = 0 and meta = {0, 1, 0, 1} for every group.
 * g must not overlap any output buffer.  The moments used in the weight
 * update are the fp32 values before re-quantization.
 */
coat_status coat_fp8_adamw_step(float *w, const uint16_t *g, uint8_t *m_q, uint8_t *v_q,
                                coat_group_meta *meta, int64_t n, int32_t G, float beta1,
                                float beta2, float lr, float eps, float weight_decay,
                                int64_t step, void *stream);

/*
 * The same step with the optimizer state and the gradient in HOST memory
 * (state offloading).  w, g, m_q, v_q and meta are host pointers, laid out as
 * for coat_fp8_adamw_step; page-locked (pinned) memory lets the copies run
 * asynchronously and overlap, pageable memory works but is slower.  The
 * state is streamed through `workspace` (device memory owned by the caller,
 * 256-byte aligned, `workspace_bytes` long) in chunks of equal size, a
 * multiple of 4096 parameters: host->device copies, the kernel and
 * device->host copies of consecutive chunks run on three internal streams
 * that start after the work already queued on `stream`.  The call returns
 * once the host buffers hold the updated state (or on error); the result is
 * bit-identical to coat_fp8_adamw_step on device copies of the same buffers.
 * COAT_ERR_INVALID_ARG also covers: a state buffer that is device memory, a
 * workspace too small for one chunk (see coat_fp8_adamw_step_host_workspace_bytes).
 */
coat_status coat_fp8_adamw_step_host(float *w, const uint16_t *g, uint8_t *m_q, uint8_t *v_q,
                                     coat_group_meta *meta, int64_t n, int32_t G, float beta1,
                                     float beta2, float lr, float eps, float weight_decay,
                                     int64_t step, void *workspace, size_t workspace_bytes,
                                     void *stream);

/* Workspace bytes coat_fp8_adamw_step_host needs to stream chunks of
 * `chunk_params` parameters (rounded up to a multiple of 4096); 0 for a bad G. */
size_t coat_fp8_adamw_step_host_workspace_bytes(int64_t chunk_params, int32_t G);

/*
 * coat_fp8_adamw_step_host for callers that cannot allocate device memory.
 * The COAT review page has no counterpart: this entry point serves how the
 * library is deployed, not the method.
 *
 * Who needs it: a process whose caching allocator already holds the device
 * memory it may use (a workspace allocation would fail or fragment it), code
 * that must not call cudaMalloc / cudaFree between steps (both can
 * synchronize the whole device), and runtimes whose device footprint is fixed
 * at start-up.  Instead of a caller's workspace, the step streams the state
 * through a scratch buffer of COAT_STATIC_SCRATCH_BYTES (16 MiB) that is a
 * file-scope __device__ array of the library: the CUDA runtime reserves it on
 * a device when the library's module that holds it is loaded there.  The
 * call allocates no memory (no cudaMalloc, no allocating library routine)
 * and creates no stream or event.
 *
 * Everything runs on `stream`, one chunk after another: host->device copies,
 * the step kernel, device->host copies.  Copies and compute do not overlap;
 * where a workspace can be allocated, coat_fp8_adamw_step_host is faster.  The
 * call returns once the host buffers hold the result, which is bit-identical
 * to coat_fp8_adamw_step on device copies of the same buffers.
 *
 *   w, g, m_q, v_q, meta, n, G, beta1, beta2, lr, eps, weight_decay, step:
 *                 as for coat_fp8_adamw_step_host (host pointers).
 *   chunk_params  parameters per chunk, rounded up to a multiple of 4096;
 *                 0 = the largest chunk that fits the scratch (about 2.06
 *                 million parameters at G = 128, about 0.7 million at G = 1).
 *
 * Set-up: every call looks up the scratch's device address on the current
 * device (cudaGetSymbolAddress, which allocates nothing; the address is not
 * cached, so a device reset between calls is safe).  The first call on a
 * device may load the library's module there: make that first call before
 * any stream capture begins.  `stream` must belong to the current device
 * (COAT_ERR_INVALID_ARG otherwise, before anything is copied).  Nothing in
 * the scratch has to start at zero: each chunk's bytes are copied in by the
 * same call before the kernel reads them.
 * One scratch per device: calls that overlap in time on one device (from
 * several host threads, or on several streams) race on it; the caller must
 * serialize them.
 * Errors: COAT_ERR_SCRATCH_LIMIT when one chunk of chunk_params parameters
 * needs more than COAT_STATIC_SCRATCH_BYTES (nothing is copied or launched);
 * otherwise as coat_fp8_adamw_step_host.
 */
coat_status coat_fp8_adamw_step_host_static(float *w, const uint16_t *g, uint8_t *m_q,
                                            uint8_t *v_q, coat_group_meta *meta, int64_t n,
                                            int32_t G, float beta1, float beta2, float lr,
                                            float eps, float weight_decay, int64_t step,
                                            int64_t chunk_params, void *stream);

/*
 * DRE + E4M3 quantization of one fp32 tensor (COAT review page, section 3,
 * FP8 quantization and Dynamic Range Expansion equations).
 *   x [n] float32 in;  q [n] uint8 out;  scale, k [ceil(n/G)] float32 out.
 * x must not overlap the outputs.
 */
coat_status coat_dre_quantize(const float *x, int64_t n, int32_t G, uint8_t *q, float *scale,
                              float *k, void *stream);

/*
 * Per-group FP8 quantization WITHOUT the expansion (COAT review page,
 * section 3, the FP8 quantization equation alone): scale = max|X| / 448
 * rounded to float, q = E4M3(X / scale) rounded to nearest even and saturating
 * at +-448; an all-zero group gets scale 0 and zero codes.  It is the plain
 * per-group FP8 storage that Dynamic Range Expansion is measured against
 * (the section 4 table credits the expansion with a 1.63x lower quantization
 * MSE).  Decode with coat_dre_dequantize and k = 1 for every group.
 *   x [n] float32 in;  q [n] uint8 out;  scale [ceil(n/G)] float32 out.
 */
coat_status coat_fp8_quantize_absmax(const float *x, int64_t n, int32_t G, uint8_t *q,
                                     float *scale, void *stream);

/*
 * Per-group (1 x G) FP8 quantization of an activation with a transposed FP8
 * second output (COAT review page: section 3, Triton kernels, "non-linear
 * layer optimisation": a quantized FP8 output plus a transposed FP8 output for
 * the backward pass; section 3, mixed-granularity activation quantization:
 * 1 x G groups for non-linear layers; section 4 table, group-scaling row:
 * two-stage maximum; the section 5 group-size table sweeps G = 4 ... 64 and
 * 1 x 128).  Each row of x is split into groups
 * of G consecutive elements: scale = max|x| / 448 rounded to float, and
 * q = E4M3(x / scale) rounded to nearest even, saturating; an all-zero group
 * has scale 0 and zero codes.
 *   x      [M x N] bfloat16 (raw 16-bit patterns), row-major, in.
 *   q      [M x N] uint8 out: the codes in the layout of x.
 *   qt     [N x M] uint8 out: the same codes transposed (qt[c*M + r] = q[r*N + c]);
 *          NULL to skip it.
 *   scale  [M x N/G] float32 out, row-major (group g of row r at r*N/G + g).
 *   G a power of two in [4, 128]; M and N multiples of 16; N a multiple of G;
 *   M <= 4,194,240 (65535 tiles of 64 rows).
 * The outputs must not overlap x or each other.
 */
coat_status coat_act_quantize_fp8(const uint16_t *x, int64_t M, int64_t N, int32_t G, uint8_t *q,
                                  uint8_t *qt, float *scale, void *stream);

/*
 * FP8 linear layer whose output is already the next layer's per-group FP8
 * activation (COAT review page, section 3: "mixed-granularity activation
 * quantization" gives linear layers per-tensor FP8 inputs; "Triton kernels",
 * linear layer optimisation, quantizes the GEMM's output tile per 1 x G group
 * in the epilogue).
 *   xq [M x K] uint8 E4M3 codes in, row-major, X = sx E4M3(xq);
 *   wq [N x K] uint8 E4M3 codes in, row-major (the weight as stored by a
 *      linear layer, out_features x in_features), W = sw E4M3(wq);
 *   y = X W^T accumulated in float32 on the tensor cores, one float32 product
 *      by RN(sx sw) at the end;
 *   per row, per group of G consecutive columns: scale = RN(max|y| / 448),
 *      q = E4M3(y / scale) (nearest even of the exact quotient, saturating);
 *      a group of zeros has scale 0 and zero codes;
 *   q [M x N] uint8 out;  scale [M x N/G] float32 out (group g of row r at
 *      r*N/G + g);  y [M x N] float32 out, or NULL to skip writing it.
 * sx, sw finite and > 0; G a power of two in [8, 128]; N a multiple of 16
 * and of G; K a multiple of 16; M, N, K below 2^31 (M, N and K need not be
 * multiples of the kernel's tiles).  All pointers 16-byte aligned device
 * memory of the current device; the outputs overlap neither the inputs nor
 * each other.  Asynchronous on `stream`.  The kernel waits on its own
 * pipeline with bounded waits; a wait that gives up (which would be a bug)
 * leaves the outputs unspecified and is counted by coat_kernel_wait_timeouts.
 */
coat_status coat_fp8_linear_group_quantize(const uint8_t *xq, float sx, const uint8_t *wq, float sw,
                                           int64_t M, int64_t N, int64_t K, int32_t G, uint8_t *q,
                                           float *scale, float *y, void *stream);

/*
 * Inverse of coat_dre_quantize: x = sign(q) (|E4M3(q)| scale)^(1/k).
 *   q [n] uint8 in;  scale, k [ceil(n/G)] float32 in (k > 0);  x [n] float32 out.
 */
coat_status coat_dre_dequantize(const uint8_t *q, const float *scale, const float *k, int64_t n,
                                int32_t G, float *x, void *stream);

/*
 * Diagnostics of the step's correctly rounded exact path.  The step
 * re-evaluates every group's extreme moments and its exponent k in
 * double-float arithmetic and rounds each once to float32 (COAT review page,
 * section 3: the dequantized state is an fp32 tensor X_FP32, and k and S follow
 * from the group's max|X| and min|X|).  When a double-float value lies too close
 * to an fp32 rounding midpoint for that rounding to be certain, the value is
 * recomputed in float64 from its definition.  This call reads how often that
 * happened on the current device since the library was loaded there (or since
 * the last reset):
 *   counts[0]  dequantized moments recomputed,
 *   counts[1]  exponents k recomputed.
 * reset != 0 clears both counters after reading them.  The call synchronizes
 * with the current device (it copies from device memory) and must not overlap
 * a running step if exact counts are wanted.
 */
coat_status coat_exact_recompute_counts(uint64_t counts[2], int32_t reset);

/*
 * How many bounded waits inside the library's kernels gave up on the current
 * device since the library was loaded there (or since the last reset).  The
 * pipelined kernels (coat_fp8_linear_group_quantize) wait on their own
 * producers with an iteration limit instead of forever; a non-zero count
 * means a launch returned without finishing its work.  reset != 0 clears the
 * counter after reading it.  Synchronizes with the current device.
 */
coat_status coat_kernel_wait_timeouts(uint64_t *count, int32_t reset);

/* Static description of a status code (never NULL). */
const char *coat_status_string(coat_status status);

/* The R_E4M3 the library uses: 448 / 2^-9 = 229376. */
double coat_r_e4m3(void);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int32_t coat_version(void);

#ifdef __cplusplus
}
#endif

#endif /* COAT_H_ */
