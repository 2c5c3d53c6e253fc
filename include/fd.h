/*
 * fd.h - C ABI of the fused memory-bound decode kernels for GB300 (sm_103a).
 *
 * Two operations of an LLM decode layer, each one kernel launch:
 *
 *   fd_swiglu_w4a16_gemv   y = (silu(g) * u) . dequant(W_int4)^T   ("GEMM prologue
 *                          fusion": the activation and the int4 dequantisation are done
 *                          as the weights stream in; the (M, K, N) product and the
 *                          silu/mul intermediate never exist in memory).
 *   fd_add_rmsnorm         h = x + residual; out = RMSNorm(h) * weight  (one kernel, two
 *                          outputs: the new residual h and the normalised row).
 *   fd_swiglu_w4a16_gemv_residual
 *                          the same GEMV with a residual-add epilogue: out = residual + y
 *                          (the down projection of a fused layer writes the new residual).
 *   fd_w4a16_gate_up_gemv  the horizontally fused gate and up projections of the MLP, one
 *                          W4A16 GEMV over both weight matrices ("horizontal fusion"):
 *                          one read of x, g and u written for the down projection.
 *   fd_swiglu_w4a16_gemv_add_rmsnorm
 *                          the down projection with the next layer's add + RMSNorm folded
 *                          into its tail (one launch per decode layer instead of two).
 *   fd_nvfp4_scaled_mm     the NVFP4 (packed FP4, E4M3 1x16 block scales) matmul of batched
 *                          decode with its fp32 output multiplier folded in, on the
 *                          tensor cores' block-scaled MMA.
 *   fd_decode_mlp_step     a whole decode step (add-RMSNorm + down projection per layer)
 *                          as one persistent launch, bit-identical to the chain of calls.
 *
 * Sources (web pages, cited by title and section):
 *   [FIX]  "PyTorch Community Proposes Fusion Fix as Large Intermediate Buffers May Slow
 *          Single-Token Decoding in Quantized LLMs" - "Reproduction and analysis" (the
 *          (1, K, N) product an M=1 matmul must not materialise), "Fix proposal" (int4
 *          weights with a SwiGLU pre-operation).
 *   [FUSE] "09 - Operator fusion" - section 5, "The taxonomy of fusions" (items 2 and 4:
 *          reduction + elementwise; GEMM prologue dequantisation for W4A16; item 3: GEMM
 *          epilogue fusion; item 5: horizontal fusion, gate_proj and up_proj as one
 *          gate_up_proj) and "The fusion boundary problem" (add_rmsnorm with two
 *          outputs; act @ W_down; kernel 3: the down projection with a residual-add
 *          epilogue that writes new_residual = x + out).
 *   [KFM]  "Kernel Fusion, torch.compile and CUDA Graphs, Measured" - "Step 1" (silu(g) *
 *          u), "Step 2: fusing them by hand in Triton" (add + RMSNorm order and roundings).
 *   [NVFP4] "PyTorch folds NVFP4 output scaling into NVGEMM candidates for decode
 *          workloads" - body and metrics table (the scaled FP4 matmul and the fold of its
 *          output multiplier).
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer (cudaMalloc / PyTorch CUDA memory) on the
 *     current device, contiguous, row-major, 16-byte aligned. The caller allocates and
 *     owns every buffer. The library allocates no memory and keeps no state beyond a
 *     per-device cache of the SM count.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls are
 *     asynchronous and stream-ordered: no host synchronisation, no host<->device copy.
 *   - bf16 is IEEE bfloat16 stored as 16-bit words.
 *   - Arguments are checked on the host before anything is launched. A bad call
 *     returns a nonzero fd_status and launches nothing. A failed launch returns
 *     FD_ERR_CUDA (from cudaGetLastError); faults inside a kernel surface, as in CUDA,
 *     at the caller's next synchronisation.
 *   - All entry points are thread-safe.
 */
#ifndef FD_H_
#define FD_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *fd_stream_t;

typedef enum fd_status {
    FD_OK = 0,
    FD_ERR_NULL = 1,        /* a required pointer is NULL */
    FD_ERR_SHAPE = 2,       /* a size is negative, zero where it may not be, or breaks a
                               divisibility rule */
    FD_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
    FD_ERR_UNSUPPORTED = 4, /* a size is above the supported maximum */
    FD_ERR_CUDA = 5,        /* the CUDA runtime reported an error */
    FD_ERR_OVERLAP = 6      /* outputs overlap inputs in a way the kernel does not allow */
} fd_status;

/* Largest supported sizes (checked, FD_ERR_UNSUPPORTED above them). */
#define FD_MAX_K 32768        /* gemv: reduction length */
#define FD_MAX_M 256          /* gemv: activation rows (batched decode) */
#define FD_MAX_HIDDEN 32768   /* add_rmsnorm: row length */

/*
 * fd_swiglu_w4a16_gemv - SwiGLU-prologue W4A16 matrix-vector / skinny-matrix product.
 *
 *   a[m, k]  = silu(gate[m, k]) * up[m, k],   silu(x) = x / (1 + exp(-x))      [KFM Step 1]
 *   W[n, k]  = q[n, k] * scales[n, k / group]                                 [FUSE item 4]
 *   out[m, n] = bf16( sum_k a[m, k] * W[n, k] )   (fp32 accumulation, one RNE rounding)
 *
 * gate, up  bf16 [M, K] row-major.
 * qweight   int32 [N, K/8] row-major (nn.Linear [out, in] orientation). Nibble j
 *           (bits 4j..4j+3) of word p in row n holds q[n, 8p + j] as a 4-bit two's
 *           complement integer in [-8, 7] (symmetric, no zero point).
 * scales    bf16 [N, K/group] row-major; group consecutive k share one scale.
 * out       bf16 [M, N] row-major. Must not overlap any input.
 * Requires  0 <= M <= FD_MAX_M, 32 <= K <= FD_MAX_K, N >= 0, K % 32 == 0,
 *           group % 32 == 0, K % group == 0.
 * Empty     M == 0 or N == 0 (with valid K and group) returns FD_OK at once: no
 *           pointer is read (any may be NULL) and nothing is launched.
 * The silu/mul intermediate and the dequantised weights are kept on chip; the kernel
 * reads each packed weight word from HBM once per call.
 */
int fd_swiglu_w4a16_gemv(const void *gate, const void *up, const void *qweight,
                         const void *scales, void *out, int M, int K, int N, int group,
                         fd_stream_t stream);

/*
 * fd_swiglu_w4a16_gemv_residual - fd_swiglu_w4a16_gemv with a residual-add epilogue
 * ("kernel 3" of a fused layer, [FUSE] "The fusion boundary problem"; GEMM epilogue
 * fusion, [FUSE] item 3):
 *
 *   out[m, n] = bf16( f32(residual[m, n]) + sum_k a[m, k] * W[n, k] )   (one RNE rounding)
 *
 * The sum is the fp32 accumulator of fd_swiglu_w4a16_gemv: the product is not rounded to
 * bf16 before the add (eager PyTorch would round twice, out = bf16(bf16(y) + residual)).
 * residual  bf16 [M, N] row-major: x, the pre-norm residual stream of the layer (the
 *           residual_out of fd_add_rmsnorm).
 * out       bf16 [M, N]: the new residual. out == residual (exactly the same pointer, in
 *           place) is allowed; any other overlap of out with an input, or of residual
 *           with gate, up, qweight or scales, returns FD_ERR_OVERLAP.
 * Other arguments, requirements and the kernels used are those of fd_swiglu_w4a16_gemv.
 */
int fd_swiglu_w4a16_gemv_residual(const void *gate, const void *up, const void *qweight,
                                  const void *scales, const void *residual, void *out, int M,
                                  int K, int N, int group, fd_stream_t stream);

/*
 * fd_w4a16_gate_up_gemv - the gate and up projections of the MLP as one W4A16 GEMV
 * ([FUSE] item 5, horizontal fusion: gate_proj and up_proj become one gate_up_proj;
 * "The fusion boundary problem": gate, up = h @ W_gate_up):
 *
 *   W[n, k]          = q[n, k] * scales[n, k / group],   n < 2I (rows 0..I-1: gate,
 *                                                         rows I..2I-1: up)
 *   gate_out[m, j]   = bf16( sum_k x[m, k] * W[j, k] )
 *   up_out[m, j]     = bf16( sum_k x[m, k] * W[I + j, k] )   (fp32 accumulation)
 *
 * x          bf16 [M, K] row-major (the normalised row, out of fd_add_rmsnorm).
 * qweight    int32 [2I, K/8], the gate projection's I rows followed by the up
 *            projection's I rows, each in the nibble layout of fd_swiglu_w4a16_gemv.
 * scales     bf16 [2I, K/group].
 * gate_out, up_out  bf16 [M, I] row-major; they may not overlap each other or an input.
 * Requires   0 <= M <= FD_MAX_M, 32 <= K <= FD_MAX_K, I >= 0, K % 32 == 0,
 *            group % 32 == 0, K % group == 0. M == 0 or I == 0 is an empty call:
 *            FD_OK at once, no pointer read, nothing launched.
 * gate_out and up_out are the gate and up inputs of fd_swiglu_w4a16_gemv(_residual): the
 * two calls are the whole MLP, and silu(g) * u exists only in the second kernel's
 * registers. x is encoded per 32-k slice like the SwiGLU activation (block-scaled int16).
 * No tensor-core kernel: every M runs on the CUDA-core kernels.
 */
int fd_w4a16_gate_up_gemv(const void *x, const void *qweight, const void *scales,
                          void *gate_out, void *up_out, int M, int K, int I, int group,
                          fd_stream_t stream);

/*
 * fd_swiglu_w4a16_gemv_add_rmsnorm - one decode layer's SwiGLU-W4A16 down projection with
 * the NEXT layer's residual add + RMSNorm folded into its tail ("09 - Operator fusion",
 * "The fusion boundary problem": the down projection's output joins the residual stream at
 * the next add_rmsnorm, whose two outputs are the new residual and the normalised row):
 *
 *   y[n]            = bf16( sum_k silu(g[k]) * u[k] * W[n, k] )       (fd_swiglu_w4a16_gemv)
 *   residual_out[n] = h[n] = bf16( f32(y[n]) + f32(residual[n]) )
 *   normed[n]       = bf16( f32(bf16( h[n] * rstd )) * f32(rms_weight[n]) ),
 *                     rstd = 1 / sqrt( (1/N) sum_n h[n]^2 + eps )        (fd_add_rmsnorm)
 *
 * One activation row (M = 1). gate, up bf16 [1, K]; qweight, scales as fd_swiglu_w4a16_gemv;
 * y, residual, residual_out, normed bf16 [1, N]; rms_weight bf16 [N]. residual_out ==
 * residual (in place) is allowed; any other overlap of an output with an input or another
 * output returns FD_ERR_OVERLAP.
 * scratch  device memory of FD_FOLD_SCRATCH_BYTES bytes, 16-byte aligned, ZERO before its
 *          first use; every completed call leaves it zero again. Each CTA of the GEMV writes
 *          its partial sum of h^2 there and takes a ticket from a counter in it; the CTA that
 *          draws the last ticket normalises the row and resets the counter, so no CTA waits
 *          for another. Calls that share a scratch buffer must not run concurrently (use one
 *          stream, or one buffer per stream).
 * Requires K, N, group as fd_swiglu_w4a16_gemv, N % 8 == 0, eps >= 0 and finite. N == 0 is an
 *          empty call: FD_OK at once, no pointer read, nothing launched.
 * Runs the bulk-copy GEMV kernel with the fold where it applies (kernel selection AUTO or
 * BULK, K % 1024 == 0, K <= 15360, (K / group) % 8 == 0); otherwise the selected GEMV kernel
 * followed by fd_add_rmsnorm's kernel (same results up to the order of the sum of squares;
 * the scratch is not touched).
 */
#define FD_FOLD_SCRATCH_BYTES 4096
int fd_swiglu_w4a16_gemv_add_rmsnorm(const void *gate, const void *up, const void *qweight,
                                     const void *scales, void *y, const void *residual,
                                     const void *rms_weight, float eps, void *normed,
                                     void *residual_out, void *scratch, int K, int N, int group,
                                     fd_stream_t stream);

/*
 * fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc - fd_swiglu_w4a16_gemv_add_rmsnorm without the
 * scratch argument: the call allocates nothing and needs no buffer from the caller. It is
 * for callers that cannot allocate device memory when they make the call: code that runs
 * while its stream is being captured into a CUDA graph (cudaMalloc is not a stream
 * operation and is not allowed during capture), a plugin run inside another runtime that
 * gives its plugins no allocator (an engine that plans all of its device memory ahead), or a
 * process whose device memory belongs to an arena it does not control. The source pages
 * have no counterpart of it; it serves these callers only.
 *
 * Results, arguments, requirements and the kernel choice are those of
 * fd_swiglu_w4a16_gemv_add_rmsnorm (gate, up, qweight, scales, y, residual, rms_weight, eps,
 * normed, residual_out, K, N, group, stream: the same meaning, layouts and rules).
 * Scratch    the library's own device array of FD_FOLD_SCRATCH_BYTES bytes (a counter and
 *            one fp32 partial sum per CTA, so at most 960 CTAs), in the memory of every GPU
 *            that loads this library until the process exits. The first call on a device
 *            looks up its device address (cudaGetSymbolAddress) and zeroes it on `stream`;
 *            make that first call before any stream capture. Every call shares the array
 *            and leaves its counter at zero: calls that overlap on the GPU (other streams,
 *            or other host threads on one device) race on it and must not be made.
 * Returns    FD_ERR_UNSUPPORTED, launching nothing, when the fold's grid would need more
 *            partial sums than the array holds (a device with more than 240 SMs). Where the
 *            fold's kernel does not run the shape, the GEMV kernel and fd_add_rmsnorm's
 *            kernel run instead; they use no scratch. No cudaMalloc, cudaFree or other
 *            allocating call is made.
 */
int fd_swiglu_w4a16_gemv_add_rmsnorm_noalloc(const void *gate, const void *up,
                                             const void *qweight, const void *scales, void *y,
                                             const void *residual, const void *rms_weight,
                                             float eps, void *normed, void *residual_out, int K,
                                             int N, int group, fd_stream_t stream);

/*
 * fd_decode_mlp_step - a whole decode step of n_layers layers in one launch:
 *     for l in 0 .. n_layers - 1:
 *         h = bf16(x_l + residual); residual = h; normed_l = add-RMSNorm(h) * rms_weight_l
 *         y_l = swiglu_w4a16_gemv(gate_l, up_l, qweight_l, scales_l);  x_{l+1} = y_l
 * with x_0 = x0: the chain of fd_add_rmsnorm (rows = 1) and fd_swiglu_w4a16_gemv (M = 1)
 * calls of "Kernel Fusion, torch.compile and CUDA Graphs, Measured", Step 4 (the step run
 * as one unit instead of per-kernel launches), and every output is bit-identical to that
 * chain of separate calls: the same row partition, reduction orders and roundings.
 * A persistent cooperative kernel: one CTA per SM for all layers, each streaming the next
 * layer's weight rows while the current layer finishes. Each CTA publishes h of its rows
 * as words tagged with the layer and counts in; every CTA, once all have counted in and it
 * has read the whole tagged row, computes the next add-RMSNorm over the whole row (the row
 * kernel's reduction order). A CTA reads layer l+1's activations only when it holds the
 * complete normed_{l+1} row, as the chain's GEMV starts only after its add-RMSNorm has
 * finished.
 * layers      DEVICE array of n_layers fd_step_layer (below); the library does not read it on
 *             the host. Every pointer in it must be a device pointer, 16-byte aligned; the
 *             tensors have the layouts of fd_swiglu_w4a16_gemv (K = inter, N = hidden,
 *             M = 1) and fd_add_rmsnorm (rows = 1); y_l, normed_l and residual must not
 *             overlap one another or any input.
 * n_layers    1 .. FD_STEP_MAX_LAYERS.
 * x0          bf16 [hidden], the first layer's input (not written).
 * residual    bf16 [hidden], in and out: the residual stream, left as h of the last layer.
 * eps         the RMSNorm epsilon (finite, >= 0).
 * hidden      the model width (the GEMV's N and the RMSNorm row), a multiple of 8.
 * inter       the GEMV's K: 14336 with group 128 (the decode shape).
 * scratch     device buffer of at least FD_STEP_SCRATCH_BYTES(n_layers, hidden) bytes,
 *             16-byte aligned, owned by the caller: one counter per layer, then two rows of
 *             tagged h words (32 bits per element). The call zeroes it on `stream` first;
 *             concurrent calls need separate buffers.
 * Returns FD_OK; FD_ERR_NULL, FD_ERR_SHAPE, FD_ERR_ALIGN, FD_ERR_OVERLAP (x0, residual,
 * scratch) for bad arguments, launching nothing; FD_ERR_UNSUPPORTED, launching nothing, for
 * another inter/group, a hidden above 64 rows per SM (9728) or above 8192 (the add-RMSNorm
 * row's 256 threads x 4 vectors), or rows that do not fit one CTA's shared memory (all of
 * a CTA's weight rows stay resident: at most 29 rows per SM, hidden <= 4408 on 152 SMs;
 * fd_debug_plan_step gives the plan);
 * FD_ERR_CUDA if the launch fails (for example when the device cannot hold one CTA per SM at
 * once).
 * A wait that gives up (about a second) writes NaN outputs and sets
 * FD_DEVICE_STATUS_WAIT_TIMEOUT (fd_device_status). Capturable in a CUDA graph (a memset and
 * one kernel node).
 */
typedef struct fd_step_layer {
    const void *gate;       /* bf16 [inter] */
    const void *up;         /* bf16 [inter] */
    const void *qweight;    /* int32 [hidden, inter / 8] */
    const void *scales;     /* bf16 [hidden, inter / group] */
    const void *rms_weight; /* bf16 [hidden] */
    void *normed;           /* bf16 [hidden], out: the layer's normalised row */
    void *y;                /* bf16 [hidden], out: the layer's GEMV output */
} fd_step_layer;
#define FD_STEP_MAX_LAYERS 1024
/* the scratch: n_layers 32-bit counters padded to 16 bytes, then two rows of 32-bit tagged
 * words */
#define FD_STEP_SCRATCH_HROWS_OFFSET(n_layers) ((((size_t)(n_layers) * 4 + 15) / 16) * 16)
#define FD_STEP_SCRATCH_BYTES(n_layers, hidden) \
    (FD_STEP_SCRATCH_HROWS_OFFSET(n_layers) + (size_t)(hidden) * 8)
int fd_decode_mlp_step(const fd_step_layer *layers, int n_layers, const void *x0,
                       void *residual, float eps, int hidden, int inter, int group,
                       void *scratch, fd_stream_t stream);

/*
 * fd_add_rmsnorm - fused residual add + RMSNorm, one pass over HBM.     [KFM Step 2]
 *
 *   h[i, j]   = bf16( f32(x[i, j]) + f32(residual[i, j]) )            -> residual_out
 *   rstd[i]   = 1 / sqrt( (1/hidden) * sum_j f32(h[i, j])^2 + eps )   (fp32)
 *   out[i, j] = bf16( f32(bf16( f32(h[i, j]) * rstd[i] )) * f32(weight[j]) )
 *
 * The two roundings of out follow the page's kernel (normalised value rounded to bf16,
 * then multiplied by the weight).
 * x, residual         bf16 [rows, hidden] row-major.
 * weight              bf16 [hidden].
 * out, residual_out   bf16 [rows, hidden] row-major.
 * Aliasing            residual_out == residual and/or out == x (exactly the same pointer)
 *                     are allowed; any other overlap returns FD_ERR_OVERLAP.
 * Requires            rows >= 0, 8 <= hidden <= FD_MAX_HIDDEN, hidden % 8 == 0,
 *                     eps >= 0 and finite. rows == 0 is an empty call: FD_OK at once,
 *                     no pointer read, nothing launched.
 * Reads 4 bytes and writes 4 bytes per element (plus the weight row once per CTA).
 */
int fd_add_rmsnorm(const void *x, const void *residual, const void *weight, float eps,
                   void *out, void *residual_out, int rows, int hidden,
                   fd_stream_t stream);

/*
 * Kernel selection for fd_swiglu_w4a16_gemv (process-wide, thread-safe; default AUTO).
 *   FD_GEMV_AUTO     M >= 16: the tensor-core kernel where its layout rules hold
 *                    (K % 1024 == 0, N % 128 == 0, group % 64 == 0, (K / group) % 8 == 0);
 *                    otherwise the CUDA-core bulk-copy kernel where its rules hold
 *                    (K % 1024 == 0, K <= 15360, (K / group) % 8 == 0), else the
 *                    CUDA-core ring kernel.
 *   FD_GEMV_CUDA_CORE  always the per-thread cp.async ring kernel (any valid shape).
 *   FD_GEMV_BULK     the bulk-copy kernel where it applies, else the ring kernel.
 *   FD_GEMV_TENSOR   the tensor-core kernel where its rules hold (any M), else as AUTO
 *                    for M < 16.
 * The CUDA-core paths compute the activation in fp32 and the weights exactly; the
 * tensor-core path rounds both MMA operands, silu(g) * u and q * s, to bf16 (fp32
 * accumulation). Every path meets the documented tolerance; the choice exists for tests
 * and for measuring one kernel against another. Returns FD_ERR_UNSUPPORTED for an
 * unknown value.
 */
#define FD_GEMV_AUTO 0
#define FD_GEMV_CUDA_CORE 1
#define FD_GEMV_BULK 2
#define FD_GEMV_TENSOR 3
int fd_set_gemv_path(int path);
int fd_get_gemv_path(void);

/* 1 if fd_swiglu_w4a16_gemv, under the current kernel selection, runs this shape on the
 * tensor-core kernel (whose operands are rounded to bf16), else 0. Host-only; no CUDA
 * call. */
int fd_gemv_uses_tensor_cores(int M, int K, int N, int group);

/*
 * Launch options (process-wide, thread-safe; default 0).
 *   FD_LAUNCH_PDL  launch with programmatic dependent launch: a kernel may begin while
 *                  the previous kernel in the same stream is still running. Each fd
 *                  kernel waits (griddepcontrol.wait) before it reads activations or
 *                  writes any output; the GEMV kernels read their weights only after it,
 *                  but add-RMSNorm loads its weight row BEFORE that wait. Set this only
 *                  when no kernel that may still be running in the stream writes that
 *                  weight row (true for model weights during decode). Works inside CUDA graph
 *                  capture (the edges become programmatic dependencies).
 * fd_set_launch_flags returns FD_ERR_UNSUPPORTED for unknown bits.
 */
#define FD_LAUNCH_PDL 1u
/* Test only: every call that would launch work instead returns FD_ERR_CUDA, with
 * fd_last_cuda_error() = cudaErrorLaunchOutOfResources, without calling CUDA (the error
 * path of a failed launch, exercised without touching the GPU). */
#define FD_LAUNCH_TEST_FAIL 256u
/* Test only: the bulk-copy GEMV kernel (the M = 1 kernel of FD_GEMV_AUTO and FD_GEMV_BULK)
 * gives its waits a limit of about 2^20 SM clocks instead of about 2^31 and its copy thread
 * leaves the first weight chunk of every CTA uncopied, so the waits for that chunk run out:
 * the call's outputs are NaN and fd_device_status reports FD_DEVICE_STATUS_WAIT_TIMEOUT. No
 * fault and no hang: every wait is bounded and no copy is left in flight.
 * fd_decode_mlp_step under this flag: the same short limit, and one CTA never adds itself to
 * the first layer's count, so every CTA's wait for that count runs out; layer 0's y and
 * normalised row are correct, every later output and the residual are NaN, and the status
 * reports FD_DEVICE_STATUS_WAIT_TIMEOUT. */
#define FD_LAUNCH_TEST_WAIT_TIMEOUT 512u
int fd_set_launch_flags(unsigned flags);
unsigned fd_get_launch_flags(void);

/*
 * fd_device_status - failures that kernels of this library recorded on the current device
 * since the last clear. Every wait inside a kernel is bounded (about a second); a CTA whose
 * wait gives up stops, waits (bounded) for the copies it issued, makes the call's outputs
 * NaN and sets FD_DEVICE_STATUS_WAIT_TIMEOUT in a device status word, so the context stays
 * usable and the failure is visible to the host.
 * stream  the status is read after the work already in `stream` (a cudaStream_t; NULL = the
 *         legacy default stream); this call synchronises that stream.
 * status  out: the OR of the recorded FD_DEVICE_STATUS_* bits (0: none).
 * clear   nonzero: reset the word after reading it.
 * Returns FD_ERR_NULL for a NULL `status`, FD_ERR_CUDA if a copy or the synchronisation
 * fails. Not capturable in a CUDA graph (it synchronises).
 */
#define FD_DEVICE_STATUS_WAIT_TIMEOUT 1u
int fd_device_status(fd_stream_t stream, unsigned *status, int clear);

/*
 * fd_w4_dequant_debug - write the dequantised weights W[n, k] = q[n, k] * s[n, k/group]
 * as fp32 [N, K] (test support: the unpack and scale of the GEMV prologue, checked bit
 * for bit). Same layouts and size rules as fd_swiglu_w4a16_gemv (N == 0 is empty);
 * `out` is fp32 [N, K].
 */
int fd_w4_dequant_debug(const void *qweight, const void *scales, float *out, int K, int N,
                        int group, fd_stream_t stream);

/*
 * fd_nvfp4_scaled_mm - NVFP4 scaled matmul with the fp32 output multiplier folded into the
 * GEMM ([NVFP4] "PyTorch folds NVFP4 output scaling into NVGEMM candidates for decode
 * workloads", body and metrics table: packed FP4 operands with E4M3 1x16 block scales and
 * a zero-dimensional fp32 multiplier applied inside the GEMM instead of by a separate
 * multiplication kernel):
 *
 *   X[m, k]   = e2m1(x[m, k]) * e4m3(x_sf[m, k / 16])
 *   W[n, k]   = e2m1(w[n, k]) * e4m3(w_sf[n, k / 16])
 *   out[m, n] = bf16( alpha * sum_k X[m, k] * W[n, k] )   (fp32 accumulation, one rounding)
 *
 * x       packed FP4 [M, K/2] bytes: element 2p in the low nibble (bits 0..3) of byte p,
 *         element 2p + 1 in the high nibble. E2M1 codes: sign bit 3, exponent bits 2..1
 *         (bias 1; field 0 is subnormal, m/2), mantissa bit 0: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
 * x_sf    E4M3 scale codes [M, K/16] bytes, row-major: one per 16 consecutive k of a row
 *         (bias 7, no infinity, S.1111.111 is NaN).
 * w, w_sf the weights [N, K/2] (nn.Linear [out, in] orientation) and their scales [N, K/16].
 * alpha   pointer to ONE fp32 in device memory (the 0-dim multiplier), read by the kernel
 *         after its dependency wait, so a previous kernel in the stream may write it.
 * out     bf16 [M, N] row-major; must not overlap any input (FD_ERR_OVERLAP).
 * Requires 0 <= M <= FD_MAX_M, N >= 0, K a multiple of 256 (FD_ERR_SHAPE otherwise) and
 *         K <= FD_NVFP4_MAX_K (FD_ERR_UNSUPPORTED otherwise). M == 0 or N == 0 is an empty
 *         call: FD_OK at once, no pointer read, nothing launched.
 *         x, x_sf, w, w_sf and out 16-byte aligned, alpha 4-byte aligned (FD_ERR_ALIGN).
 * Runs on the tensor cores' block-scaled MMA (tcgen05, kind::mxf4nvf4): each E2M1 x E2M1
 * product with both scales is exact; sums accumulate in fp32 in tensor memory, alpha
 * multiplies the fp32 sum and the result is rounded once. K is split over a thread-block
 * cluster of up to 8 CTAs whose partial sums meet in distributed shared memory: no global
 * scratch.
 */
#define FD_NVFP4_MAX_K 16384
int fd_nvfp4_scaled_mm(const void *x, const void *x_sf, const void *w, const void *w_sf,
                       const float *alpha, void *out, int M, int K, int N, fd_stream_t stream);

/*
 * fd_debug_plan_nvfp4 - test support: the launch plan of fd_nvfp4_scaled_mm for one launch
 * of M (1..128) activation rows, computed on the host without any CUDA call.
 * smem_budget  dynamic shared memory a CTA may use (bytes).
 * plan    int[13] out: split (CTAs per cluster along K), 256-k stages of K, stages of the
 *         largest slice, padded batch, 128-row weight tiles, TMEM columns, output columns
 *         (activation rows) per rank, scale bytes copied per row, shared-memory offsets of the activations, the
 *         weight scales and the activation scales (weights at 0), the reduction buffer's
 *         bytes (from offset 0), dynamic shared memory per CTA.
 * Returns FD_ERR_UNSUPPORTED when the kernel has no plan for the shape.
 */
int fd_debug_plan_nvfp4(int M, int K, int N, int smem_budget, int *plan);

/* Static, NUL-terminated description of a status code (never NULL). */
const char *fd_status_string(int status);

/*
 * fd_copy - copy `bytes` from src to dst with one kernel spread over every SM, for the
 * per-token inputs and outputs of a decode step. Either side may be device memory or
 * pinned host memory (cudaHostAlloc / torch pin_memory), which a GB300 reads and writes
 * over NVLink-C2C. When a side is not accessible to a kernel (pageable host memory) the
 * call falls back to one cudaMemcpyAsync.
 * Requires  dst, src 16-byte aligned; bytes a multiple of 16; no overlap. bytes == 0
 *           returns FD_OK at once (no pointer read, nothing launched).
 * Stream-ordered like every call here; with programmatic dependent launch the kernel
 * waits for the previous kernel before it reads src.
 */
int fd_copy(void *dst, const void *src, size_t bytes, fd_stream_t stream);

/*
 * fd_copy_rows - the same for `rows` rows of `row_bytes` each, read at a pitch of
 * src_pitch bytes and written at a pitch of dst_pitch bytes (a decode step's per-layer
 * gate and up rows, which the step keeps interleaved). When a side is not accessible to a
 * kernel the call falls back to one cudaMemcpy2DAsync.
 * Requires  dst, src 16-byte aligned; row_bytes, dst_pitch, src_pitch multiples of 16 with
 *           both pitches >= row_bytes; the two spans ((rows - 1) x pitch + row_bytes bytes
 *           from each pointer) do not overlap. row_bytes == 0 or rows == 0 returns FD_OK at
 *           once (no pointer read, nothing launched).
 * Returns FD_OK; FD_ERR_NULL, FD_ERR_SHAPE, FD_ERR_ALIGN, FD_ERR_OVERLAP for bad arguments
 * (nothing launched); FD_ERR_CUDA if the launch fails.
 */
int fd_copy_rows(void *dst, size_t dst_pitch, const void *src, size_t src_pitch,
                 size_t row_bytes, size_t rows, fd_stream_t stream);

/*
 * fd_debug_plan_gemv - test support: the launch plan the bulk-copy GEMV kernel would use,
 * computed on the host from given device facts, without any CUDA call.
 * device  int[6]: SM count, opt-in shared memory per CTA, shared memory per SM, shared
 *         memory reserved per CTA, the kernel's static shared memory, its registers per
 *         thread.
 * plain   0: the SwiGLU activation (gate and up); 1: a plain activation (gate/up GEMV).
 * plan    int[9] out: grid, rows_base, rows_extra (the first rows_extra CTAs own one more
 *         row), stages S, weight rows of shared memory, first stage the M = 1 activation
 *         copy overlays, ring (stages reused), CTAs per SM, dynamic shared memory per CTA.
 * Returns FD_ERR_UNSUPPORTED when the kernel would not run the call (the CUDA-core kernel
 * does instead).
 */
int fd_debug_plan_gemv(const int *device, int M, int K, int N, int group, int plain, int *plan);

/*
 * fd_debug_plan_step - test support: the launch plan fd_decode_mlp_step would use, computed
 * on the host from given device facts, without any CUDA call.
 * device  int[6], as for fd_debug_plan_gemv (the persistent kernel's static shared memory in
 *         device[4]; the budget is device[1] - device[4]).
 * plan    int[8] out: grid, rows_base, rows_extra (the first rows_extra CTAs own one more
 *         row), chunks of the largest CTA's rows, weight rows of shared memory, dynamic shared
 *         memory per CTA, and the add-RMSNorm row's 16-byte vectors per thread and threads.
 * Returns FD_ERR_SHAPE for a non-positive size or hidden not a multiple of 8;
 * FD_ERR_UNSUPPORTED when the step has no kernel or no plan for the shape.
 */
int fd_debug_plan_step(const int *device, int hidden, int inter, int group, int *plan);

/*
 * fd_debug_plan_tc - test support: the shared-memory plan of the tensor-core GEMV
 * (fd_swiglu_w4a16_gemv at M >= 16) for its first launch (up to 128 activation rows),
 * computed on the host without any CUDA call.
 * smem_budget  dynamic shared memory a CTA may use (bytes).
 * plan    int[10] out: the padded rows (the MMA's N), k per pipeline step, weight tiles,
 *         gate/up stages, operand stages, scale columns per row, shared-memory offsets of the
 *         gate/up ring, the operand ring and the scales (weights at 0), dynamic shared
 *         memory per CTA.
 * Returns FD_ERR_SHAPE for a non-positive size; FD_ERR_UNSUPPORTED when the tensor-core
 * kernel does not run the shape or has no plan within the budget.
 */
int fd_debug_plan_tc(int M, int K, int N, int group, int smem_budget, int *plan);

/* The cudaError_t value behind the calling thread's most recent FD_ERR_CUDA (0 if none).
 * Thread-local; not reset by successful calls. */
int fd_last_cuda_error(void);

/* Library ABI version: major * 10000 + minor * 100 + patch. */
int fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_H_ */
