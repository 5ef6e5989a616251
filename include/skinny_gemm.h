/*
 * skinny_gemm.h -- C ABI of the GB300 (sm_103a) low-latency skinny BF16 GEMM.
 *
 *     Y[m][n] = sum_k  X[m][k] * W[n][k]      0 <= m < M <= 64,  0 <= n < N
 *
 * X is [M, K] bf16, W is [N, K] bf16 (a weight, e.g. the MoE router's
 * [experts, hidden] matrix or a decode projection's [out, in] matrix), both
 * row-major with row strides ldx / ldw in elements; Y is [M, N] fp32, row
 * stride ldy >= N (strided output, the gaps n >= N are never written).
 * Accumulation is fp32.  The CUDA-core kernels round every multiply-add to
 * nearest (fused multiply-add).  The tensor-core kernels sum short chains
 * inside the tensor core, whose fp32 accumulation is not rounded to nearest
 * per add (measured biased on same-sign data), so those chains are bounded
 * (at most 4 k16 steps per mma.sync register sum, at most 16 MMAs of K = 16
 * per tcgen05 tensor-memory accumulator) and the chain sums are added with
 * round-to-nearest fp32 adds.  Every kernel keeps |y - y_exact| within
 * 1e-5 * sum_k |x * w| + 1e-6, same-sign operands at K = 14336 included.
 * The output is fp32.
 *
 * Operation defined by: "[Perf][Feat] Add generic cuteDSL LL BF16 router
 * (GEMM)" (vllm PR #42562 report), section "Implementation breakdown"
 * items 1-4 (dot-product kernel for small M, cluster split-K kernel for larger
 * M, a (M, K, N) dispatcher, the M <= 16 bf16-only router tier) and the
 * review notes on alignment and dtype guards; and "GLM-5.2 Blackwell decode
 * optimizations" (vllm PR #48597), section "Implementation breakdown" item 3
 * (bf16_skinny_gemm for the decode projections, strided output) and item 2
 * (programmatic dependent launch).
 *
 * Token range.  M = 1..16 is the router tier of the first page; every
 * backend takes it.  M = 17..64 is the medium-M regime that the second page
 * (item 3) hands to a separate GEMM before falling back to cuBLAS; here it
 * runs on the tensor cores only: the tcgen05 backend (16-byte aligned X and
 * W rows, i.e. pointers, ldx and ldw multiples of 8 elements; any K), the
 * tensor-core dot-product (weights of 16 MB or more, K % 32 == 0, X staged in
 * chunks), or the cluster split-K backend with the mma.sync consumer
 * (K % 16 == 0, 16-byte aligned W rows, and a per-CTA X slice of M x K /
 * split_k x 2 bytes, split_k <= 8, of at most 160 KB beside the W ring).
 * M > 16 calls that none of them can take return SKINNY_ERR_UNSUPPORTED.
 *
 * bf16 values are passed as their 16-bit patterns (uint16_t) so this header
 * needs no CUDA header.  Streams are passed as `void*` holding a cudaStream_t
 * (NULL = the legacy default stream).
 *
 * Ownership: the caller owns X, W and Y (device memory, e.g. allocated by
 * PyTorch).  The library allocates nothing per call, never synchronises in
 * skinny_gemm_bf16, and keeps only small per-device state created by
 * skinny_init (or by the first call on a device).
 *
 * Thread safety: calls may be made concurrently from several host threads.
 * Options (skinny_set_option) are process-wide.
 */
#ifndef SKINNY_GEMM_H_
#define SKINNY_GEMM_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKINNY_MAX_M 64

/* Exported from libskinny_gemm.so (built with hidden default visibility). */
#if defined(__GNUC__)
#define SKINNY_API __attribute__((visibility("default")))
#else
#define SKINNY_API
#endif

typedef enum {
    SKINNY_OK = 0,
    SKINNY_ERR_INVALID_VALUE = 1,   /* negative size, ld too small, NULL with work to do, Y overlaps X or W */
    SKINNY_ERR_UNSUPPORTED = 2,     /* M > 64; M > 16 on a shape no tensor-core backend can
                                       take (see "Token range"); or a forced plan that cannot
                                       run this shape */
    SKINNY_ERR_MISALIGNED = 3,      /* X or W not 2-byte aligned, Y not 4-byte aligned */
    SKINNY_ERR_LAUNCH = 4,          /* the CUDA launch failed (cudaGetLastError after the launch) */
    SKINNY_ERR_DEVICE_TIMEOUT = 5,  /* a bounded wait inside a kernel gave up (see skinny_get_device_status) */
    SKINNY_ERR_NO_DEVICE = 6        /* no usable CUDA device / the device is not sm_103 */
} skinny_status_t;

typedef enum {
    SKINNY_BACKEND_AUTO = 0,
    SKINNY_BACKEND_DOTPROD = 1,     /* one CTA per block of output columns, whole K */
    SKINNY_BACKEND_SPLITK = 2,      /* K split over the CTAs of a thread-block cluster */
    SKINNY_BACKEND_STREAM = 3,      /* one CTA per SM, whole K per 16-row tile, K-outer: X and W
                                       stream through one ring chunk by chunk (large weights;
                                       needs 16-byte aligned X and W rows, K % 16 == 0, M <= 16) */
    SKINNY_BACKEND_TCGEN05 = 4      /* the fifth-generation tensor cores (tcgen05.mma into tensor
                                       memory, drained into fp32 registers every <= 16 MMAs): W rows
                                       in grid_y balanced ranges of 8-row groups, tiles of up to
                                       block_n = 64 / 128 rows, K split over a cluster of split_k
                                       CTAs (1, 2, 4 or 8), W and X boxes by tensor-map TMA; needs
                                       16-byte aligned X and W rows (pointers, ldx and ldw);
                                       any K >= 1, M <= 64 */
} skinny_backend_t;

typedef enum {
    SKINNY_CONSUMER_AUTO = 0,
    SKINNY_CONSUMER_FMA = 1,        /* CUDA-core fp32 fused multiply-add */
    SKINNY_CONSUMER_MMA = 2         /* mma.sync m16n8k16 bf16 -> fp32, W on the MMA's M side
                                       (split-K, or the dot-product layout with block_n 16/32/64);
                                       fp32 weights: mma.sync m16n8k8 tf32 -> fp32, block_n 16/32 */
} skinny_consumer_t;

/* The launch a call would make.  Filled by skinny_query_plan / skinny_plan_for. */
typedef struct {
    int backend;       /* skinny_backend_t actually used */
    int consumer;      /* skinny_consumer_t actually used (FMA or MMA, for either backend) */
    int vec_elems;     /* W load width in elements: bf16 8 (128-bit), 4, 2 or 1; fp32 weights 4, 2 or 1 */
    int block_n;       /* output columns (rows of W) per CTA tile; tcgen05: the MMA's M (64 or 128),
                          the tile holding up to that many rows */
    int split_k;       /* CTAs per cluster along K (1 = no cluster) */
    int stages;        /* shared-memory ring depth (split-K, streaming, tcgen05) */
    int stage_k;       /* K elements of each W row per ring stage (split-K and streaming 64..2048,
                          tcgen05 64..256; multiple of 64) */
    int k_chunk;       /* dot-product: K elements of X staged in shared memory at a time (with a
                          cluster split: the rank's slice); split-K, tcgen05: K elements per CTA
                          (the cluster rank's slice) */
    int grid_x;        /* grid dimensions launched; split-K, tcgen05: grid_x = split_k CTAs per cluster, */
    int grid_y;        /* split-K: grid_y clusters, each looping over 16-row tiles y, y + grid_y, ...;
                          tcgen05: grid_y row ranges (clusters), range c holding the 8-row groups
                          [c * G / grid_y, (c + 1) * G / grid_y), G = ceil(N / 8) */
    int threads;       /* threads per CTA (split-K: (consumer warps + 1) x 32; fp32-weight tensor-core
                          plans: 256 up to 8 tokens, 128 above) */
    int smem_bytes;    /* dynamic shared memory per CTA */
    int pdl;           /* 1 if launched with programmatic dependent launch */
    int tuned;         /* 1 if the plan came from the measured tuning table */
} skinny_plan_t;

typedef enum {
    SKINNY_OPT_PDL = 1,              /* programmatic dependent launch: 0 off; 1 on for calls whose plan
                                        stages W through shared memory (split-K, streaming, tcgen05)
                                        and for dot-product calls whose weight is under 16 MB (a larger
                                        dot-product call started beside a shared-memory-heavy kernel
                                        runs with a small L1 and measured slower on GB300); 2 on for
                                        every call (default: env SKINNY_PDL = 1 or 2, else 0) */
    SKINNY_OPT_FORCE_BACKEND = 2,    /* skinny_backend_t; AUTO = dispatcher (tests / tuning only) */
    SKINNY_OPT_FORCE_CONSUMER = 3,   /* skinny_consumer_t for split-K; AUTO = dispatcher */
    SKINNY_OPT_FORCE_SPLIT_K = 4,    /* 0 = dispatcher, 1..8 = cluster size */
    SKINNY_OPT_FORCE_BLOCK_N = 5,    /* 0 = dispatcher; dot-product FMA 1/2/4/8, MMA 16/32/64; split-K 16 */
    SKINNY_OPT_FORCE_STAGES = 6,     /* 0 = dispatcher, 1..16 */
    SKINNY_OPT_WAIT_TIMEOUT_US = 7,  /* budget of each bounded wait in a kernel, microseconds
                                        (default 500000).  0 makes every such wait give up at once,
                                        which exercises the timeout path without any real hang */
    SKINNY_OPT_LOG = 8,              /* 1: print the plan chosen for each new call shape to stderr
                                        (default: env SKINNY_LOG) */
    SKINNY_OPT_FORCE_CLUSTERS = 9,   /* 0 = dispatcher; split-K: the number of (persistent) clusters,
                                        each looping over row tiles; tcgen05: the number of row
                                        ranges (grid_y) (tests / tuning only) */
    SKINNY_OPT_FORCE_STAGE_K = 10,   /* split-K, streaming, tcgen05: 0 = dispatcher, else K elements
                                        per ring stage (multiple of 64; split-K and streaming
                                        64..2048, tcgen05 64..256; tests / tuning only) */
    SKINNY_OPT_FUSE_NORM = 11,       /* 1: skinny_rmsnorm_gemm_bf16 runs the norm inside the tcgen05
                                        GEMM when its plan allows; 0 (default): two launches, measured
                                        faster on GB300 (the fused form's resident X halves its ring) */
    SKINNY_OPT_LATE_TRIGGER = 12     /* 1: a call with 16 MB or more of weight lets a programmatically
                                        dependent launch start only once each of its CTAs has issued
                                        its last W load; 0 (default): at kernel entry, measured faster
                                        on GB300 with mode 1 of SKINNY_OPT_PDL */
} skinny_option_t;

/*
 * Y = X . W^T on `stream` (asynchronous; no host synchronisation, no
 * allocation, so it can be captured in a CUDA graph).
 *
 *   X      device pointer, bf16 [M, K], row stride ldx >= K (elements), 2-byte aligned
 *   W      device pointer, bf16 [N, K], row stride ldw >= K (elements), 2-byte aligned
 *   Y      device pointer, fp32 [M, N], row stride ldy >= N (elements), 4-byte aligned;
 *          must not overlap X or W.  Only Y[m*ldy + n], m < M, n < N, is written.
 *   M      1..64 tokens (0 is a no-op; 17..64 only on the shapes listed under "Token
 *          range" above); N, K >= 0.  K == 0 writes zeros (the empty sum).
 *
 * 16-byte alignment is not required: the dispatcher picks the widest W load
 * that the base pointer and ldw allow (see skinny_plan_t.vec_elems).
 *
 * With PDL on, W is read before the kernel waits for the preceding kernel in
 * the stream (W is a weight); X is read and Y written only after that wait.
 * So W must not be written by the kernel launched just before on the stream.
 *
 * Returns SKINNY_OK once the launch is queued; every argument error is
 * detected on the host before anything is launched.  Errors inside a kernel
 * (a bounded wait that gave up) are recorded in a per-device status word read
 * by skinny_get_device_status.
 */
SKINNY_API skinny_status_t skinny_gemm_bf16(const uint16_t *X, int ldx,
                                 const uint16_t *W, int ldw,
                                 float *Y, int ldy,
                                 int M, int N, int K, void *stream);

/*
 * As skinny_gemm_bf16, but Y is bf16 (uint16_t bit patterns, 2-byte aligned,
 * row stride ldy >= N): each output is the same fp32 result the fp32 entry
 * point computes with the same plan, rounded once to the nearest bf16 (ties to
 * even).  The inputs, plans, checks and errors are those of skinny_gemm_bf16
 * (Y misaligned = not 2-byte aligned; the overlap check uses 2-byte elements).
 *
 * Defined by: "[Perf][Feat] Add generic cuteDSL LL BF16 router (GEMM)",
 * section "Review highlights" (the output type is hard-coded to Float32, noted
 * there as a limitation to lift), and "GLM-5.2 Blackwell decode optimizations",
 * Implementation breakdown item 3 (bf16 decode projections, whose consumers
 * take bf16 activations).
 */
SKINNY_API skinny_status_t skinny_gemm_bf16_bf16out(const uint16_t *X, int ldx,
                                         const uint16_t *W, int ldw,
                                         uint16_t *Y, int ldy,
                                         int M, int N, int K, void *stream);

/* Optional: prepare `device` (query it, check it is sm_103, set kernel
 * attributes, find the status word).  The first call on a device does the
 * same; calling this first keeps that work out of a CUDA-graph capture.
 * Leaves the current device unchanged. */
SKINNY_API skinny_status_t skinny_init(int device);

/* The plan skinny_gemm_bf16 would launch for these arguments on the current
 * device (after the same argument checks).  Host only, no launch. */
SKINNY_API skinny_status_t skinny_query_plan(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                  const float *Y, int ldy, int M, int N, int K,
                                  skinny_plan_t *plan);

/* The dispatcher as a pure function of the arguments and an SM count: no
 * CUDA call at all (usable without a GPU).  Honours the force options. */
SKINNY_API skinny_status_t skinny_plan_for(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                const float *Y, int ldy, int M, int N, int K,
                                int num_sms, skinny_plan_t *plan);

SKINNY_API skinny_status_t skinny_set_option(int option, int value);
SKINNY_API skinny_status_t skinny_get_option(int option, int *value);

/*
 * fp32 router weights: Y = X . W^T with X bf16 [M, K] and W fp32 [N, K]
 * (ldw in fp32 elements), fp32 Y.  For models that keep fp32 router weights
 * ("GLM-5.2 Blackwell decode optimizations", the linked "FP32 router GEMM
 * shape support and tuning" and "Preserve FP32 router weights" changes), and
 * the review note on the first page that fp32 weights must not reach the
 * bf16 kernel: they have their own entry point.  M = 1..16 (else
 * UNSUPPORTED), any K, W 4-byte aligned, W traffic 4NK bytes.  Two kernels:
 *   - the dot-product kernel (CUDA cores): fp32 multiply-add, each fmaf
 *     rounding once; loads of 4, 2 or 1 fp32 as the W pointer and ldw allow;
 *   - from 6 tokens on weights of 4 MB or more, when W rows are 16-byte
 *     aligned (W and ldw) and K % 32 == 0: the tensor-core dot-product.  Each
 *     weight is carried as two tf32 terms (its top bits, then the rest), so
 *     every product is within 2^-20 of x * w; sums in fp32, K over a cluster
 *     of CTAs reduced in a fixed order.
 * Either way |y - y_exact| stays within 1e-5 * sum_k |x w| + 1e-6 and a
 * plan's results are bit-identical from run to run.  Non-finite weights
 * propagate as in IEEE arithmetic.  The force options SKINNY_OPT_FORCE_CONSUMER
 * (FMA / MMA), SKINNY_OPT_FORCE_SPLIT_K and SKINNY_OPT_FORCE_BLOCK_N (16 / 32,
 * MMA only) apply.  Other arguments, errors, PDL and graph capture as
 * skinny_gemm_bf16.
 */
SKINNY_API skinny_status_t skinny_gemm_bf16_f32w(const uint16_t *X, int ldx, const float *W, int ldw,
                                      float *Y, int ldy, int M, int N, int K, void *stream);

/* The launch skinny_gemm_bf16_f32w would make, as a pure function of the
 * arguments and an SM count (no CUDA call).  M == 0, N == 0 or K == 0 give a
 * zeroed plan (nothing or only a zero fill is launched). */
SKINNY_API skinny_status_t skinny_plan_for_f32w(const uint16_t *X, int ldx, const float *W, int ldw,
                                     const float *Y, int ldy, int M, int N, int K, int num_sms,
                                     skinny_plan_t *plan);

/*
 * The q_b projection with its query RMS norm in front: for each token m < M,
 *
 *     r_m     = 1 / sqrt( (1/K) sum_k x(m,k)^2 + eps )          (fp32)
 *     XN(m,k) = bf16_rn( x(m,k) * r_m * gamma(k) )               (written to XN)
 *     Y       = XN . W^T                                          (skinny_gemm_bf16)
 *
 * Operation defined by: "GLM-5.2 Blackwell decode optimizations", section
 * "Implementation breakdown" item 2 (the fused_norm_rope kernel's Q RMS norm
 * branch, q_c = _rms_norm(q_c, q_rms_norm_w, eps, Q_DIM), stored to q_c_out)
 * and item 3 (the q_b bf16_skinny_gemm that consumes it).
 *
 *   X      device, bf16 [M, K] (the query latent q_c), row stride ldx >= K, 2-byte aligned
 *   gamma  device, bf16 [K] (the norm weight); eps >= 0, finite
 *   XN     device, bf16 [M, K] written (q_c_out), row stride ldxn >= K; the GEMM's X, so it
 *          obeys skinny_gemm_bf16's rules for X, and may overlap none of X, gamma, W, Y
 *   W, Y, M (1..64), N, K, stream: as skinny_gemm_bf16 with X = XN.  K == 0 gives Y = 0 and
 *          leaves XN untouched.
 *
 * One launch when the option SKINNY_OPT_FUSE_NORM is on (off by default), the
 * GEMM's plan is tcgen05 without a K split, M <= 16, and X's rows are 16-byte
 * aligned (pointer and ldx): every CTA of the GEMM loads the raw rows of X
 * by TMA into shared memory, computes the r_m of all tokens (the sum of
 * squares in the same fixed order as the norm kernel below, so the same
 * bits), normalises X in place and streams W meanwhile; the CTAs of the first
 * row range also store XN.  Otherwise two launches on `stream`: a norm kernel (one CTA
 * per token; fixed-order fp32 sum of squares, IEEE sqrt and division, one
 * bf16 rounding per element) and then the GEMM, with PDL letting the GEMM
 * stream W while the norm runs.  Either way bit-identical run to run, and the
 * fused and the two-launch forms give the same XN and, under the same plan,
 * the same Y.  Every argument is checked and the plan made before anything is
 * launched.
 */
SKINNY_API skinny_status_t skinny_rmsnorm_gemm_bf16(const uint16_t *X, int ldx, const uint16_t *gamma, float eps,
                                         uint16_t *XN, int ldxn, const uint16_t *W, int ldw, float *Y, int ldy,
                                         int M, int N, int K, void *stream);

/*
 * Router epilogue: for each token m < M, the softmax of its N logits
 * (logits[m*ldl + n], fp32) and its k largest ones.
 *
 *     p_n          = exp(l_n - max_j l_j) / sum_j exp(l_j - max_j l_j)
 *     ids[m*ldid+i]     = index of the i-th largest logit (i < k), descending;
 *                         equal logits: lower index first; a NaN logit ranks
 *                         below every other value (-inf included), NaNs among
 *                         themselves by index, so the k ids are always
 *                         distinct indices in [0, N)
 *     weights[m*ldw+i]  = p of that expert, or with renormalize != 0 that p
 *                         divided by the sum of the k chosen p
 *
 * Operation defined by: "[Perf][Feat] Add generic cuteDSL LL BF16 router
 * (GEMM)", section "Implementation breakdown" item 4 (the MoE gate's forward
 * consumes the router logits); the pages print no epilogue, so this is the
 * plainest softmax / top-k one.  fp32 arithmetic (CUDA expf); the selection
 * compares the fp32 logits exactly as stored; bit-identical run to run.
 *
 *   logits   device, fp32 [M, N], row stride ldl >= N, 4-byte aligned.  The
 *            softmax is IEEE arithmetic: a NaN or +inf logit makes its token's
 *            sum of exponentials NaN, so every weight of that token is NaN
 *            (its ids stay as above)
 *   weights  device, fp32 [M, k], row stride ldw >= k; ids device, int32 [M, k],
 *            row stride ldid >= k; 4-byte aligned; neither may overlap the
 *            logits or each other.  Only the [M, k] entries are written.
 *   M >= 0 (0: no-op), 1 <= N <= 8192, 0 <= k <= min(N, 64) (k = 0: no-op).
 *
 * Asynchronous on `stream`; with PDL on (SKINNY_OPT_PDL) it may start while
 * the preceding kernel (the router GEMM) drains and waits for it before
 * reading the logits.  Errors are found on the host: INVALID_VALUE (sizes,
 * strides, NULL, overlap), UNSUPPORTED (N > 8192, k > 64, M > 65535),
 * MISALIGNED, NO_DEVICE, LAUNCH.
 */
SKINNY_API skinny_status_t skinny_router_topk(const float *logits, int ldl, int M, int N, int k, int renormalize,
                                   float *weights, int ldw, int32_t *ids, int ldid, void *stream);

/*
 * The router in one call: skinny_gemm_bf16(X, W -> logits) then
 * skinny_router_topk(logits -> weights, ids) on the same stream.  `logits` is
 * the caller's [M, N] fp32 buffer (row stride ldl), written by the GEMM and
 * read by the epilogue; nothing is allocated.  Every argument of both steps is
 * checked before anything is launched (weights / ids must not overlap X, W or
 * the logits); the statuses are those of the two calls.
 */
SKINNY_API skinny_status_t skinny_router_bf16_topk(const uint16_t *X, int ldx, const uint16_t *W, int ldw,
                                        float *logits, int ldl, int M, int N, int K, int k, int renormalize,
                                        float *weights, int ldwt, int32_t *ids, int ldid, void *stream);

/* Reads and clears the current device's status word once the work queued on
 * `stream` before the call has finished: a one-thread kernel on `stream`
 * swaps the word with 0 atomically, and the call waits for `stream`.  *code =
 * 0 if no kernel reported an error since the last read, else the first error
 * reported since then: low 8 bits a skinny_status_t (SKINNY_ERR_DEVICE_TIMEOUT),
 * upper bits the wait that gave up (1 = consumer / MMA full-slot wait,
 * 2 = producer empty-slot wait, 3 = drain wait, 4 = X staging wait,
 * 5 = tcgen05 accumulator-full wait, 6 = tcgen05 accumulator-free wait).  The
 * word is shared by every stream of the device: a report made by a kernel on
 * another stream is returned by this read or kept for the next one, never
 * lost.  Test and diagnostic use. */
SKINNY_API skinny_status_t skinny_get_device_status(void *stream, int *code);

/* Static string for a status code (never NULL). */
SKINNY_API const char *skinny_status_string(skinny_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
SKINNY_API int skinny_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SKINNY_GEMM_H_ */
