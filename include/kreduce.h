/*
 * kreduce.h -- C ABI of the symbolic kernel-reduction library for one sm_103a GPU.
 *
 * The library reduces an M x N matrix whose entries are a formula of two point
 * clouds, x_i in R^D (i < M) and y_j in R^D (j < N), without ever storing the
 * matrix: the entries are evaluated in registers, tile by tile, and reduced over j.
 *
 *   Sum       a_ie = sum_j exp(-|x_i - y_j|^2 / sigma^2) b_je
 *   LogSumExp L_ie = log sum_j exp(-|x_i - y_j|^2 / sigma^2 + w_je)
 *   grad-x    gx_id = d/dx_id sum_{i,e} g_ie a_ie
 *                   = -(2/sigma^2) sum_j k_ij (sum_e g_ie b_je)(x_id - y_jd)
 *   grad-y    gy_jd = d/dy_jd sum_{i,e} g_ie a_ie
 *                   = (2/sigma^2) sum_i k_ij (sum_e g_ie b_je)(x_id - y_jd)
 *   grad-b    gb_je = d/db_je sum_{i,e} g_ie a_ie = sum_i k_ij g_ie
 *   K-min     the K pairs (|x_i - y_j|^2, j) that are smallest in lexicographic
 *             order, sorted ascending; K = 1 is ArgMin.
 *
 * Sources: "Kernel Operations on the GPU, with Autodiff, without Memory Overflows",
 * §1 Introduction (target operation: a_i = sum_j k(x_i, y_j) b_j with a Gaussian
 * k of width sigma) and §2 (generic reductions: sum, logsumexp, argmin, argKmin;
 * autodiff); KeOps README, PyTorch usage example (squared distances, exp(-D),
 * .sum / .logsumexp / .argmin, gradient of sum_i a_i^2 wrt x) and feature list
 * (Sum, LogSumExp, ArgMin, K-min); GitHub issue "Transparent interface for
 * billion-scale matrices" (caller-allocated output, calls that do not hold the
 * caller's interpreter lock).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.   All arrays are float32 (int32 for indices), row-major, contiguous:
 *           x: M x D, y: N x D, b and w: N x E, g: M x E, out: M x E,
 *           gx: M x D, gy: N x D, gb: N x E, idx and dist: M x K.  Each
 *           pointer may address device memory or host memory (pageable or
 *           pinned); host arrays are staged
 *           through device memory allocated for the call, and the call then
 *           blocks until its host outputs are written.  With device pointers
 *           only, the call is asynchronous on `stream`.
 * Ownership. The caller owns every array, outputs included; the library never
 *           frees or keeps caller memory.  Workspace (split-j partials, staging)
 *           is taken stream-ordered on `stream` from a memory pool the library
 *           creates on each device (cudaMemPoolCreate; cudaMallocFromPoolAsync /
 *           cudaFreeAsync) and released in stream order after the work it serves.
 *           The pool keeps up to 256 MiB of freed workspace across
 *           synchronisations for the next call and returns the rest.
 * Aliasing. Outputs must not overlap inputs or each other.
 * Stream.   `stream` is a cudaStream_t (NULL = the legacy default stream).  The
 *           device is the current device of the calling thread.
 * Errors.   Arguments are validated before any CUDA call; an invalid call
 *           returns a status and launches nothing.  The return value reports
 *           validation, allocation and launch errors; with device pointers,
 *           errors during execution surface at the caller's next synchronisation.
 * Threads.  Calls from several host threads on different streams are safe; the
 *           library's only global state is per-device cached attributes.
 * Limits.   1 <= D <= 128, 1 <= E <= 16, 1 <= K <= 32; M >= 0; 0 <= N < 2^31 - 1
 *           (indices are int32); M*D, N*D, M*E, N*E and M*K at most 2^60 elements
 *           (every element index is 64-bit: y may exceed 2^31 floats, e.g.
 *           N = 10^9 points in D = 50).  sigma finite and > 0.
 *           M = 0 is a no-op; N = 0 gives Sum 0, LogSumExp -inf, grad 0,
 *           K-min indices -1 and distances +inf.
 * Numerics. fp32 inputs and outputs; exp is computed as ex2.approx on arguments
 *           prescaled by sqrt(log2 e)/sigma; sums over j use per-tile partials
 *           with a compensated running sum; split-j partials are combined in a
 *           fixed order, so results are deterministic run to run.
 */
#ifndef KREDUCE_H
#define KREDUCE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so this header needs no CUDA header. */
typedef struct CUstream_st *kr_stream_t;

typedef enum {
    KR_SUM = 0, /* a_ie = sum_j k_ij b_je */
    KR_LSE = 1, /* L_ie = log sum_j exp(-|x_i - y_j|^2/sigma^2 + w_je); b holds w */
    KR_MAX = 2, /* m_ie = max_j k_ij b_je (ArgMax: the lowest j attaining it) */
    KR_MIN = 3  /* m_ie = min_j k_ij b_je (ArgMin: the lowest j attaining it) */
} kr_reduction;

/* Radial kernel k_ij = k(|x_i - y_j|) of width sigma, chosen with kr_options.kernel. */
typedef enum {
    KR_KERNEL_GAUSSIAN = 0,             /* exp(-|x - y|^2 / sigma^2) */
    KR_KERNEL_LAPLACE = 1,              /* exp(-|x - y| / sigma) */
    KR_KERNEL_CAUCHY = 2,               /* 1 / (1 + |x - y|^2 / sigma^2) */
    KR_KERNEL_INVERSE_MULTIQUADRIC = 3  /* 1 / sqrt(1 + |x - y|^2 / sigma^2) */
} kr_kernel;

typedef enum {
    KR_OK = 0,
    KR_ERR_INVALID = 1,     /* null pointer with a nonzero size, negative size, bad sigma,
                               unknown reduction, overlapping outputs */
    KR_ERR_UNSUPPORTED = 2, /* valid request outside the limits above */
    KR_ERR_ALLOC = 3,       /* workspace or staging allocation failed; outputs untouched */
    KR_ERR_CUDA = 4         /* a CUDA runtime call failed; see kr_last_cuda_error() */
} kr_status;

/* Optional knobs; pass NULL for the defaults (a zeroed struct is the defaults). */
typedef struct {
    int split;       /* S >= 1 forces S disjoint j-ranges (split-j); 0 = automatic */
    int path;        /* KR_PATH_*: which units evaluate the Sum (0 = automatic) */
    int kernel;      /* KR_KERNEL_*: the radial kernel (0 = Gaussian).  Other kernels serve
                        the Sum, Max and Min (and the b-gradient); the LogSumExp, the x- and
                        y-gradients and the K-min give KR_ERR_UNSUPPORTED for them. */
    int batch;       /* B >= 2: B independent problems of the given sizes in one call (batch
                        dimension; "Kernel Operations on the GPU...", §2: LazyTensors support
                        batch dimensions).  Every array then holds its B problems one after
                        the other (x: B x M x D, ..., out: B x M x E), each row-major; the
                        sizes M, N, D, E, K are per problem.  0 or 1: one problem.  At most
                        65535; batched Sums run on the CUDA cores. */
    int reserved[4]; /* must be zero */
} kr_options;

typedef enum {
    KR_PATH_AUTO = 0,         /* tensor cores where eligible, else CUDA cores */
    KR_PATH_CUDA_CORES = 1,   /* FP32 pipe: direct differences, every shape */
    KR_PATH_TENSOR_CORES = 2  /* tcgen05 split-fp16 expansion: Gaussian Sum (E = 1,
                                 32 <= D <= 62) and LogSumExp (E = 1, 32 <= D <= 61), no
                                 batch; ignored elsewhere.  At run
                                 time it stands down to the CUDA cores when max |x'|^2 +
                                 max |y'|^2 exceeds 16 (x' = x sqrt(log2 e)/sigma), where the
                                 expansion's rounding would exceed the tolerance.  The
                                 K-min (32 <= D <= 62, K <= 32, no batch) screens its pairs
                                 with one fp16 product of the expansion's high halves and
                                 stands down when max |x|^2 + max |y|^2 exceeds 4096. */
} kr_path;

/*
 * Sum, LogSumExp, Max or Min over j ("Kernel Operations on the GPU...", §1 target
 * operation, §2 generic reductions; KeOps README .sum(dim=1), .logsumexp() and the
 * Min / Max reductions of its feature list).
 *   x [M x D], y [N x D]: point clouds.
 *   b [N x E]: the signal b_je for KR_SUM, KR_MAX, KR_MIN; the additive log-weight
 *              w_je for KR_LSE (pass log b for positive weights; -inf is allowed and
 *              means weight 0).
 *   out [M x E]: written with a (KR_SUM), L (KR_LSE) or the extreme value of
 *              k_ij b_je over j (KR_MAX, KR_MIN; -inf / +inf when N = 0).
 *   sigma: kernel width; the kernel is the Gaussian exp(-|x - y|^2 / sigma^2)
 *          unless kr_options.kernel picks another (Sum, Max, Min only).
 * Returns a kr_status.
 */
int kernel_reduce(const float *x, const float *y, const float *b, float *out,
                  int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                  kr_stream_t stream);
int kernel_reduce_ex(const float *x, const float *y, const float *b, float *out,
                     int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                     kr_stream_t stream, const kr_options *opt);

/*
 * Max or Min of k_ij b_je over j together with its Arg ("Kernel Operations on the
 * GPU...", §2: max, min and argmin reductions; KeOps README feature list: Min, Max,
 * ArgMin, ArgMax).
 *   reduction: KR_MAX or KR_MIN.
 *   idx [M x E] (int32): the lowest j attaining the extreme value (-1 when N = 0).
 *   out [M x E] (nullable): the extreme value, as kernel_reduce writes it.
 * The values k_ij b_je are computed in fp32 (the kernel with ex2 / rcp / rsqrt /
 * sqrt approximations), and the comparison that picks the index is taken on those
 * values, so where two candidates agree to within fp32 rounding either index may
 * be returned.
 */
int kernel_reduce_arg(const float *x, const float *y, const float *b, float *out, int32_t *idx,
                      int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                      kr_stream_t stream);
int kernel_reduce_arg_ex(const float *x, const float *y, const float *b, float *out, int32_t *idx,
                         int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                         kr_stream_t stream, const kr_options *opt);

/*
 * Block-sparse (cluster-wise truncated) Sum, Max or Min ("Kernel Operations on the
 * GPU...", §3 "Applications": cluster-wise block-sparsity for large kernel systems;
 * §4: the block-sparse truncation rule; KeOps README: an interface for block-sparse
 * strategies).  The rows of x are grouped in clusters; cluster c owns rows
 * ranges_i[2c] <= i < ranges_i[2c+1] and reduces only over the column ranges
 * redranges_j[2r] <= j < redranges_j[2r+1] for slices_i[c-1] <= r < slices_i[c]
 * (slices_i[-1] = 0).  A point in two ranges of one cluster counts twice in the Sum.
 * Rows in no cluster reduce over nothing (Sum 0, Max -inf, Min +inf, index -1).
 *   reduction: KR_SUM (out required, idx must be NULL), KR_MAX or KR_MIN (out and/or
 *              idx; idx = the lowest j attaining the extreme, whatever the order of
 *              the ranges).
 *   ranges_i [nclusters x 2], slices_i [nclusters], redranges_j [nranges x 2]: int64
 *              HOST arrays, read during the call (the library copies the tables it
 *              builds from them); clusters must not overlap, slices must not
 *              decrease and end at most at nranges, ranges must lie in [0, N).
 *              Anything else gives KR_ERR_INVALID.
 *   opt: kernel kind as for kernel_reduce; split and batch are not available in this
 *        mode (KR_ERR_UNSUPPORTED).  Other arrays as for kernel_reduce_arg.
 * One thread block serves at most 128 R consecutive rows of one cluster (R the rows
 * per thread of the instance) and walks all of that cluster's ranges.
 */
int kernel_reduce_ranges(const float *x, const float *y, const float *b, float *out, int32_t *idx,
                         int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                         int64_t nclusters, const int64_t *ranges_i, const int64_t *slices_i,
                         int64_t nranges, const int64_t *redranges_j, kr_stream_t stream,
                         const kr_options *opt);

/*
 * kernel_reduce without any device allocation.  The pages have no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory when
 * they call -- a process whose own memory arena already holds (almost) all of the
 * GPU, so cudaMalloc / cudaMallocAsync would fail, or a latency-critical loop that
 * must not wait on the driver's allocator.  Same arguments and result as
 * kernel_reduce, always in split-j mode, with the split partials kept in a 16 MiB
 * static device array that every GPU loading this library reserves until exit.
 *   - All four arrays must be device (or managed) memory; host arrays, which would
 *     need staging memory, give KR_ERR_INVALID.
 *   - Limit: M * E <= 1048576 (two splits of partials must fit the 16 MiB array);
 *     larger requests give KR_ERR_UNSUPPORTED.  Use kernel_reduce for them.
 *   - The first call on a device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream
 *     capture.  A failed lookup gives KR_ERR_CUDA (kr_last_cuda_error is not set
 *     by this entry point).
 *   - Every call on a device shares the one array, which keeps the last call's
 *     contents; each call overwrites every partial it reads, so nothing needs
 *     clearing, but calls whose work overlaps on the GPU (different streams, or
 *     threads without ordering between them) race on it and must be serialised.
 */
int kernel_reduce_noalloc(const float *x, const float *y, const float *b, float *out,
                          int64_t M, int64_t N, int D, int E, float sigma, int reduction,
                          kr_stream_t stream);

/*
 * Gradient wrt x of sum_{i,e} g_ie a_ie, a the Sum reduction (KeOps README usage
 * example: torch.autograd.grad((a_i ** 2).sum(), [x]), i.e. g = 2a).
 *   x [M x D], y [N x D], b [N x E], g [M x E] (upstream gradient), gx [M x D] output.
 */
int kernel_reduce_grad_x(const float *x, const float *y, const float *b, const float *g,
                         float *gx, int64_t M, int64_t N, int D, int E, float sigma,
                         kr_stream_t stream);
int kernel_reduce_grad_x_ex(const float *x, const float *y, const float *b, const float *g,
                            float *gx, int64_t M, int64_t N, int D, int E, float sigma,
                            kr_stream_t stream, const kr_options *opt);

/*
 * Gradient wrt y of sum_{i,e} g_ie a_ie ("Kernel Operations on the GPU...", §2
 * "Performance and differentiation": gradients wrt every input through autodiff):
 *   gy_jd = (2/sigma^2) sum_i k_ij (sum_e g_ie b_je) (x_id - y_jd).
 *   x [M x D], y [N x D], b [N x E], g [M x E] (upstream gradient), gy [N x D] output.
 * Computed by the x-gradient kernels with the two clouds exchanged, so it plans,
 * splits and performs exactly like kernel_reduce_grad_x on (y, x).
 */
int kernel_reduce_grad_y(const float *x, const float *y, const float *b, const float *g,
                         float *gy, int64_t M, int64_t N, int D, int E, float sigma,
                         kr_stream_t stream);
int kernel_reduce_grad_y_ex(const float *x, const float *y, const float *b, const float *g,
                            float *gy, int64_t M, int64_t N, int D, int E, float sigma,
                            kr_stream_t stream, const kr_options *opt);

/*
 * Gradient wrt b of sum_{i,e} g_ie a_ie, the transposed product
 *   gb_je = sum_i k_ij g_ie
 * (same section; a is linear in b).  x [M x D], y [N x D], g [M x E], gb [N x E]
 * output.  Computed as kernel_reduce(y, x, g) (every kernel here is symmetric), so
 * it takes the tensor-core path under the same conditions as that call, and
 * kr_options.kernel picks the kernel as for the Sum.
 */
int kernel_reduce_grad_b(const float *x, const float *y, const float *g, float *gb,
                         int64_t M, int64_t N, int D, int E, float sigma, kr_stream_t stream);
int kernel_reduce_grad_b_ex(const float *x, const float *y, const float *g, float *gb,
                            int64_t M, int64_t N, int D, int E, float sigma, kr_stream_t stream,
                            const kr_options *opt);

/*
 * K-min / ArgMin over squared Euclidean distance (KeOps README feature list:
 * ArgMin and K-min reductions; "Kernel Operations on the GPU...", §2 argKmin).
 *   idx [M x K] (int32): the K indices j with the smallest (|x_i - y_j|^2, j),
 *                        ascending; ties keep the lowest j; -1 past N.
 *   dist [M x K] (nullable): the matching fp32 squared distances, +inf past N.
 * The reported distance is always the direct fp32 sum over d of (x_id - y_jd)^2.  On the
 * tensor-core path (kr_path above) the expansion |x|^2 + |y|^2 - 2 x.y only screens: a
 * point whose screened distance is above the row's current K-th plus a bound on the
 * expansion's rounding cannot enter the list and is skipped; every other point gets
 * the direct distance, so the result is the CUDA-core path's up to the order of ties
 * within fp32 rounding of the distance.
 */
int kernel_knn(const float *x, const float *y, int32_t *idx, float *dist,
               int64_t M, int64_t N, int D, int K, kr_stream_t stream);
int kernel_knn_ex(const float *x, const float *y, int32_t *idx, float *dist,
                  int64_t M, int64_t N, int D, int K, kr_stream_t stream,
                  const kr_options *opt);

/* Static text for a kr_status value. */
const char *kr_status_string(int status);

/* The cudaError_t of the last KR_ERR_CUDA returned on the calling thread (0 if none). */
int kr_last_cuda_error(void);

/*
 * Sticky device status of the calling thread's current device (failure detection; no
 * counterpart on the pages).  Every wait of the tensor-core kernels on
 * their mbarriers is bounded (2 s of global time by default); a block whose wait gives
 * up writes NaN for its rows and sets bit 0 of this status.  Reads the status into
 * *status (0 = nothing happened since the last clear) and clears it when `clear` is
 * nonzero.  Synchronous: waits for the device's work.  The environment variable
 * KREDUCE_TC_WAIT_MS (read once per process) sets another wait bound in ms.
 */
int kr_device_status(unsigned *status, int clear);

/*
 * Test hook of the failure detection above (no counterpart on the pages).  Sets the
 * tensor-core wait bound to wait_ms (0: back to 2000) for the whole process, and with
 * starve = 1 makes the tensor-core kernels withhold their B tiles, so that every wait
 * runs out (rows NaN, status bit 0; the context stays usable and the next call with
 * starve = 0 works normally).  Starvation exists only in the debug build
 * (kr_debug_build() == 1): the release library returns KR_ERR_UNSUPPORTED for
 * starve = 1 and carries no such path.  KR_ERR_INVALID for wait_ms < 0 or starve not
 * 0 or 1.  Not thread-safe against calls in flight on other threads.
 */
int kr_set_tc_test_hooks(int wait_ms, int starve);

/*
 * 1 for a debug build of the library (compiled with -DKR_DEBUG, libkreduce_debug.so),
 * else 0.  In a debug build every global-memory access of the CUDA-core kernels checks
 * its element index against the array's extent; a violation skips the access and sets a
 * bit (x 1, y 2, b 4, g 8, out 16, idx 32, split partials 64, shared memory 128) that
 * kr_device_status reports shifted left by 8.  (Test infrastructure for index arithmetic;
 * no counterpart on the pages.)
 */
int kr_debug_build(void);

/*
 * Launch plan, exposed so that the host logic can be inspected without a GPU.
 * op: 0 = Sum, 1 = LogSumExp, 2 = grad-x, 3 = K-min, 4 = Max / Min; EK = E (ops 0-2, 4)
 * or K (op 3).  opt->kernel selects the radial kernel of ops 0 and 4.
 * num_sms and blocks_per_sm describe the device (blocks_per_sm <= 0: use the
 * plan's own estimate).  Fills *plan and returns a kr_status; no CUDA call.
 */
typedef struct {
    int d_pad;         /* compile-time coordinate count of the kernel instance (>= D) */
    int ek_pad;        /* compile-time E (or K) of the instance (>= E or K) */
    int rows_per_thread; /* CUDA-core kernels; the tensor-core kernel has 128 rows per block */
    int threads;       /* per block */
    int tile_points;   /* points of y per shared-memory tile */
    int64_t row_blocks;
    int split;         /* S */
    int64_t chunk;     /* columns per split; the last split may be shorter */
    int64_t workspace_bytes;
    int path;          /* KR_PATH_CUDA_CORES or KR_PATH_TENSOR_CORES */
} kr_plan_t;

int kr_plan(int op, int64_t M, int64_t N, int D, int EK, int num_sms, int blocks_per_sm,
            const kr_options *opt, kr_plan_t *plan);

/*
 * The plan a call with these arguments makes on the calling thread's current device:
 * kr_plan with that device's SM count and the kernel instance's resident blocks per
 * SM.  Queries device attributes; launches nothing and allocates nothing.  Useful to
 * size workspace in advance and to count launches (1 + (split > 1) per call).
 */
int kr_plan_device(int op, int64_t M, int64_t N, int D, int EK, const kr_options *opt,
                   kr_plan_t *plan);

#ifdef __cplusplus
}
#endif

#endif /* KREDUCE_H */
