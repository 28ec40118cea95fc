/*
 * dion.h -- C ABI of libdion.so: the Dion / Orth-Dion optimizer step, batched
 * over many weight matrices, on one NVIDIA B300 (sm_103a).
 *
 * The operation (junaidaliop.github.io "Orth-Dion", update equations and the
 * symbol glossary under them; Dion's column normalisation from the abstract
 * of Orth-Dion, thelatestinai.com 2605.16341), applied independently to every
 * matrix of a plan:
 *
 *     M     = G + R                       m x n   (error-feedback buffer)
 *     U     = orth(M V)                   m x r   (V: warm start, n x r)
 *     W     = M^T U                       n x r
 *     Vbar  = orth(W)        Orth-Dion    n x r
 *           = colnorm(W)     Dion         (each column scaled to unit length)
 *     X    <- X - eta * s * U Vbar^T      (s = scale; sqrt(m/n) when scale <= 0)
 *     R    <- beta * (M - U W^T)          (= beta (M - U U^T M))
 *     V    <- Vbar                        (warm start of the next step)
 *
 * orth() is the Q factor of a thin QR whose triangular factor has a positive
 * diagonal (the pages leave the sign open; this choice makes Q unique).
 *
 * Conventions shared by every entry point:
 *  - All matrices are row-major.  X, R (fp32) and G (fp32 or bf16) are m x n
 *    with leading dimensions ld_x, ld_g, ld_r in ELEMENTS (>= n).  V is a
 *    dense n x r fp32 array (leading dimension r).
 *  - Every data pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates device memory and never frees caller memory.  Pointers
 *    must stay valid while a plan that names them is used.
 *  - X, R, V are updated in place; G is only read.  The writable buffers of
 *    different matrices must not overlap (checked at plan creation).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Entry points that launch work are asynchronous with respect to
 *    the host unless stated otherwise.
 *  - Return values are host-side status codes (dion_status_t).  Numerical
 *    trouble inside a step never traps or hangs: it sets per-matrix bits in
 *    device status words, read with dion_plan_get_status().  A matrix whose
 *    status has any bit other than DION_MAT_SHIFTED set after a step was left
 *    unchanged (X, R, V), except after DION_MAT_TIMEOUT (update incomplete).
 *  - Thread safety: a plan may be used by one host thread at a time.
 *    dion_last_error() is per host thread.
 */
#ifndef DION_H_
#define DION_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DION_ABI_VERSION 1

#if defined(__GNUC__)
#define DION_API __attribute__((visibility("default")))
#else
#define DION_API
#endif

typedef enum {
  DION_OK = 0,
  DION_ERR_INVALID_ARG = 1,   /* bad pointer, size, rank, dtype, overlap ... */
  DION_ERR_CUDA = 2,          /* a CUDA runtime call or launch failed        */
  DION_ERR_WORKSPACE = 3,     /* workspace NULL, too small or misaligned     */
  DION_ERR_UNSUPPORTED = 4    /* valid request this build does not handle    */
} dion_status_t;

/* Per-matrix device status bits (OR-ed together). */
enum {
  DION_MAT_OK = 0,
  DION_MAT_CHOL_BREAKDOWN = 1,  /* orth(): non-positive Cholesky pivot (rank-deficient argument) */
  DION_MAT_NONFINITE = 2,       /* orth(): non-finite value met (NaN / Inf in the inputs)        */
  DION_MAT_TIMEOUT = 4,         /* a pipeline wait inside a tensor-core kernel gave up (after 2 s);
                                   the kernel returned early and this matrix's update is incomplete */
  DION_MAT_SHIFTED = 8          /* informational: an orth() of this matrix was ill conditioned
                                   (kappa > ~1e3) and took shifted CholeskyQR3; the update is complete */
};

/*
 * Right factor and state of a matrix:
 *   DION_VARIANT_DION          Vbar = colnorm(W); R is the error-feedback residual (above)
 *   DION_VARIANT_ORTH          Vbar = orth(W);    R is the error-feedback residual (above)
 *   DION_VARIANT_LOWRANK_MUON  low-rank Muon, this library's reading of the
 *       low-rank orthogonalisation abstract quoted on thelatestinai.com
 *       (2605.16341 listing; the algorithm is not on the pages): R holds Muon's
 *       momentum and V a fresh Gaussian sketch written by the caller before
 *       every step; with mu = the descriptor's `beta`,
 *           M = G + mu R;  U = orth(M V);  W = M^T U;  Vbar = orth(W);
 *           X <- X - eta s U Vbar^T;  R <- M;  V <- Vbar
 */
typedef enum { DION_VARIANT_DION = 0, DION_VARIANT_ORTH = 1, DION_VARIANT_LOWRANK_MUON = 2 } dion_variant_t;
typedef enum { DION_DTYPE_F32 = 0, DION_DTYPE_BF16 = 1 } dion_dtype_t;

/* One weight matrix and its optimizer state (all device pointers, caller-owned).
 * Requirements: 1 <= m, n < 2^31; 1 <= r <= min(m, n); ld_* >= n; every pointer 16-byte aligned;
 * ld_x, ld_r multiples of 4 and ld_g a multiple of 16 bytes / element size. */
typedef struct {
  float* X;          /* parameters, m x n fp32, updated in place                 */
  const void* G;     /* gradient, m x n, fp32 or bf16 (g_dtype), read only        */
  float* R;          /* error-feedback residual, m x n fp32, updated in place     */
  float* V;          /* n x r fp32: V_prev on entry, Vbar on exit                 */
  int64_t m, n, r;
  int64_t ld_x, ld_g, ld_r;
  int32_t g_dtype;   /* dion_dtype_t */
  int32_t variant;   /* dion_variant_t */
  float eta;         /* learning rate                                             */
  float beta;        /* error-feedback coefficient (momentum mu for LOWRANK_MUON)  */
  float scale;       /* s; <= 0 selects sqrt(m / n)                               */
  float reserved;    /* must be 0                                                 */
} dion_matrix_desc;

typedef struct dion_plan dion_plan;

/* Version of this ABI (DION_ABI_VERSION of the built library). */
DION_API int32_t dion_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
DION_API const char* dion_status_string(dion_status_t s);

/* Detail of the last error returned on the calling host thread ("" if none). */
DION_API const char* dion_last_error(void);

/*
 * Validate `count` descriptors and build a plan (host only: no CUDA call).
 * On success *out receives the plan and *workspace_bytes the size of the
 * device workspace every launching call needs (caller-allocated, 256-byte
 * aligned, contents need not be initialised).  The descriptors are copied.
 * Errors: DION_ERR_INVALID_ARG (bad descriptor or overlapping buffers; see
 * dion_last_error()), DION_ERR_UNSUPPORTED (alignment / leading dimension).
 */
DION_API dion_status_t dion_plan_create(const dion_matrix_desc* descs, int32_t count,
                               size_t* workspace_bytes, dion_plan** out);

/* Free a plan (host memory only).  NULL is ignored. */
DION_API void dion_plan_destroy(dion_plan* plan);

/* Number of matrices in the plan, or -1 for NULL. */
DION_API int32_t dion_plan_count(const dion_plan* plan);

/*
 * Change eta / beta of matrix `idx` (host only).  Takes effect at the next
 * launching call, which re-uploads the plan's tables into the workspace.
 */
DION_API dion_status_t dion_plan_set_hparams(dion_plan* plan, int32_t idx, float eta, float beta);

/*
 * Copy the plan's device tables into `workspace` on `stream` (one
 * cudaMemcpyAsync).  Launching calls do this themselves whenever the
 * workspace pointer or the hyper-parameters changed; call it explicitly
 * before capturing dion_step_batched() into a CUDA graph.
 */
DION_API dion_status_t dion_plan_upload(dion_plan* plan, void* workspace, size_t ws_bytes, void* stream);

/*
 * One full optimizer step for every matrix of the plan, enqueued on
 * `stream` (phases (a)-(e) below, all asynchronous, no host sync).
 */
DION_API dion_status_t dion_step_batched(dion_plan* plan, void* workspace, size_t ws_bytes, void* stream);

/*
 * Run phases first..last (inclusive) of a step, for tests and profiling:
 *   0 (a): reset status, P = (G + R) V                    (P in the workspace;
 *          for Dion matrices V is first replaced by orth(V), which leaves
 *          orth(P) unchanged and keeps P well conditioned)
 *   1 (b): U = orth(P)                                     (U in the workspace)
 *   2 (c): W = (G + R)^T U                                 (W in the workspace)
 *   3 (d): Vbar = orth(W) or colnorm(W), written into V
 *   4 (e): X <- X - eta s U Vbar^T,  R <- beta (G + R - U W^T), one launch per
 *          256 of r (later launches carry X and R forward in fp32)
 * The tf32 halves of U, U^T, W and Vbar that the tensor-core kernels read
 * (workspace) are written by the phase that produces each factor.
 * Running 0..4 equals dion_step_batched().
 */
DION_API dion_status_t dion_step_phases(dion_plan* plan, void* workspace, size_t ws_bytes,
                               int32_t first, int32_t last, void* stream);

/* Intermediates of matrix `idx` that tests may read back from the workspace. */
enum { DION_BUF_P = 0, DION_BUF_U = 1, DION_BUF_W = 2 };

/*
 * Locate intermediate `which` of matrix `idx`: byte offset from the
 * workspace base, rows, valid columns (= r) and leading dimension (elements,
 * fp32).  Host only.
 */
DION_API dion_status_t dion_plan_buffer(const dion_plan* plan, int32_t idx, int32_t which,
                               size_t* byte_offset, int64_t* rows, int64_t* cols, int64_t* ld);

/*
 * Copy the per-matrix status words of the last step into host array
 * `per_matrix` (count entries).  Synchronises `stream`.
 */
DION_API dion_status_t dion_plan_get_status(dion_plan* plan, const void* workspace, size_t ws_bytes,
                                   uint32_t* per_matrix, void* stream);

/* Kernel launches enqueued by one dion_step_batched() call of this plan. */
DION_API int32_t dion_plan_launches_per_step(const dion_plan* plan);

/*
 * Row-sharded step (the sharded setting of the Dion abstract, searcharxiv
 * 2504.05295, "integrating cleanly with weight sharding"; Orth-Dion abstract,
 * thelatestinai.com 2605.16341: the same per-step communication as Dion).
 *
 * Every rank makes a plan over its own rows of each matrix (the descriptors
 * hold the local m; n, r, variant and the hyper-parameters are the same on
 * every rank, and `scale` must be set explicitly to s of the whole matrix,
 * e.g. sqrt(m_total / n)); V is replicated.  One step is five stages, with the
 * caller summing a workspace region over all ranks (an all-reduce, e.g. NCCL)
 * after stages 0, 1, 2 (region DION_EXCHANGE_GRAM: the r x r Grams of every
 * CholeskyQR pass of orth(P)) and 3 (region DION_EXCHANGE_W: every W = M^T U):
 *   0  P = M V over the local rows, its Gram       -> all-reduce GRAM
 *   1  CholeskyQR pass 1 on the summed Gram        -> all-reduce GRAM
 *   2  CholeskyQR pass 2 (U, unless shifted)       -> all-reduce GRAM
 *   3  shifted pass (if any), W over local rows    -> all-reduce W
 *   4  Vbar = orth(W) | colnorm(W), X and R update of the local rows, V <- Vbar
 * On one rank with no exchange, stages 0..4 compute the same step as
 * dion_step_batched().  Asynchronous on `stream`; the caller's all-reduce must
 * be ordered after the stage on that stream.  The per-matrix status words are
 * the same as for the fused step.
 */
enum { DION_EXCHANGE_GRAM = 0, DION_EXCHANGE_W = 1 };
DION_API dion_status_t dion_shard_stage(dion_plan* plan, void* workspace, size_t ws_bytes, int32_t stage,
                                        void* stream);

/*
 * Testing hook for the bounded waits (no counterpart on the pages).  Sets, on
 * `stream`, the limit after which every pipeline wait of the tensor-core
 * kernels gives up (limit_ns <= 0 restores the default of 2 s), and makes the
 * update kernel's operand producer stop issuing at the first tile of plan
 * matrix `withhold_matrix` (-1: off), so that a consumer's wait on it runs
 * out: the kernel raises its abort flag, drains its own copies, frees its
 * TMEM, returns, and marks DION_MAT_TIMEOUT on every matrix the aborting CTA
 * had work for.  Both settings are process-wide for the current device and
 * stay until changed; for tests only.
 */
DION_API dion_status_t dion_debug_expire_wait(int64_t limit_ns, int32_t withhold_matrix, void* stream);

/* Byte offset from the workspace base and size of exchange region `which`
 * (DION_EXCHANGE_GRAM: the matrices' rp x rp fp32 Grams back to back; DION_EXCHANGE_W:
 * their n x rp fp32 W back to back; rp = r rounded up to 32).  Host only. */
DION_API dion_status_t dion_plan_exchange(const dion_plan* plan, int32_t which, size_t* byte_offset, size_t* bytes);

/*
 * orth() of one matrix for callers that cannot allocate device memory.
 *
 * Some callers may not call cudaMalloc at all: code running inside a CUDA
 * graph capture, inside another library's allocator callback, or under a
 * memory manager that owns every device byte.  This entry point needs nothing
 * beyond the caller's input and output: its scratch is a fixed array of
 * 4,760,320 bytes inside libdion.so itself (one copy on every GPU that loads
 * the library, kept until the process exits).  It has no counterpart on the pages; it
 * computes the same orth() as the plan-based step (the Q factor of a thin QR
 * whose triangular factor has a positive diagonal), with the CUDA-core kernels
 * of that step (CholeskyQR2, shifted CholeskyQR3 for kappa(A) > ~1e3).
 *
 *   A  rows x r fp32 row-major device array (leading dimension lda >= r), read only
 *   Q  rows x r fp32 row-major device array (ldq >= r), written; may not overlap A
 *   1 <= r <= min(rows, DION_NOALLOC_MAX_RANK), rows <= DION_NOALLOC_MAX_ROWS
 *
 * Returns DION_ERR_UNSUPPORTED for sizes beyond those limits or a device
 * index of 64 or more (nothing is launched), DION_ERR_INVALID_ARG for NULL
 * pointers or bad leading dimensions, DION_ERR_CUDA if a launch fails.  The
 * work is enqueued on `stream`; with status != NULL the call then copies the
 * matrix's status word (DION_MAT_* bits; Q is valid when no bit other than
 * DION_MAT_SHIFTED is set) to *status and synchronises the stream, with
 * status == NULL it returns without waiting.  Pass status == NULL while the
 * stream is being captured: the copy to pageable host memory and the
 * synchronisation are not allowed inside a capture.
 *
 * Every call shares the one scratch array and overwrites it (the status word
 * is cleared by each call).  Calls whose work overlaps on the GPU (different
 * streams, different host threads) race on it: order them on one stream.  The
 * first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before starting any
 * stream capture.  That address is cached and not looked up again after a
 * cudaDeviceReset().  The call allocates nothing: no cudaMalloc, no cudaFree,
 * no allocating library routine.
 */
#define DION_NOALLOC_MAX_ROWS 8192
#define DION_NOALLOC_MAX_RANK 64
DION_API dion_status_t dion_orth_noalloc(const float* A, int64_t rows, int64_t r, int64_t lda, float* Q,
                                         int64_t ldq, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DION_H_ */
