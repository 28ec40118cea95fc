/*
 * muon.h -- C ABI of the Muon comparator in libdion.so: the step that the
 * Dion / Orth-Dion step is measured against, on the same shapes and GPU.
 *
 * The pages describe Muon only in words: it orthogonalises the momentum of
 * each weight matrix with a Newton-Schulz iteration whose cost is cubic in the
 * matrix size (searcharxiv 2608.11612 "Dion3" abstract; the artiverse.ca post
 * "What Made Muon Stand Out").  They print no coefficients or momentum rule;
 * the readings taken here, for every matrix of a plan:
 *
 *     B    <- mu B + G                       momentum, m x n fp32
 *     Y_0   = B / ||B||_F
 *     Y_k+1 = 1.5 Y_k - 0.5 Y_k Y_k^T Y_k    k = 0 .. ns_iters - 1 (cubic Newton-Schulz)
 *     X    <- X - eta s Y_K                  s = scale, sqrt(m / n) when scale <= 0
 *
 * The iteration forms the smaller Gram: (Y Y^T) for m <= n, (Y^T Y) for m > n.
 * Its two products per iteration are plain library GEMMs (cuBLAS, batched over
 * the matrices of equal shape); the momentum, the norms, the start of the
 * iteration and the update are this library's kernels.
 *
 * Conventions as in dion.h: row-major matrices, caller-owned device pointers
 * (X, B updated in place, G read only), leading dimensions in elements,
 * `stream` a cudaStream_t passed as void*, dion_status_t return codes, error
 * text from dion_last_error().  The workspace is caller-allocated (256-byte
 * aligned).  The cuBLAS handle a plan creates on its first step allocates
 * cuBLAS's own small state; its GEMM scratch is taken from the workspace.
 */
#ifndef MUON_H_
#define MUON_H_

#include "dion.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Arithmetic of the Newton-Schulz products (the momentum, the norms and the
 * update are fp32 in every mode). */
typedef enum {
  MUON_NS_BF16 = 0,   /* Y and the Gram stored in bf16, fp32 accumulation (common practice) */
  MUON_NS_TF32 = 1,   /* fp32 storage, TF32 tensor-core products                           */
  MUON_NS_FP32 = 2    /* fp32 storage and fp32 products                                     */
} muon_precision_t;

/* One weight matrix and its state.  Requirements: 1 <= m, n < 2^31; ld_* >= n;
 * pointers 16-byte aligned. */
typedef struct {
  float* X;          /* parameters, m x n fp32, updated in place           */
  const void* G;     /* gradient, m x n, fp32 or bf16 (g_dtype), read only  */
  float* B;          /* momentum, m x n fp32, updated in place             */
  int64_t m, n;
  int64_t ld_x, ld_g, ld_b;
  int32_t g_dtype;   /* dion_dtype_t */
  float eta;         /* learning rate                                       */
  float mu;          /* momentum coefficient                                */
  float scale;       /* s; <= 0 selects sqrt(m / n)                         */
} muon_matrix_desc;

typedef struct muon_plan muon_plan;

/*
 * Validate `count` descriptors and build a plan (host only).  ns_iters >= 0
 * Newton-Schulz iterations; precision a muon_precision_t.  *workspace_bytes
 * receives the device workspace every step needs.
 *
 * row_fraction in (0, 1] selects the Dion3 row-selection variant when below 1
 * (searcharxiv 2608.11612 "Dion3" abstract: only a fraction of the momentum
 * matrix's rows is orthogonalised at each step; the rule is not on the pages,
 * this library's reading): after the momentum update the k = ceil(row_fraction
 * m) rows of B with the largest Euclidean norms (ties: the lower row index) are
 * taken, the iteration runs on that k x n block normalised by its own Frobenius
 * norm, and only those rows of X are updated.  row_fraction = 1 is Muon itself.
 * The variant needs m <= DION3_MAX_ROWS (DION_ERR_UNSUPPORTED otherwise).
 */
#define DION3_MAX_ROWS 16384
DION_API dion_status_t muon_plan_create(const muon_matrix_desc* descs, int32_t count, int32_t ns_iters,
                                        int32_t precision, float row_fraction, size_t* workspace_bytes,
                                        muon_plan** out);

/*
 * Rows selected by the last step for matrix `idx` (row-selection variant):
 * byte offset from the workspace base of k int32 row indices, in increasing
 * order, and k.  Host only; DION_ERR_INVALID_ARG for a plan without selection.
 */
DION_API dion_status_t muon_plan_selected_rows(const muon_plan* plan, int32_t idx, size_t* byte_offset, int64_t* k);

/* One Muon step of every matrix of the plan, enqueued on `stream` (no host sync). */
DION_API dion_status_t muon_step_batched(muon_plan* plan, void* workspace, size_t ws_bytes, void* stream);

/* Kernel and GEMM launches enqueued by one muon_step_batched() call. */
DION_API int32_t muon_plan_launches_per_step(const muon_plan* plan);

/* Free a plan and its cuBLAS handle.  NULL is ignored. */
DION_API void muon_plan_destroy(muon_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* MUON_H_ */
