// Device-side tables shared by every kernel of libdion.
//
// The host builds these once per plan (dion_plan_create) and copies them into
// the caller's workspace (dion_plan_upload); every grouped launch walks them.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace dion {

// Per-matrix status bits (same values as DION_MAT_* in dion.h).
constexpr unsigned ST_BREAKDOWN = 1u;
constexpr unsigned ST_NONFINITE = 2u;
constexpr unsigned ST_TIMEOUT = 4u;     // a bounded wait inside a tensor-core kernel gave up
constexpr unsigned ST_SHIFTED = 8u;     // informational: an orth() of this matrix needed the shifted pass

// Layout of the tf32 operand halves that the update kernel (tcepi) reads: the
// shared-memory image of its K-major operand tiles, stored tile after tile, so
// that one tile is one contiguous 8 KB bulk copy (a TMA box of 64-byte rows is
// 128 row requests).  Tile (row / 128, k / 16) of a rows x rp matrix holds rows
// 128 t .. 128 t + 127 and columns 16 u .. 16 u + 15 in the 64-byte swizzle (row
// r at 64 r bytes, its 16-byte piece q at q ^ ((r / 2) mod 4)); rows are padded to
// a multiple of 128.  Returns the float offset of element (row, k).
constexpr int OPT_ROWS = 128, OPT_K = 16, OPT_FLOATS = OPT_ROWS * OPT_K;
__host__ __device__ __forceinline__ long long optile_idx(long long row, long long k, long long rp) {
  const long long t = (row / OPT_ROWS) * (rp / OPT_K) + k / OPT_K;
  const long long r = row % OPT_ROWS, kk = k % OPT_K;
  return t * OPT_FLOATS + r * OPT_K + ((((kk >> 2) ^ (r >> 1)) & 3) << 2) + (kk & 3);
}

// One weight matrix of the batch, with the workspace buffers of its step.
struct MatDev {
  float* X;            // m x n, ld ldx
  const void* G;       // m x n, ld ldg, fp32 or bf16
  float* R;            // m x n, ld ldr
  float* V;            // n x r dense: V_prev in, Vbar out
  const float* Vin;    // warm start read by phase (a): V itself (Orth-Dion) or orth(V) (Dion)
  long long ldvin;     // its leading dimension (r or rp)
  long long m, n, r, rp;       // rp = r rounded up to the tile granule
  long long ldx, ldg, ldr;
  int g_bf16;          // 1: G is bf16
  int variant;         // 0 Dion (colnorm), 1 Orth-Dion (QR)
  float eta_s;         // eta * s
  float beta;
  float mu;            // M = G + mu R (1, or the momentum coefficient of the low-rank Muon variant)
  float* P;            // m x rp   P = M V
  float* U;            // m x rp   U = orth(P)
  float* W;            // n x rp   W = M^T U
  float* Wpart;        // ksplit x n x rp partial sums of W (when ksplit > 1)
  float* Wh;           // n x rp   tf32 halves of W (operands of the update, optile layout), zero beyond column r
  float* Wl;
  int ksplit;          // split of the m-range in phase (c)
  int kchunk;          // rows of M per split
  unsigned* status;    // per-matrix status word
};

// Status bits that stop the rest of a matrix's step.
constexpr unsigned ST_FATAL = ST_BREAKDOWN | ST_NONFINITE;

// One orth() problem: A (rows x r, lda) -> out (rows x r, ldo), by CholeskyQR2,
// or shifted CholeskyQR3 when the first Cholesky shows A is ill conditioned.
struct OrthJob {
  const float* A;      // input, rows x r (ld lda)
  long long lda;
  float* Q;            // first-pass factor, rows x rp (ld rp)
  float* Q2;           // second-pass factor of a shifted (three-pass) job, rows x rp
  unsigned* flag;      // 1: this job took the shifted first pass and needs a third
  float* out;          // result, rows x out_cols (ld ldo)
  long long ldo;
  long long out_cols;  // columns written to out (rp in the workspace, r into V)
  float* gpart;        // nchunk x rp x rp Gram partial sums
  float* gsum;         // rp x rp: their sum (k_gram_reduce), read by a reduced Cholesky
  float* S;            // rp x rp Gram / Cholesky factor
  float* T;            // rp x rp inverse of the Cholesky factor
  float* Tt_hi;        // rp x rp: T^T split into tf32 halves (B operand of the tensor-core A T)
  float* Tt_lo;
  long long rows, r, rp;
  int nchunk;          // row chunks of the Gram reduction
  int chunk;           // rows per chunk
  unsigned* status;
};

// Largest j in [0, n) with start[j] <= t (start[0] == 0, start[n] == total).
__device__ __forceinline__ int find_job(const int* __restrict__ start, int n, int t) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (start[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

}  // namespace dion
