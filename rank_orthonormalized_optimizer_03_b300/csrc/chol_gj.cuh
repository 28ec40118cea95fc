// Cholesky factorisation and inverse of the Gram of orth() for ranks up to 192
// (CholeskyQR: S = A^T A = Rc^T Rc, T = Rc^-1, Q = A T; orth() = the Q factor of
// a thin QR with a positive diagonal, junaidaliop.github.io "Orth-Dion", symbol
// glossary), one CTA per job, the whole r x r array in registers.
//
// Symmetric Gauss-Jordan elimination: step j subtracts l_ij = S_ij / S_jj times
// row j from every row i > j, on the upper triangle of S (which stays the upper
// triangle of the trailing Gram) and, in the strict lower triangle, on the
// identity, which becomes L^-1 for S = L D L^T (L unit lower triangular, D the
// pivots).  Then Rc = D^1/2 L^T and T = Rc^-1 = L^-T D^-1/2, so row c of T^T is
// row c of L^-1 over sqrt(d_c): the kernel writes T^T's tf32 halves directly.
// One barrier per column (the pivot row is published to shared memory in a
// double buffer); no serial single-warp phase.
//
// Thread (warp w, lane l) holds the 72 entries (w + 16 a, l + 32 b), a < 12, b < 6.
// Conditioning as in simt::k_chol_inv: in pass 0 a breakdown or pivots implying
// kappa > ~1e3 (min pivot < 1e-6 max diagonal) repeat the elimination on the
// shifted Gram of shifted CholeskyQR and flag the job for a third pass.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace gj {

constexpr int NT = 512;
constexpr int NW = NT / 32;          // 16 warps
constexpr int PR = 12;               // rows per thread (w + 16 a)
constexpr int PC = 6;                // columns per thread (l + 32 b)
constexpr int RMAX = NW * PR;        // 192
static_assert(RMAX == 32 * PC, "rows and columns cover the same 192");

// The elimination itself, by the whole CTA: loads the upper triangle of the n x n
// symmetric S (leading dimension ld; + shift on the diagonal) into E, eliminates,
// and returns 0 or the status bits of a breakdown.  Afterwards E's upper triangle
// holds row i of D L^T (E[i][i] = d_i, also in piv[i]) and its strict lower
// triangle L^-1; *minp receives the smallest pivot.  `row` is 2 x RMAX floats of
// shared memory, `piv` RMAX floats.
__device__ __forceinline__ unsigned eliminate(float (&E)[PR][PC], const float* S, long long ld, int n, float shift,
                                              float (*row)[RMAX], float* piv, float* minp_out) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int a = 0; a < PR; ++a)
#pragma unroll
    for (int b = 0; b < PC; ++b) {
      const int i = w + NW * a, c = l + 32 * b;
      E[a][b] = (i < n && c < n && c >= i) ? S[(long long)i * ld + c] + (i == c ? shift : 0.f) : 0.f;
    }
  unsigned bad = 0u;
  float minp = INFINITY;
  for (int j = 0; j < n; ++j) {
    float* buf = row[j & 1];
    if (w == j % NW) {
      const int a = j / NW;
#pragma unroll
      for (int aa = 0; aa < PR; ++aa)
        if (aa == a)
#pragma unroll
          for (int b = 0; b < PC; ++b) buf[l + 32 * b] = E[aa][b];
    }
    __syncthreads();
    const float d = buf[j];
    if (!(d > 0.f) || !isfinite(d)) {      // the same decision in every thread
      bad = isfinite(d) ? ST_BREAKDOWN : (ST_BREAKDOWN | ST_NONFINITE);
      break;
    }
    if (threadIdx.x == 0) piv[j] = d;
    minp = fminf(minp, d);
    const float inv = 1.f / d;
#pragma unroll
    for (int a = 0; a < PR; ++a) {
      const int i = w + NW * a;
      if (i <= j || i >= n) continue;
      const float f = buf[i] * inv;        // l_ij = S_ji / S_jj (S_ji in row j's upper part)
#pragma unroll
      for (int b = 0; b < PC; ++b) {
        const int c = l + 32 * b;
        if (c >= n) continue;
        if (c >= i || c < j) E[a][b] = fmaf(-f, buf[c], E[a][b]);   // S_ic, or (L^-1)_ic
        else if (c == j) E[a][b] = -f;                               // (L^-1)_ij
      }
    }
  }
  __syncthreads();
  *minp_out = minp;
  return bad;
}

__global__ void __launch_bounds__(NT, 1) k_chol_gj(const OrthJob* __restrict__ jobs, int pass,
                                                   const int* __restrict__ order) {
  __shared__ float row[2][RMAX];     // the pivot row of the current step
  __shared__ float piv[RMAX];        // the pivots d_j
  __shared__ float red[2];
  const OrthJob& o = jobs[order ? order[blockIdx.x] : blockIdx.x];
  if (*o.status & ST_FATAL) return;
  if (pass == 2 && !*o.flag) return;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int r = (int)o.r, rp = (int)o.rp;
  // trace and largest diagonal entry of the Gram
  float tr = 0.f, mx = 0.f;
  if (w == 0)
    for (int j = l; j < r; j += 32) {
      const float d = o.gsum[(long long)j * rp + j];
      tr += d;
      mx = fmaxf(mx, d);
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    tr += __shfl_xor_sync(0xffffffffu, tr, off);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (threadIdx.x == 0) { red[0] = tr; red[1] = mx; }
  __syncthreads();
  const float trace = red[0], maxd = red[1];

  float E[PR][PC];
  unsigned bad = 0u;
  int attempt = 0;
  for (;; ++attempt) {
    const float shift =
        attempt ? 11.f * ((float)o.rows * (float)r + (float)r * (float)(r + 1)) * 5.9604645e-8f * trace : 0.f;
    float minp;
    bad = eliminate(E, o.gsum, rp, r, shift, row, piv, &minp);
    const bool shifted_try = pass == 0 && attempt == 0 && (bad || minp < 1e-6f * maxd);
    if (!shifted_try) break;
  }
  if (bad) {
    if (threadIdx.x == 0) atomicOr(o.status, bad);
    return;
  }
  if (attempt == 1 && threadIdx.x == 0) {
    *o.flag = 1u;
    atomicOr(o.status, ST_SHIFTED);
  }
  // T^T[c][a] = (L^-1)[c][a] / sqrt(d_c) for a < c, 1 / sqrt(d_c) for a = c, 0 above;
  // zero in the padding rows and columns r .. rp-1
#pragma unroll
  for (int a = 0; a < PR; ++a) {
    const int c = w + NW * a;              // row of T^T
    if (c >= rp) continue;
    const float sc = c < r ? 1.f / sqrtf(piv[c]) : 0.f;
#pragma unroll
    for (int b = 0; b < PC; ++b) {
      const int k = l + 32 * b;            // column of T^T
      if (k >= rp) continue;
      const float v = (c < r && k < r) ? (k < c ? E[a][b] * sc : (k == c ? sc : 0.f)) : 0.f;
      float h, lo;
      tc::split_tf32(v, h, lo);
      o.Tt_hi[(long long)c * rp + k] = h;
      o.Tt_lo[(long long)c * rp + k] = lo;
    }
  }
}

}  // namespace gj
}  // namespace dion
