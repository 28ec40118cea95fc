// Cholesky factorisation and inverse of the Gram of orth() for ranks up to 192
// (CholeskyQR: S = A^T A = Rc^T Rc, T = Rc^-1, Q = A T; orth() = the Q factor of
// a thin QR with a positive diagonal, junaidaliop.github.io "Orth-Dion", symbol
// glossary), one CTA per job, the whole r x r array in registers.
//
// Symmetric Gauss-Jordan elimination: step j subtracts l_ij = S_ij / S_jj times
// row j from every row i > j.  The array holds, in place, the upper triangle of
// the eliminated Gram (row i of D L^T for S = L D L^T, L unit lower triangular,
// D the pivots) and, in the strict lower triangle, the identity that the same
// row operations turn into L^-1.  Then Rc = D^1/2 L^T and T = Rc^-1 = L^-T D^-1/2,
// so row c of T^T is row c of L^-1 over sqrt(d_c): the kernel writes T^T's tf32
// halves directly.
//
// The steps are taken 16 at a time (a block J of pivots, one row per warp):
//   1. the 16 rows of J are staged in shared memory;
//   2. one warp eliminates the 16 x 16 diagonal block (lane c holds column c;
//      the multipliers come by shuffle), giving D_J, the upper part D_J L_JJ^T
//      and L_JJ^-1;
//   3. the rows of J are multiplied by L_JJ^-1 (their columns outside J: the
//      finished part of L^-1 on the left, the Gram on the right);
//   4. every row i after J takes the rank-16 update row_i -= sum_j l_ij row_j,
//      j in J, over its L^-1 columns and its Gram columns.
// Step 4 is where the work is; it has no per-element conditions: the rows after
// J carry their strict lower Gram entries along as scratch (kept only where a
// 16 x 32 register tile reaches the diagonal) and zero them when their block's
// L^-1 columns start.  Three barriers per block instead of one per column.
//
// Thread (warp w, lane l) holds the 72 entries (w + 16 a, l + 32 b), a < 12, b < 6:
// block J is row group a = J, and lanes 16 (J mod 2) .. + 15 of column group J / 2.
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
constexpr int JB = 16;               // pivots per block: one row group
constexpr int NBLK = RMAX / JB;      // 12
constexpr int LDA = RMAX + 1;        // staged row (odd: the diagonal warp reads rows and columns)
constexpr int LDD = JB + 1;

// dynamic shared memory, in floats
constexpr int OFF_A = 0;                         // JB x LDA: rows of J as they were
constexpr int OFF_P = OFF_A + JB * LDA;           // JB x RMAX: rows of J after step 3
constexpr int OFF_M = OFF_P + JB * RMAX;          // JB x RMAX: l_ij of row i at (i % 16) * 12 + i / 16
constexpr int OFF_D = OFF_M + JB * RMAX;          // JB x LDD: the eliminated diagonal block
constexpr int OFF_PIV = OFF_D + JB * LDD;         // RMAX pivots
constexpr int OFF_FLAG = OFF_PIV + RMAX;          // status and smallest pivot of the block
constexpr int SMEM_FLOATS = OFF_FLAG + 4;
constexpr size_t SMEM_BYTES = sizeof(float) * SMEM_FLOATS;
static_assert(OFF_M % 4 == 0, "multiplier rows are read as float4");

// lane l of column group J / 2 holds a column of block J
template <int J>
__device__ __forceinline__ bool in_block(int l) { return (l >> 4) == (J & 1); }

// Step 2, by warp 0: lane l holds rows 8 (l / 16) .. + 7 of column c = l mod 16 of
// the diagonal block (upper triangle from the staged rows, mirrored below) and
// eliminates them; the pivot row and the multipliers come by shuffle.  Afterwards
// column c holds d_k L_ck (k < c), d_c (k = c) and (L_JJ^-1)_kc (k > c).
__device__ __forceinline__ void diag_block(float* sm, int j0, int n) {
  const int l = threadIdx.x & 31, c = l & 15, hf = l >> 4;
  const float* A = sm + OFF_A;
  float v[8];
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const int k = 8 * hf + s;
    v[s] = k <= c ? A[k * LDA + j0 + c] : A[c * LDA + j0 + k];
  }
  unsigned bad = 0u;
  float minp = INFINITY;
#pragma unroll
  for (int t = 0; t < JB; ++t) {
    const int th = t >> 3, ts = t & 7;
    const float d = __shfl_sync(0xffffffffu, v[ts], t + 16 * th);
    const float pc = __shfl_sync(0xffffffffu, v[ts], c + 16 * th);   // row t at this lane's column
    if (j0 + t < n) {                      // the same decision in every lane
      if (!(d > 0.f) || !isfinite(d)) bad |= isfinite(d) ? ST_BREAKDOWN : (ST_BREAKDOWN | ST_NONFINITE);
      minp = fminf(minp, d);
    }
    if (threadIdx.x == 0) sm[OFF_PIV + j0 + t] = d;
    const float inv = 1.f / d;
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      const float f = __shfl_sync(0xffffffffu, v[s], t + 16 * hf) * inv;   // l_kt, k = 8 hf + s
      if (8 * hf + s > t) v[s] = c == t ? -f : fmaf(-f, pc, v[s]);
    }
  }
  float* D = sm + OFF_D;
#pragma unroll
  for (int s = 0; s < 8; ++s) D[(8 * hf + s) * LDD + c] = v[s];
  if (threadIdx.x == 0) {
    reinterpret_cast<unsigned*>(sm)[OFF_FLAG] = bad;
    sm[OFF_FLAG + 1] = minp;
  }
}

// Step 3: row j0 + w times L_JJ^-1 (unit diagonal), in the registers and in P;
// the multipliers l_ij = (row j of D L^T)_i / d_j of the rows i after J into M.
template <int J>
__device__ __forceinline__ void transform_row(float (&E)[PR][PC], float* sm) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const float* A = sm + OFF_A;
  const float* D = sm + OFF_D;
  float* P = sm + OFF_P;
  float* M = sm + OFF_M;
  float acc[PC];
#pragma unroll
  for (int b = 0; b < PC; ++b) acc[b] = A[w * LDA + l + 32 * b];
  for (int k = 0; k < w; ++k) {
    const float lk = D[w * LDD + k];       // (L_JJ^-1)_wk
#pragma unroll
    for (int b = 0; b < PC; ++b) acc[b] = fmaf(lk, A[k * LDA + l + 32 * b], acc[b]);
  }
  const float invd = 1.f / sm[OFF_PIV + J * JB + w];
  const int cc = l & 15;
  const bool inb = in_block<J>(l);
#pragma unroll
  for (int b = 0; b < PC; ++b) {
    float e = acc[b], pv = acc[b];
    if (b == J / 2 && inb) {
      e = D[w * LDD + cc];
      // the L^-1 columns of J as the later rows see them: unit diagonal, zero above
      pv = cc < w ? e : (cc == w ? 1.f : 0.f);
    }
    E[J][b] = e;
    P[w * RMAX + l + 32 * b] = pv;
    if (b > J / 2 || (b == J / 2 && (J & 1) == 0 && l >= 16))
      M[w * RMAX + cc * 12 + 2 * b + (l >> 4)] = acc[b] * invd;
  }
}

// Step 4 for the row groups a = J + 1 .. AMAX - 1 below the block (every a < AMAX
// when FULL, else the ones below amax): zero the L^-1 columns of J, then
// row_i -= sum_k l_ik P_k over the column groups up to J / 2 (L^-1, and the next
// block's diagonal) and the Gram tiles that reach the diagonal or above.
template <int J, bool FULL>
__device__ __forceinline__ void update_rows(float (&E)[PR][PC], const float* sm, int amax) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const float* P = sm + OFF_P;
  const float4* M4 = reinterpret_cast<const float4*>(sm + OFF_M);
  const bool inb = in_block<J>(l);
#pragma unroll
  for (int a = J + 1; a < PR; ++a)
    if (inb) E[a][J / 2] = 0.f;
#pragma unroll 2
  for (int k = 0; k < JB; ++k) {
    const float4 q0 = M4[k * (RMAX / 4) + w * 3], q1 = M4[k * (RMAX / 4) + w * 3 + 1],
                 q2 = M4[k * (RMAX / 4) + w * 3 + 2];
    const float m[PR] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w, q2.x, q2.y, q2.z, q2.w};
    float p[PC];
#pragma unroll
    for (int b = 0; b < PC; ++b) p[b] = P[k * RMAX + l + 32 * b];
#pragma unroll
    for (int a = J + 1; a < PR; ++a)
      if (FULL || a < amax)
#pragma unroll
        for (int b = 0; b < PC; ++b)
          if (b <= J / 2 || 2 * b + 2 > a) E[a][b] = fmaf(-m[a], p[b], E[a][b]);
  }
}

// Steps 1, 3 and 4 of block J (J a template argument, so that its register rows
// are addressed statically); step 2 is shared by all blocks.
template <int J>
__device__ __forceinline__ void stage_rows(const float (&E)[PR][PC], float* sm) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int b = 0; b < PC; ++b) sm[OFF_A + w * LDA + l + 32 * b] = E[J][b];
}

template <int J>
__device__ __forceinline__ void transform_update(float (&E)[PR][PC], float* sm, int nblk) {
  transform_row<J>(E, sm);
  __syncthreads();
  if constexpr (J + 1 < PR) {
    // row groups from nblk on are padding: they need no update
    if (nblk == NBLK) update_rows<J, true>(E, sm, NBLK);
    else if (J + 1 < nblk) update_rows<J, false>(E, sm, nblk);
  }
}

// CALL with J bound to the block index jb as a compile-time constant
#define GJ_SWITCH(CALL)                                                 \
  switch (jb) {                                                         \
    case 0: { constexpr int J = 0; CALL; } break;                       \
    case 1: { constexpr int J = 1; CALL; } break;                       \
    case 2: { constexpr int J = 2; CALL; } break;                       \
    case 3: { constexpr int J = 3; CALL; } break;                       \
    case 4: { constexpr int J = 4; CALL; } break;                       \
    case 5: { constexpr int J = 5; CALL; } break;                       \
    case 6: { constexpr int J = 6; CALL; } break;                       \
    case 7: { constexpr int J = 7; CALL; } break;                       \
    case 8: { constexpr int J = 8; CALL; } break;                       \
    case 9: { constexpr int J = 9; CALL; } break;                       \
    case 10: { constexpr int J = 10; CALL; } break;                     \
    default: { constexpr int J = 11; CALL; } break;                     \
  }

// The elimination itself, by the whole CTA: loads the upper triangle of the n x n
// symmetric S (leading dimension ld; + shift on the diagonal; identity on the
// padding up to the next multiple of 16) into E, eliminates, and returns 0 or the
// status bits of a breakdown.  Afterwards E's upper triangle holds row i of D L^T
// (E[i][i] = d_i, also at sm[OFF_PIV + i]) and its strict lower triangle L^-1;
// *minp receives the smallest pivot.  sm: SMEM_BYTES of shared memory.
__device__ __forceinline__ unsigned eliminate(float (&E)[PR][PC], const float* S, long long ld, int n, float shift,
                                              float* sm, float* minp_out) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int a = 0; a < PR; ++a)
#pragma unroll
    for (int b = 0; b < PC; ++b) {
      const int i = w + NW * a, c = l + 32 * b;
      E[a][b] = (i < n && c < n && c >= i) ? S[(long long)i * ld + c] + (i == c ? shift : 0.f)
                                           : (i == c && i >= n ? 1.f : 0.f);
    }
  const int nblk = (n + JB - 1) / JB;
  unsigned bad = 0u;
  float minp = INFINITY;
  for (int jb = 0; jb < nblk; ++jb) {
    GJ_SWITCH(stage_rows<J>(E, sm))
    __syncthreads();
    // one copy of the diagonal elimination for every block (its code is the largest part)
    if (w == 0) diag_block(sm, jb * JB, n);
    __syncthreads();
    bad = reinterpret_cast<const unsigned*>(sm)[OFF_FLAG];
    minp = fminf(minp, sm[OFF_FLAG + 1]);
    if (bad) break;                        // the same decision in every thread
    GJ_SWITCH(transform_update<J>(E, sm, nblk))
    // the next block's rows are staged over A and its diagonal over D only after
    // every thread has finished reading them
    __syncthreads();
  }
  *minp_out = minp;
  return bad;
}

__global__ void __launch_bounds__(NT, 1) k_chol_gj(const OrthJob* __restrict__ jobs, int pass,
                                                   const int* __restrict__ order) {
  extern __shared__ float4 gj_smem4[];
  float* sm = reinterpret_cast<float*>(gj_smem4);
  const float* piv = sm + OFF_PIV;   // the pivots d_j
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
    bad = eliminate(E, o.gsum, rp, r, shift, sm, &minp);
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
      o.Tt_hi[c * rp + k] = h;             // rp <= 192: 32-bit offsets
      o.Tt_lo[c * rp + k] = lo;
    }
  }
}

}  // namespace gj
}  // namespace dion
