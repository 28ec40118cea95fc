// Blocked Cholesky factorisation and triangular inverse of the Grams of orth()
// (CholeskyQR: S = A^T A = Rc^T Rc, T = Rc^-1, Q = A T; orth() = the Q factor of
// a thin QR with a positive diagonal, junaidaliop.github.io "Orth-Dion", symbol
// glossary) for ranks whose r x r Gram does not fit one CTA's shared memory.
//
// Every job's Gram (the reduced sum in o.gsum, rp x rp, row-major) is copied to
// o.S (k_stats, k_copy) and factored in place in 128-wide panels; T is built in
// o.T.  Per panel p (one launch each, all jobs at once):
//   k_diag_gj one CTA per job: Cholesky + inverse of the diagonal block S_pp by the
//             register Gauss-Jordan elimination of chol_gj.cuh
//   k_panel   one CTA per 64-column slab: the row panel R_pc = T_pp^T S_pc
//   k_update  one CTA per 64 x 64 tile of the trailing upper triangle:
//             S_ac -= R_pa^T R_pc
// then k_check (pivots; pass 0 may ask for the shifted repetition of shifted
// CholeskyQR, see simt.cuh), and the off-diagonal blocks of T by recursive
// doubling over pairs of diagonal blocks A, C (levels of NB, 2 NB, 4 NB ...):
//   k_inv_pairs  one CTA per 64 x 64 tile: Y = R_AC T_C, then T_AC = -T_A Y
// All arithmetic is fp32 with fp32 accumulation in a fixed order.  A job whose
// rank ends before panel p (or before a level's pair) skips that launch.
#pragma once

#include "chol_gj.cuh"
#include "common.cuh"
#include "simt.cuh"

namespace dion {
namespace bchol {

constexpr int NB = 128;        // panel width
constexpr int SLAB = 64;       // output column slab of k_panel
constexpr int NT = 256;        // threads of k_stats, k_copy, k_panel
// dynamic shared memory of k_panel: T_pp and the slab of S
constexpr size_t PANEL_SMEM = sizeof(float) * (NB * (NB + 1) + NB * SLAB);
constexpr int COPY_ELEMS = 4096;   // elements of S and of T per CTA of k_copy

// Per-job scratch after the rp x rp factor in o.S (the S region has rp + 32 rp floats more).
struct Scr {
  float minp;       // smallest squared pivot of the factorisation
  float maxd;       // largest diagonal entry of the factored Gram
  unsigned bad;     // status bits of a failed factorisation (0: none)
  float shift;      // shift of the repeated pass 0 (shifted CholeskyQR)
  unsigned retry;   // pass 0 asked for the shifted repetition
};

__device__ __forceinline__ Scr* scr(const OrthJob& o) { return reinterpret_cast<Scr*>(o.S + o.rp * o.rp); }

// Does this launch of pass `pass` work on job o?  retry: the shifted repetition of pass 0.
__device__ __forceinline__ bool live(const OrthJob& o, int pass, int retry) {
  if (*o.status & ST_FATAL) return false;
  if (pass == 2 && !*o.flag) return false;
  if (retry && !scr(o)->retry) return false;
  return true;
}

// Scratch reset, largest diagonal and (first attempt of pass 0) the shift, one CTA per job.
__global__ void __launch_bounds__(NT) k_stats(const OrthJob* __restrict__ jobs, int pass, int retry) {
  __shared__ float s_tr[NT / 32], s_mx[NT / 32];
  const OrthJob& o = jobs[blockIdx.x];
  if (!live(o, pass, retry)) return;
  Scr* sc = scr(o);
  const int r = (int)o.r, rp = (int)o.rp;
  const float shift = retry ? sc->shift : 0.f;
  float tr = 0.f, mx = 0.f;
  for (int a = threadIdx.x; a < r; a += NT) {
    const float d = o.gsum[(long long)a * rp + a];
    tr += d;
    mx = fmaxf(mx, d + shift);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    tr += __shfl_xor_sync(0xffffffffu, tr, off);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if ((threadIdx.x & 31) == 0) { s_tr[threadIdx.x >> 5] = tr; s_mx[threadIdx.x >> 5] = mx; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f, m = 0.f;
    for (int w = 0; w < NT / 32; ++w) { t += s_tr[w]; m = fmaxf(m, s_mx[w]); }
    sc->minp = INFINITY;
    sc->maxd = m;
    sc->bad = 0u;
    if (!retry) {
      // shift of shifted CholeskyQR: 11 (rows r + r (r + 1)) u ||A||_F^2, ||A||_F^2 = trace(S)
      sc->shift = 11.f * ((float)o.rows * (float)r + (float)r * (float)(r + 1)) * 5.9604645e-8f * t;
      sc->retry = 0u;
    }
  }
}

// S = gsum (+ the shift on the diagonal in the shifted repetition), T = 0; COPY_ELEMS
// elements of each per CTA, `nblk` CTAs per job.
__global__ void __launch_bounds__(NT) k_copy(const OrthJob* __restrict__ jobs, int pass, int retry, int nblk) {
  const OrthJob& o = jobs[blockIdx.x / nblk];
  if (!live(o, pass, retry)) return;
  const long long r = o.r, rp = o.rp;
  const long long e0 = (long long)(blockIdx.x % nblk) * COPY_ELEMS;
  const float shift = retry ? scr(o)->shift : 0.f;
  for (int k = threadIdx.x; k < COPY_ELEMS; k += NT) {
    const long long e = e0 + k;
    if (e < r * r) {
      const long long a = e / r, c = e % r;
      o.S[a * rp + c] = o.gsum[a * rp + c] + (a == c ? shift : 0.f);
    }
    if (e < rp * rp) o.T[e] = 0.f;
  }
}

// The diagonal block of panel p (nb <= 128) by the register Gauss-Jordan elimination
// of chol_gj.cuh, one CTA per job: Rc_pp = D^1/2 L^T into S, T_pp = L^-T D^-1/2 into T.
__global__ void __launch_bounds__(gj::NT, 1) k_diag_gj(const OrthJob* __restrict__ jobs, int pass, int retry, int p) {
  extern __shared__ float4 gj_smem4[];
  float* sm = reinterpret_cast<float*>(gj_smem4);
  const float* piv = sm + gj::OFF_PIV;
  const OrthJob& o = jobs[blockIdx.x];
  if (!live(o, pass, retry)) return;
  Scr* sc = scr(o);
  if (sc->bad) return;
  const int r = (int)o.r, rp = (int)o.rp, k0 = p * NB;
  if (k0 >= r) return;
  const int nb = min(NB, r - k0);
  float E[gj::PR][gj::PC];
  float minp;
  const unsigned bad = gj::eliminate(E, o.S + (long long)k0 * rp + k0, rp, nb, 0.f, sm, &minp);
  if (bad) {
    if (threadIdx.x == 0) sc->bad = bad;
    return;
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
  for (int a = 0; a < gj::PR; ++a) {
    const int i = w + gj::NW * a;
    if (i >= nb) continue;
    const float si = sqrtf(piv[i]), ti = 1.f / si;
#pragma unroll
    for (int b = 0; b < gj::PC; ++b) {
      const int c = l + 32 * b;
      if (c >= nb) continue;
      if (c >= i) o.S[(long long)(k0 + i) * rp + k0 + c] = E[a][b] / si;            // Rc[i][c] = d_i L_ci / sqrt(d_i)
      if (c < i) o.T[(long long)(k0 + c) * rp + k0 + i] = E[a][b] * ti;             // T[c][i] = (L^-1)_ic / sqrt(d_i)
      else if (c == i) o.T[(long long)(k0 + i) * rp + k0 + i] = ti;
    }
  }
  if (threadIdx.x == 0) sc->minp = fminf(sc->minp, minp);
}

// Row panel of panel p, 64 columns per CTA: R_pc = T_pp^T S_pc (in place in S).
__global__ void __launch_bounds__(NT) k_panel(const OrthJob* __restrict__ jobs, int pass, int retry, int p,
                                              int nslab) {
  extern __shared__ float sm_panel[];
  float (*Tp)[NB + 1] = reinterpret_cast<float (*)[NB + 1]>(sm_panel);               // T_pp, T[t][i] (upper)
  float (*Sp)[SLAB] = reinterpret_cast<float (*)[SLAB]>(sm_panel + NB * (NB + 1));   // S_pc slab
  const OrthJob& o = jobs[blockIdx.x / nslab];
  const int slab = blockIdx.x % nslab;
  if (!live(o, pass, retry) || scr(o)->bad) return;
  const int r = (int)o.r, rp = (int)o.rp, k0 = p * NB;
  if (k0 >= r) return;
  const int nb = min(NB, r - k0);
  const int c0 = k0 + nb + slab * SLAB;
  if (c0 >= r) return;
  const int nc = min(SLAB, r - c0);
  for (int e = threadIdx.x; e < nb * nb; e += NT) {
    const int t = e / nb, i = e % nb;
    Tp[t][i] = o.T[(long long)(k0 + t) * rp + k0 + i];
  }
  for (int e = threadIdx.x; e < nb * SLAB; e += NT) {
    const int t = e / SLAB, c = e % SLAB;
    Sp[t][c] = c < nc ? o.S[(long long)(k0 + t) * rp + c0 + c] : 0.f;
  }
  __syncthreads();
  float out[NB * SLAB / NT];
#pragma unroll
  for (int q = 0; q < NB * SLAB / NT; ++q) {
    const int e = threadIdx.x + q * NT, i = e / SLAB, c = e % SLAB;
    float v = 0.f;
    if (i < nb)
      for (int t = 0; t <= i; ++t) v = fmaf(Tp[t][i], Sp[t][c], v);
    out[q] = v;
  }
  __syncthreads();
#pragma unroll
  for (int q = 0; q < NB * SLAB / NT; ++q) {
    const int e = threadIdx.x + q * NT, i = e / SLAB, c = e % SLAB;
    if (i < nb && c < nc) o.S[(long long)(k0 + i) * rp + c0 + c] = out[q];
  }
}

// Trailing update after panel p, one 64 x 64 tile (ta <= tc) of the upper triangle
// per CTA: S_ac -= sum_i R_p,a[i] R_p,c[i].
__global__ void __launch_bounds__(simt::NT) k_update(const OrthJob* __restrict__ jobs, int pass, int retry, int p,
                                                     int ntile) {
  __shared__ float As[simt::TK * simt::LDS], Bs[simt::TK * simt::LDS];
  const OrthJob& o = jobs[blockIdx.x / ntile];
  int t = blockIdx.x % ntile;
  if (!live(o, pass, retry) || scr(o)->bad) return;
  const int r = (int)o.r, rp = (int)o.rp, k0 = p * NB;
  if (k0 >= r) return;
  const int nb = min(NB, r - k0);
  const int c0 = k0 + nb;
  if (c0 >= r) return;
  const int T = (r - c0 + simt::TM - 1) / simt::TM;
  if (t >= T * (T + 1) / 2) return;
  int ta = 0;
  while (t >= T - ta) { t -= T - ta; ++ta; }
  const int tc = ta + t;
  const long long a0 = c0 + (long long)ta * simt::TM, cc0 = c0 + (long long)tc * simt::TN;
  float acc[4][4];
  simt::zero(acc);
  // A(i, k) = S[k0 + k][i], B(k, j) = S[k0 + k][j]: rows of the panel are K
  simt::LoadRMT la{o.S + (long long)k0 * rp, rp, nb, r};
  simt::LoadRM lb{o.S + (long long)k0 * rp, rp, nb, r};
  simt::tile_acc<false, true>(la, lb, a0, cc0, 0, nb, acc, As, Bs);
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long a = a0 + ty * 4 + u;
    if (a >= r) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const long long c = cc0 + tx * 4 + v;
      if (c < r) o.S[a * rp + c] -= acc[u][v];
    }
  }
}

// Pivot checks, one thread per job.  Pass 0: a breakdown or pivots implying
// kappa > ~1e3 ask for the shifted repetition; the repetition's outcome sets the
// status (DION_MAT_SHIFTED and the three-pass flag, or the failure bits).
// Passes 1 and 2: a failure sets the status.
__global__ void k_check(const OrthJob* __restrict__ jobs, int njob, int pass, int retry) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= njob) return;
  const OrthJob& o = jobs[j];
  if (!live(o, pass, retry)) return;
  Scr* sc = scr(o);
  if (pass == 0 && !retry) {
    if (sc->bad || sc->minp < 1e-6f * sc->maxd) sc->retry = 1u;
  } else if (pass == 0) {
    if (sc->bad) {
      atomicOr(o.status, sc->bad);
    } else {
      *o.flag = 1u;
      atomicOr(o.status, ST_SHIFTED);
    }
  } else if (sc->bad) {
    atomicOr(o.status, sc->bad);
  }
}


// Off-diagonal blocks of T = Rc^-1 by recursive doubling, level `level` (block size
// s = NB << level): for every pair of diagonal blocks A = [a, a + s) and
// C = [a + s, min(a + 2 s, r)) with T_A and T_C complete,
//     step 0:  Y   = R_AC T_C       (into the rows and columns of T_AC of Tt_hi, free
//                                     until T's tf32 halves are written)
//     step 1:  T_AC = -T_A Y
// (the inverse of [[R_A, R_AC], [0, R_C]]).  One CTA per 64 x 64 output tile; T_C
// upper triangular limits step 0's K to the tile's last column, T_A step 1's K to
// the tile's first row.  log2 of the number of panels levels instead of one launch
// per block diagonal, each over every pair of the level at once.
__global__ void __launch_bounds__(simt::NT) k_inv_pairs(const OrthJob* __restrict__ jobs, int pass, int level,
                                                        int step, int ntile) {
  __shared__ float As[simt::TK * simt::LDS], Bs[simt::TK * simt::LDS];
  const OrthJob& o = jobs[blockIdx.x / ntile];
  int t = blockIdx.x % ntile;
  if (!live(o, pass, 0) || scr(o)->bad) return;
  const int r = (int)o.r, rp = (int)o.rp;
  const int sz = NB << level, tps = sz / simt::TM;       // tiles per side of a pair's block
  const int m = t / (tps * tps);
  t %= tps * tps;
  const long long a = 2LL * sz * m, c_beg = a + sz;
  if (c_beg >= r) return;
  const long long c_end = a + 2LL * sz < r ? a + 2LL * sz : (long long)r;
  const long long i0 = a + (long long)(t / tps) * simt::TM, c0 = c_beg + (long long)(t % tps) * simt::TN;
  if (c0 >= c_end) return;
  float* Y = o.Tt_hi;
  float acc[4][4];
  simt::zero(acc);
  if (step == 0) {
    simt::LoadRM la{o.S, rp, r, r};                     // R_AC(i, t) = S[i][t]
    simt::LoadRM lb{o.T, rp, r, r};                     // T_C(t, c)
    const long long ke = c0 + simt::TN < c_end ? c0 + simt::TN : c_end;   // T_C[t][c] = 0 for t > c
    simt::tile_acc<true, true>(la, lb, i0, c0, c_beg, ke, acc, As, Bs);
  } else {
    simt::LoadRM la{o.T, rp, r, r};                     // T_A(i, u)
    simt::LoadRM lb{Y, rp, r, r};                       // Y(u, c)
    simt::tile_acc<true, true>(la, lb, i0, c0, i0, c_beg, acc, As, Bs);
  }
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float* dst = step == 0 ? Y : o.T;
  const float sign = step == 0 ? 1.f : -1.f;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long i = i0 + ty * 4 + u;
    if (i >= c_beg) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const long long c = c0 + tx * 4 + v;
      if (c < c_end) dst[i * rp + c] = sign * acc[u][v];
    }
  }
}

}  // namespace bchol
}  // namespace dion
