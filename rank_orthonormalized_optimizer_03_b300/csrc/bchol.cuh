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
// CholeskyQR, see simt.cuh), and the off-diagonal blocks of T by block
// diagonals d = q - p:
//   k_inv     one CTA per 64-column slab of block (p, q):
//             T_pq = -T_pp sum_{k=p+1..q} R_pk T_kq
// All arithmetic is fp32 with fp32 accumulation in a fixed order.  A job whose
// rank ends before panel p (or diagonal d) skips that launch.
#pragma once

#include "chol_gj.cuh"
#include "common.cuh"
#include "simt.cuh"

namespace dion {
namespace bchol {

constexpr int NB = 128;        // panel width
constexpr int SLAB = 64;       // output column slab of k_panel and k_inv
constexpr int NT = 256;        // threads of k_stats, k_copy, k_panel, k_inv
// dynamic shared memory: k_inv holds T_pp (NB x NB+1) and C (NB x SLAB+1), k_panel
// T_pp and the slab of S
constexpr size_t INV_SMEM = sizeof(float) * (NB * (NB + 1) + NB * (SLAB + 1));
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

// Block (p, p + d) of T, one 64-column slab per CTA:
//   C = sum_{k = p+1 .. q} R_pk T_kq  (K = the rows of panels p+1 .. q),  T_pq = -T_pp C.
__global__ void __launch_bounds__(NT) k_inv(const OrthJob* __restrict__ jobs, int pass, int d, int nitem) {
  extern __shared__ float sm_inv[];
  const OrthJob& o = jobs[blockIdx.x / nitem];
  const int it = blockIdx.x % nitem;
  if (!live(o, pass, 0) || scr(o)->bad) return;
  const int r = (int)o.r, rp = (int)o.rp;
  const int np = (r + NB - 1) / NB;
  if (d >= np || it >= (np - d) * (NB / SLAB)) return;
  const int p = it / (NB / SLAB), q = p + d;
  const int k0 = p * NB, nb = min(NB, r - k0);
  const int c0 = q * NB + (it % (NB / SLAB)) * SLAB;
  if (c0 >= r) return;
  const int nc = min(SLAB, r - c0);
  const int kb = k0 + nb, ke = min(r, c0 + nc);     // T[t][c] = 0 for t > c
  float* Tp = sm_inv;                                // NB x (NB + 1)
  float* Cs = sm_inv + NB * (NB + 1);                // NB x (SLAB + 1)
  float* Rs = Tp;                                    // phase 1 tiles reuse Tp's space:
  float* Ts = Tp + 16 * (NB + 1);                    //   Rs 16 x (NB + 1) (k, i), Ts 16 x SLAB (k, c)
  // thread tile: rows i = ty * 8 + u (u < 8), columns c = tx * 4 + v (v < 4)
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  float acc[8][4];
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
  for (int kt = kb; kt < ke; kt += 16) {
    // 16 consecutive threads read 16 consecutive columns t of one row of S (a row
    // segment, not a column walk); the padded row of Rs keeps the transposed
    // stores off a single bank
    for (int e = threadIdx.x; e < 16 * NB; e += NT) {
      const int kk = e % 16, i = e / 16, t = kt + kk;
      Rs[kk * (NB + 1) + i] = (t < ke && i < nb) ? o.S[(long long)(k0 + i) * rp + t] : 0.f;
    }
    for (int e = threadIdx.x; e < 16 * SLAB; e += NT) {
      const int kk = e / SLAB, c = e % SLAB, t = kt + kk;
      Ts[kk * SLAB + c] = (t < ke && c < nc) ? o.T[(long long)t * rp + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[8], b[4];
#pragma unroll
      for (int u = 0; u < 8; ++u) a[u] = Rs[kk * (NB + 1) + ty * 8 + u];
#pragma unroll
      for (int v = 0; v < 4; ++v) b[v] = Ts[kk * SLAB + tx * 4 + v];
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int u = 0; u < 8; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) Cs[(ty * 8 + u) * (SLAB + 1) + tx * 4 + v] = acc[u][v];
  for (int e = threadIdx.x; e < nb * nb; e += NT) {
    const int i = e / nb, u = e % nb;
    Tp[i * (NB + 1) + u] = o.T[(long long)(k0 + i) * rp + k0 + u];
  }
  __syncthreads();
  // T_pq[i][c] = -sum_{u >= i} T_pp[i][u] C[u][c]
#pragma unroll
  for (int u8 = 0; u8 < 8; ++u8) {
    const int i = ty * 8 + u8;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int c = tx * 4 + v;
      if (i < nb && c < nc) {
        float s = 0.f;
        for (int u = i; u < nb; ++u) s = fmaf(Tp[i * (NB + 1) + u], Cs[u * (SLAB + 1) + c], s);
        o.T[(long long)(k0 + i) * rp + c0 + c] = -s;
      }
    }
  }
}

}  // namespace bchol
}  // namespace dion
