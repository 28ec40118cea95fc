// CUDA-core kernels of the step: the small, latency-bound pieces that do not
// map to tensor-core tiles, each a grouped launch over all matrices (or orth
// jobs) of a plan.  fp32 storage, fp32 accumulation in a fixed order, so
// results are bitwise reproducible run to run.
//
// Kernel map (junaidaliop.github.io "Orth-Dion", update equations and glossary):
//   k_gram          partial Grams A^T A of a row chunk   orth() (the plan path for r > 192, and
//   k_trmm          Q = A T  (T upper triangular)        dion_orth_noalloc)
//   k_gram_reduce   sum of the Gram partials             orth(), tensor-core path
//   k_chol_inv      Cholesky + inverse, one CTA per job  orth(), positive diagonal, shifted pass
//   k_wreduce       W = sum of the K-range partials      equation 3 (and its tf32 halves)
//   k_colnorm       Vbar = W diag(1/||w_j||)             Dion right factor
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace simt {

constexpr int TM = 64, TN = 64, TK = 16, NT = 256;
constexpr int LDS = TM + 4;  // padded shared row

// acc[u][v] += sum_{k in [kb, ke)} A(i0 + ty*4 + u, k) * B(k, j0 + tx*4 + v)
// A_KC: consecutive threads walk k when loading A (A is k-contiguous in memory);
// B_JC: consecutive threads walk j when loading B.
template <bool A_KC, bool B_JC, class LA, class LB>
__device__ __forceinline__ void tile_acc(const LA& la, const LB& lb, long long i0, long long j0,
                                         long long kb, long long ke, float (&acc)[4][4],
                                         float* As, float* Bs) {
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  for (long long k0 = kb; k0 < ke; k0 += TK) {
#pragma unroll
    for (int e = 0; e < (TM * TK) / NT; ++e) {
      const int idx = tid + e * NT;
      const int ii = A_KC ? idx / TK : idx % TM;
      const int kk = A_KC ? idx % TK : idx / TM;
      const long long k = k0 + kk;
      As[kk * LDS + ii] = (k < ke) ? la(i0 + ii, k) : 0.f;
    }
#pragma unroll
    for (int e = 0; e < (TN * TK) / NT; ++e) {
      const int idx = tid + e * NT;
      const int jj = B_JC ? idx % TN : idx / TK;
      const int kk = B_JC ? idx / TN : idx % TK;
      const long long k = k0 + kk;
      Bs[kk * LDS + jj] = (k < ke) ? lb(k, j0 + jj) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) a[u] = As[kk * LDS + ty * 4 + u];
#pragma unroll
      for (int v = 0; v < 4; ++v) b[v] = Bs[kk * LDS + tx * 4 + v];
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) acc[u][v] = fmaf(a[u], b[v], acc[u][v]);
    }
    __syncthreads();
  }
}

// Row-major fp32 loader with bounds: element (i, k) of a rows x cols array.
struct LoadRM {
  const float* p; long long ld, rows, cols;
  __device__ float operator()(long long i, long long k) const {
    return (i < rows && k < cols) ? p[i * ld + k] : 0.f;
  }
};
// Transposed view: element (i, k) = p[k][i].
struct LoadRMT {
  const float* p; long long ld, rows, cols;  // rows/cols of the stored array
  __device__ float operator()(long long i, long long k) const {
    return (k < rows && i < cols) ? p[k * ld + i] : 0.f;
  }
};
__device__ __forceinline__ void zero(float (&acc)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) acc[u][v] = 0.f;
}

// ---------------------------------------------------------------- orth()
// Partial Gram of one row chunk: gpart[chunk][a][b] = sum_i A[i][a] A[i][b].
// pass 0 reads the job's input A, pass 1 its first-pass factor Q.
__global__ void __launch_bounds__(NT) k_gram(const OrthJob* __restrict__ jobs,
                                             const int* __restrict__ tstart, int njob, int pass) {
  __shared__ float As[TK * LDS], Bs[TK * LDS];
  const int j = find_job(tstart, njob, blockIdx.x);
  const OrthJob& o = jobs[j];
  if (*o.status & ST_FATAL) return;
  if (pass == 2 && !*o.flag) return;
  const int local = blockIdx.x - tstart[j];
  const int nt = (int)((o.rp + TN - 1) / TN);
  const int chunk = local / (nt * nt), rem = local % (nt * nt);
  const long long a0 = (long long)(rem / nt) * TM, b0 = (long long)(rem % nt) * TN;
  const float* A = pass == 0 ? o.A : (pass == 1 ? o.Q : o.Q2);
  const long long lda = pass == 0 ? o.lda : o.rp;
  const long long ib = (long long)chunk * o.chunk;
  const long long ie = ib + o.chunk < o.rows ? ib + o.chunk : o.rows;
  float acc[4][4];
  zero(acc);
  LoadRMT la{A, lda, o.rows, o.r};   // (a, i) = A[i][a]
  LoadRM lb{A, lda, o.rows, o.r};    // (i, b) = A[i][b]
  tile_acc<false, true>(la, lb, a0, b0, ib, ie, acc, As, Bs);
  float* out = o.gpart + (long long)chunk * o.rp * o.rp;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long a = a0 + ty * 4 + u;
    if (a >= o.rp) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const long long b = b0 + tx * 4 + v;
      if (b < o.rp) out[a * o.rp + b] = acc[u][v];
    }
  }
}

// One CTA per job: S = sum of the Gram partials (fixed order), upper Cholesky
// S = Rc^T Rc with a positive diagonal, T = Rc^{-1} (upper triangular, zero
// elsewhere, rp x rp).  S lives in shared memory when it fits (sm != 0), else
// in the job's global scratch.
//
// Pass 0 is where conditioning is decided.  CholeskyQR2 in fp32 needs
// kappa(A) well below u^{-1/2} ~ 4e3; when the unshifted factorisation breaks
// down or its pivots imply kappa(A) > ~1e3 (min pivot^2 < 1e-6 max diagonal),
// the Gram is rebuilt with the shift s = 11 (rows r + r (r + 1)) u ||A||_F^2 of
// shifted CholeskyQR (Fukaya, Kannan, Nakatsukasa, Yamamoto, Yanagisawa 2020) and
// the job is flagged for a third pass.  Every factor stays upper triangular
// with a positive diagonal, so the final Q is still the unique thin-QR factor.
// A failure in pass 1 or 2 (or of the shifted pass) marks the matrix and
// leaves it unchanged.
constexpr int CHOL_NT = 512;
constexpr int CHOL_SMEM_MAX = 200 * 1024;

// Sum of the Gram partials of every job, in a fixed order, into gsum (gsum =
// sum_c gpart[c], on the upper triangle's 16-column blocks); one thread per Gram
// element over the whole GPU, four partials in flight per thread.
constexpr int GRED_ELEMS = 1024;
__global__ void __launch_bounds__(256) k_gram_reduce(const OrthJob* __restrict__ jobs,
                                                     const int* __restrict__ tstart, int njob, int pass) {
  const int j = find_job(tstart, njob, blockIdx.x);
  const OrthJob& o = jobs[j];
  if (*o.status & ST_FATAL) return;
  if (pass == 2 && !*o.flag) return;
  const long long rp2 = o.rp * o.rp;
  for (int e = threadIdx.x; e < GRED_ELEMS; e += blockDim.x) {
    const long long idx = (long long)(blockIdx.x - tstart[j]) * GRED_ELEMS + e;
    if (idx >= rp2) break;
    // the partials hold, and the consumers read, the 16-column blocks of row a
    // from the one with column a on (the upper triangle with a margin)
    const long long ra = idx / o.rp, cb = (idx % o.rp) / 16;
    if (cb * 16 + 15 < ra) continue;
    const float* g = o.gpart + idx;
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
    int c = 0;
    for (; c + 4 <= o.nchunk; c += 4) {
      s0 += g[(long long)c * rp2];
      s1 += g[(long long)(c + 1) * rp2];
      s2 += g[(long long)(c + 2) * rp2];
      s3 += g[(long long)(c + 3) * rp2];
    }
    for (; c < o.nchunk; ++c) s0 += g[(long long)c * rp2];
    o.gsum[idx] = (s0 + s1) + (s2 + s3);
  }
}

// The job's Gram into S (r x lds): the reduced sum gsum when `reduced`, else the
// sum of its nchunk partials.
__device__ void chol_load(const OrthJob& o, int reduced, float* S, int lds, float shift, float* s_trace) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int r = o.r, rp = o.rp;
  float tr = 0.f;
  for (int e = tid; e < r * r; e += nth) {
    const int a = e / r, b = e % r;
    float v = 0.f;
    if (reduced) v = o.gsum[a * rp + b];
    else
      for (int c = 0; c < o.nchunk; ++c) v += o.gpart[(long long)c * rp * rp + a * rp + b];
    if (a == b) { tr += v; v += shift; }
    S[a * lds + b] = v;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tr += __shfl_xor_sync(0xffffffffu, tr, off);
  if ((tid & 31) == 0) s_trace[tid >> 5] = tr;
  __syncthreads();
}

// Storage of the factorisation in the r x lds array S: Rc (upper triangular,
// S = Rc^T Rc) in the upper triangle, T = Rc^{-1} (upper triangular) transposed
// into the strict lower triangle (T[a][c] at S[c][a], a < c), diag(T) in tdiag.
__device__ __forceinline__ float Rv(const float* S, int lds, int r, int a, int b) {
  return (a <= b && b < r) ? S[a * lds + b] : 0.f;
}
__device__ __forceinline__ float Tv(const float* S, int lds, const float* tdiag, int r, int a,
                                    int c) {
  if (c >= r) return 0.f;
  return a < c ? S[c * lds + a] : (a == c ? tdiag[a] : 0.f);
}

// In-place upper Cholesky, blocked right-looking with 32-wide panels.  Per panel:
// one warp factors the diagonal block in registers (lane l holds column l) and
// inverts it (T_pp = Rc_pp^{-1}); the row panel is Rc_pc = T_pp^T S_pc (a
// product, no substitution chain); the trailing matrix takes a rank-32 update.
// Returns 0 or the status bits of a failure; *s_min / *s_max receive the
// smallest squared pivot and the largest diagonal.  `scratch` holds 32 * r floats.
__device__ int chol_factor(float* S, int lds, int r, float* tdiag, float* scratch, int* s_bad,
                           float* s_min, float* s_max) {
  const int tid = threadIdx.x, nth = blockDim.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 0) {
    float mx = 0.f;
    for (int j = lane; j < r; j += 32) mx = fmaxf(mx, S[j * lds + j]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) { *s_max = mx; *s_bad = 0; *s_min = INFINITY; }
  }
  __syncthreads();
  for (int k0 = 0; k0 < r; k0 += 32) {
    const int nb = (int)min(32, r - k0);
    // (1) diagonal block, one warp: col[i] = S[k0 + i][k0 + lane] for i <= lane
    if (warp == 0) {
      float col[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) col[i] = (i <= lane && lane < nb) ? S[(k0 + i) * lds + k0 + lane] : 0.f;
      int bad = 0;
      float mn = INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j < nb && !bad) {
          const float d = __shfl_sync(0xffffffffu, col[j], j);
          if (!isfinite(d)) bad = (int)(ST_BREAKDOWN | ST_NONFINITE);
          else if (!(d > 0.f)) bad = (int)ST_BREAKDOWN;
          if (!bad) {
            mn = fminf(mn, d);
            const float piv = sqrtf(d);
            if (lane == j) col[j] = piv;
            else if (lane > j) col[j] = col[j] / piv;          // Rc[j][lane]
#pragma unroll
            for (int i = j + 1; i < 32; ++i) {
              const float rji = __shfl_sync(0xffffffffu, col[j], i);   // Rc[j][i]
              if (lane >= i) col[i] = fmaf(-rji, col[j], col[i]);
            }
          }
        }
      }
      if (lane == 0) { *s_bad = bad; *s_min = fminf(*s_min, mn); }
      if (!bad) {
        // T_pp = Rc_pp^{-1}, column `lane`: t[i] = T_pp[i][lane]
        float t[32];
#pragma unroll
        for (int i = 31; i >= 0; --i) {
          const float rii = __shfl_sync(0xffffffffu, col[i], i);
          float sum = 0.f;
#pragma unroll
          for (int k = i + 1; k < 32; ++k) {
            const float rik = __shfl_sync(0xffffffffu, col[i], k);   // Rc[i][k]
            if (k <= lane) sum = fmaf(rik, t[k], sum);
          }
          t[i] = i == lane ? 1.f / rii : (i < lane ? -sum / rii : 0.f);
        }
        if (lane < nb) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i <= lane) S[(k0 + i) * lds + k0 + lane] = col[i];     // Rc (upper, with the diagonal)
            if (i < lane) S[(k0 + lane) * lds + k0 + i] = t[i];        // T (lower, transposed)
            if (i == lane) tdiag[k0 + lane] = t[i];
          }
        }
      }
    }
    __syncthreads();
    if (*s_bad) return *s_bad;
    const int c0 = k0 + nb;
    if (c0 >= r) break;
    const int n2 = r - c0;
    // (2) row panel Rc[k0 + i][c] = sum_{t <= i} T_pp[t][i] S[k0 + t][c], via scratch
    for (int e = tid; e < nb * n2; e += nth) {
      const int i = e / n2, c = c0 + e % n2;
      float y = 0.f;
      for (int t = 0; t <= i; ++t) y = fmaf(Tv(S, lds, tdiag, r, k0 + t, k0 + i), S[(k0 + t) * lds + c], y);
      scratch[e] = y;
    }
    __syncthreads();
    for (int e = tid; e < nb * n2; e += nth) {
      const int i = e / n2, c = c0 + e % n2;
      S[(k0 + i) * lds + c] = scratch[e];
    }
    __syncthreads();
    // (3) trailing update of the upper triangle: S[a][c] -= sum_i Rc[k0 + i][a] Rc[k0 + i][c]
    for (int e = tid; e < n2 * n2; e += nth) {
      const int a = c0 + e / n2, c = c0 + e % n2;
      if (a > c) continue;
      float v = S[a * lds + c];
#pragma unroll 8
      for (int i = 0; i < nb; ++i) v = fmaf(-S[(k0 + i) * lds + a], S[(k0 + i) * lds + c], v);
      S[a * lds + c] = v;
    }
    __syncthreads();
  }
  return 0;
}

// Off-diagonal blocks of T = Rc^{-1}, by block diagonals d = q - p:
//   T_pq = -T_pp (sum_{k = p+1..q} Rc_pk T_kq),
// with the diagonal blocks T_pp already in place.  `scratch` holds 32 * r floats.
__device__ void inverse_blocks(float* S, int lds, int r, float* tdiag, float* scratch) {
  const int tid = threadIdx.x, nth = blockDim.x;
  const int np = (int)((r + 31) / 32);
  for (int d = 1; d < np; ++d) {
    const int nout = (int)(np - d) * 1024;
    for (int e = tid; e < nout; e += nth) {
      const int p = (int)(e >> 10), i = (int)((e >> 5) & 31), j = (int)(e & 31), q = p + d;
      const int a = 32 * p + i, c = 32 * q + j;
      float sum = 0.f;
      for (int kk = 32 * (p + 1); kk < min(r, 32 * (q + 1)); ++kk)
        sum = fmaf(Rv(S, lds, r, a, kk), Tv(S, lds, tdiag, r, kk, c), sum);
      scratch[e] = sum;   // C_pq[i][j]
    }
    __syncthreads();
    for (int e = tid; e < nout; e += nth) {
      const int p = (int)(e >> 10), i = (int)((e >> 5) & 31), j = (int)(e & 31), q = p + d;
      const int a = 32 * p + i, c = 32 * q + j;
      if (a >= r || c >= r) continue;
      float sum = 0.f;
      for (int t = i; t < 32; ++t) sum = fmaf(Tv(S, lds, tdiag, r, a, 32 * p + t), scratch[(p << 10) + t * 32 + j], sum);
      S[c * lds + a] = -sum;
    }
    __syncthreads();
  }
}

// order (optional): job of each CTA, largest rank first, so that the big jobs
// share the first wave of CTAs.
template <bool SMEM>
__global__ void __launch_bounds__(CHOL_NT, 1) k_chol_inv(const OrthJob* __restrict__ jobs, int pass, int reduced,
                                                        const int* __restrict__ order) {
  extern __shared__ float sm_dyn[];
  const OrthJob& o = jobs[order ? order[blockIdx.x] : blockIdx.x];
  __shared__ int s_bad;
  __shared__ float s_min, s_max;
  __shared__ float s_trace[CHOL_NT / 32];
  if (*o.status & ST_FATAL) return;
  if (pass == 2 && !*o.flag) return;
  const int tid = threadIdx.x, nth = blockDim.x;
  const int r = o.r, rp = o.rp;
  // shared (or the job's global scratch): S r x lds, tdiag r, scratch 32 r
  float* S = SMEM ? sm_dyn : o.S;
  const int lds = SMEM ? r + 1 : rp;
  float* tdiag = S + r * lds;
  float* scratch = tdiag + r;
  chol_load(o, reduced, S, lds, 0.f, s_trace);
  int bad = chol_factor(S, lds, r, tdiag, scratch, &s_bad, &s_min, &s_max);
  if (pass == 0 && (bad || s_min < 1e-6f * s_max)) {
    float trace = 0.f;
    for (int w = 0; w < nth / 32; ++w) trace += s_trace[w];
    const float shift = 11.f * ((float)o.rows * (float)r + (float)r * (float)(r + 1)) * 5.9604645e-8f * trace;
    __syncthreads();
    chol_load(o, reduced, S, lds, shift, s_trace);
    bad = chol_factor(S, lds, r, tdiag, scratch, &s_bad, &s_min, &s_max);
    if (!bad && tid == 0) { *o.flag = 1u; atomicOr(o.status, ST_SHIFTED); }
  }
  if (bad) {
    if (tid == 0) atomicOr(o.status, (unsigned)bad);
    return;
  }
  inverse_blocks(S, lds, r, tdiag, scratch);
  // outputs: T^T split for the tensor core (row c of T^T = column c of T), or T
  if (o.Tt_hi) {
    for (int e = tid; e < rp * rp; e += nth) {
      const int c = e / rp, a = e % rp;
      float h, l;
      tc::split_tf32(a < r ? Tv(S, lds, tdiag, r, a, c) : 0.f, h, l);
      o.Tt_hi[e] = h;
      o.Tt_lo[e] = l;
    }
  } else {
    for (int e = tid; e < rp * rp; e += nth) {
      const int a = e / rp, c = e % rp;
      o.T[e] = a < r ? Tv(S, lds, tdiag, r, a, c) : 0.f;
    }
  }
}

// out = A T with T upper triangular (rp x rp), one CholeskyQR pass.
__global__ void __launch_bounds__(NT) k_trmm(const OrthJob* __restrict__ jobs,
                                             const int* __restrict__ tstart, int njob, int pass) {
  __shared__ float As[TK * LDS], Bs[TK * LDS];
  const int j = find_job(tstart, njob, blockIdx.x);
  const OrthJob& o = jobs[j];
  if (*o.status & ST_FATAL) return;
  const bool three = *o.flag != 0;
  if (pass == 2 && !three) return;
  const int local = blockIdx.x - tstart[j];
  const int ntc = (int)((o.rp + TN - 1) / TN);
  const long long i0 = (long long)(local / ntc) * TM, c0 = (long long)(local % ntc) * TN;
  const float* A = pass == 0 ? o.A : (pass == 1 ? o.Q : o.Q2);
  const long long lda = pass == 0 ? o.lda : o.rp;
  float acc[4][4];
  zero(acc);
  LoadRM la{A, lda, o.rows, o.r};
  LoadRM lb{o.T, o.rp, o.rp, o.rp};
  const long long ke = (c0 + TN < o.r) ? c0 + TN : o.r;
  tile_acc<true, true>(la, lb, i0, c0, 0, ke, acc, As, Bs);
  // pass 0 -> Q; pass 1 -> the result, or Q2 when a third pass follows; pass 2 -> the result
  const bool final_pass = pass == 2 || (pass == 1 && !three);
  float* out = final_pass ? o.out : (pass == 0 ? o.Q : o.Q2);
  const long long ldo = final_pass ? o.ldo : o.rp;
  const long long ncol = final_pass ? o.out_cols : o.rp;
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const long long i = i0 + ty * 4 + u;
    if (i >= o.rows) continue;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const long long c = c0 + tx * 4 + v;
      if (c < ncol) out[i * ldo + c] = acc[u][v];
    }
  }
}

// ---------------------------------------------------------------- phase (c)
// W = sum over splits (fixed order), with its tf32 halves for the update;
// one CTA covers 1024 elements.
__global__ void __launch_bounds__(NT) k_wreduce(const MatDev* __restrict__ mats,
                                                const int* __restrict__ tstart, int nmat) {
  const int j = find_job(tstart, nmat, blockIdx.x);
  const MatDev& d = mats[j];
  if ((*d.status & ST_FATAL) || d.ksplit <= 1) return;
  const long long base = (long long)(blockIdx.x - tstart[j]) * 1024;
  const long long tot = d.n * d.rp;
  for (int e = threadIdx.x; e < 1024; e += NT) {
    const long long idx = base + e;
    if (idx >= tot) break;
    float s = 0.f;
    for (int sp = 0; sp < d.ksplit; ++sp) s += d.Wpart[(long long)sp * tot + idx];
    d.W[idx] = s;
    float h, l;
    tc::split_tf32(idx % d.rp < d.r ? s : 0.f, h, l);
    const long long o = optile_idx(idx / d.rp, idx % d.rp, d.rp);   // the update's tile layout
    d.Wh[o] = h;
    d.Wl[o] = l;
  }
}

// ---------------------------------------------------------------- phase (d), Dion
// Vbar[:, c] = W[:, c] / ||W[:, c]||, 32 columns per CTA; a zero column stays zero.
__global__ void __launch_bounds__(NT) k_colnorm(const MatDev* __restrict__ mats,
                                                const int* __restrict__ tstart,
                                                const int* __restrict__ idx, int nidx) {
  __shared__ float part[NT / 32][33];
  __shared__ float scale[32];
  const int jj = find_job(tstart, nidx, blockIdx.x);
  const MatDev& d = mats[idx[jj]];
  if (*d.status & ST_FATAL) return;
  const long long c = (long long)(blockIdx.x - tstart[jj]) * 32 + (threadIdx.x & 31);
  const int w = threadIdx.x >> 5;
  float s = 0.f;
  if (c < d.r)
    for (long long row = w; row < d.n; row += NT / 32) {
      const float x = d.W[row * d.rp + c];
      s = fmaf(x, x, s);
    }
  part[w][threadIdx.x & 31] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float t = 0.f;
    for (int k = 0; k < NT / 32; ++k) t += part[k][threadIdx.x];
    scale[threadIdx.x] = t > 0.f ? 1.f / sqrtf(t) : 0.f;
  }
  __syncthreads();
  if (c < d.r) {
    const float sc = scale[threadIdx.x & 31];
    for (long long row = w; row < d.n; row += NT / 32) d.V[row * d.r + c] = d.W[row * d.rp + c] * sc;
  }
}

}  // namespace simt
}  // namespace dion
