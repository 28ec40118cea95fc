// The Muon comparator (include/muon.h): momentum, Frobenius normalisation, the
// cubic Newton-Schulz iteration and the update, batched over every matrix of a
// plan.  The pages describe Muon as orthogonalising the momentum with a
// Newton-Schulz iteration of cubic cost (searcharxiv 2608.11612 "Dion3"
// abstract; the artiverse.ca post "What Made Muon Stand Out"); the momentum
// rule and the textbook cubic coefficients 1.5 / -0.5 are this library's
// reading.
//
// Per step:
//   k_momentum       B <- mu B + G, per-block partial sums of B^2       (HBM pass over G, B)
//   k_norm           1 / ||B||_F per matrix (partials summed in a fixed order)
//   k_start          Y_0 = B / ||B||_F into the group's Y buffer (bf16 or fp32)
//   per iteration, per group of equal shape (cuBLAS strided-batched GEMMs):
//     A  = -0.5 Y Y^T (m <= n)  or  -0.5 Y^T Y (m > n)                   Gram of the smaller side
//     k_add_diag     A <- A + 1.5 I
//     Y' = A Y  or  Y A                                                  (= 1.5 Y - 0.5 Y Y^T Y)
//   k_update         X <- X - eta s Y_K
//
// Row-selection variant (row_fraction < 1, the Dion3 reading in include/muon.h):
// k_rownorm (row norms of B, one warp per row, fixed order), k_select (per
// matrix: bitonic sort of (norm, row) in shared memory, the k largest rows in
// increasing row order, 1 / Frobenius norm of that block), k_gather (Y_0 = the
// selected rows / their norm), the same iteration on k x n blocks, and
// k_update_rows (only the selected rows of X).
#include "muon.h"

#include <cublas_v2.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <map>
#include <utility>
#include <vector>

#include "host_errors.h"

namespace {

constexpr int NT = 256;
constexpr int EPB = NT * 16;                  // elements per block of the streaming kernels
constexpr size_t kAlign = 256;
constexpr size_t kCublasWs = 32u << 20;       // cuBLAS GEMM scratch, taken from the workspace

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

struct MuMat {
  float* X;
  const void* G;
  float* B;
  long long m, n, ldx, ldg, ldb;
  long long kr;        // rows orthogonalised: m, or k of the row-selection variant
  int* sel;            // row-selection variant: the k selected rows, increasing
  float* rownorm;      // row-selection variant: sum of squares of each row of B
  void* Y[2];          // this matrix's slot in its group's ping-pong buffers (dense, ld n)
  float* partial;      // per-block partial sums of B^2
  float* inv_norm;     // 1 / ||B||_F
  int g_bf16;
  int nblk;
  float eta_s, mu;
};

// Largest j in [0, n) with start[j] <= t.
__device__ __forceinline__ int find_mat(const int* __restrict__ start, int n, int t) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (start[mid] <= t) lo = mid; else hi = mid;
  }
  return lo;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < NT / 32; ++w) t += red[w];
  return t;
}

// B <- mu B + G over one block of EPB elements; partial[block] = sum of the new B^2.
__global__ void __launch_bounds__(NT) k_momentum(const MuMat* __restrict__ mats, const int* __restrict__ ts, int nmat) {
  __shared__ float red[NT / 32];
  const int j = find_mat(ts, nmat, blockIdx.x);
  const MuMat& d = mats[j];
  const long long lb = blockIdx.x - ts[j];
  const long long tot = d.m * d.n;
  float sq = 0.f;
#pragma unroll 4
  for (int k = 0; k < EPB / NT; ++k) {
    const long long e = lb * EPB + (long long)k * NT + threadIdx.x;
    if (e < tot) {
      const long long r = e / d.n, c = e % d.n;
      const float g = d.g_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(d.G)[r * d.ldg + c])
                               : static_cast<const float*>(d.G)[r * d.ldg + c];
      float* bp = d.B + r * d.ldb + c;
      const float b = fmaf(d.mu, *bp, g);
      *bp = b;
      sq = fmaf(b, b, sq);
    }
  }
  const float t = block_sum(sq, red);
  if (threadIdx.x == 0) d.partial[lb] = t;
}

// inv_norm = 1 / sqrt(sum of the partials), summed in a fixed order (0 for a zero matrix).
__global__ void __launch_bounds__(NT) k_norm(const MuMat* __restrict__ mats) {
  __shared__ float red[NT / 32];
  const MuMat& d = mats[blockIdx.x];
  float s = 0.f;
  for (int i = threadIdx.x; i < d.nblk; i += NT) s += d.partial[i];
  const float t = block_sum(s, red);
  if (threadIdx.x == 0) *d.inv_norm = t > 0.f ? 1.f / sqrtf(t) : 0.f;
}

// Y_0 = B * inv_norm, stored dense (ld n) as bf16 or fp32.
__global__ void __launch_bounds__(NT) k_start(const MuMat* __restrict__ mats, const int* __restrict__ ts, int nmat,
                                              int bf16) {
  const int j = find_mat(ts, nmat, blockIdx.x);
  const MuMat& d = mats[j];
  const long long lb = blockIdx.x - ts[j];
  const long long tot = d.m * d.n;
  const float s = *d.inv_norm;
#pragma unroll 4
  for (int k = 0; k < EPB / NT; ++k) {
    const long long e = lb * EPB + (long long)k * NT + threadIdx.x;
    if (e < tot) {
      const float y = d.B[(e / d.n) * d.ldb + e % d.n] * s;
      if (bf16) static_cast<__nv_bfloat16*>(d.Y[0])[e] = __float2bfloat16_rn(y);
      else static_cast<float*>(d.Y[0])[e] = y;
    }
  }
}

// A <- A + v I for `count` dense k x k matrices stored back to back.
__global__ void k_add_diag(void* A, long long k, long long count, float v, int bf16) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= k * count) return;
  const long long idx = (i / k) * k * k + (i % k) * (k + 1);
  if (bf16) {
    __nv_bfloat16* a = static_cast<__nv_bfloat16*>(A) + idx;
    *a = __float2bfloat16_rn(__bfloat162float(*a) + v);
  } else {
    static_cast<float*>(A)[idx] += v;
  }
}

// X <- X - eta s Y_K.
__global__ void __launch_bounds__(NT) k_update(const MuMat* __restrict__ mats, const int* __restrict__ ts, int nmat,
                                               int which, int bf16) {
  const int j = find_mat(ts, nmat, blockIdx.x);
  const MuMat& d = mats[j];
  const long long lb = blockIdx.x - ts[j];
  const long long tot = d.m * d.n;
#pragma unroll 4
  for (int k = 0; k < EPB / NT; ++k) {
    const long long e = lb * EPB + (long long)k * NT + threadIdx.x;
    if (e < tot) {
      const float y = bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(d.Y[which])[e])
                           : static_cast<const float*>(d.Y[which])[e];
      float* xp = d.X + (e / d.n) * d.ldx + e % d.n;
      *xp = fmaf(-d.eta_s, y, *xp);
    }
  }
}

// Sum of squares of every row of every B (one warp per row, fixed order).
__global__ void __launch_bounds__(NT) k_rownorm(const MuMat* __restrict__ mats, const int* __restrict__ rs, int nmat,
                                                long long total_rows) {
  const long long w = ((long long)blockIdx.x * NT + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= total_rows) return;
  const int j = find_mat(rs, nmat, (int)w);
  const MuMat& d = mats[j];
  const long long row = w - rs[j];
  const float* b = d.B + row * d.ldb;
  float s = 0.f;
  for (long long c = lane; c < d.n; c += 32) s = fmaf(b[c], b[c], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) d.rownorm[row] = s;
}

// One CTA per matrix: the kr rows with the largest norms (ties: lower row first)
// by a bitonic sort of (norm, row) in shared memory, written in increasing row
// order to sel; inv_norm = 1 / sqrt(sum of their squares), summed in row order.
constexpr int SEL_NT = 1024;
__global__ void __launch_bounds__(SEL_NT) k_select(const MuMat* __restrict__ mats) {
  extern __shared__ unsigned char sm[];
  const MuMat& d = mats[blockIdx.x];
  int P = 1;
  while (P < d.m) P <<= 1;
  float* key = reinterpret_cast<float*>(sm);
  int* idx = reinterpret_cast<int*>(sm + 4 * (size_t)P);
  for (int i = threadIdx.x; i < P; i += SEL_NT) {
    key[i] = i < d.m ? d.rownorm[i] : -1.f;
    idx[i] = i;
  }
  __syncthreads();
  // descending by key, ascending by row on ties
  for (int k = 2; k <= P; k <<= 1)
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < P; i += SEL_NT) {
        const int l = i ^ jj;
        if (l > i) {
          const bool first_before = key[i] > key[l] || (key[i] == key[l] && idx[i] < idx[l]);
          const bool up = (i & k) == 0;
          if (up != first_before) {
            const float tk = key[i]; key[i] = key[l]; key[l] = tk;
            const int ti = idx[i]; idx[i] = idx[l]; idx[l] = ti;
          }
        }
      }
      __syncthreads();
    }
  // the first kr rows, now sorted by row index
  const int kr = (int)d.kr;
  int Q = 1;
  while (Q < kr) Q <<= 1;
  for (int i = kr + threadIdx.x; i < Q; i += SEL_NT) idx[i] = 0x7fffffff;
  __syncthreads();
  for (int k = 2; k <= Q; k <<= 1)
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int i = threadIdx.x; i < Q; i += SEL_NT) {
        const int l = i ^ jj;
        if (l > i) {
          const bool up = (i & k) == 0;
          if (up == (idx[i] > idx[l])) { const int t = idx[i]; idx[i] = idx[l]; idx[l] = t; }
        }
      }
      __syncthreads();
    }
  __shared__ float red[SEL_NT / 32];
  float acc = 0.f;
  for (int i = threadIdx.x; i < kr; i += SEL_NT) {
    d.sel[i] = idx[i];
    acc += d.rownorm[idx[i]];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < SEL_NT / 32; ++w) t += red[w];
    *d.inv_norm = t > 0.f ? 1.f / sqrtf(t) : 0.f;
  }
}

// Y_0 = the selected rows of B * inv_norm (kr x n, dense).
__global__ void __launch_bounds__(NT) k_gather(const MuMat* __restrict__ mats, const int* __restrict__ ts, int nmat,
                                               int bf16) {
  const int j = find_mat(ts, nmat, blockIdx.x);
  const MuMat& d = mats[j];
  const long long lb = blockIdx.x - ts[j];
  const long long tot = d.kr * d.n;
  const float s = *d.inv_norm;
  for (int k = 0; k < EPB / NT; ++k) {
    const long long e = lb * EPB + (long long)k * NT + threadIdx.x;
    if (e < tot) {
      const float y = d.B[(long long)d.sel[e / d.n] * d.ldb + e % d.n] * s;
      if (bf16) static_cast<__nv_bfloat16*>(d.Y[0])[e] = __float2bfloat16_rn(y);
      else static_cast<float*>(d.Y[0])[e] = y;
    }
  }
}

// X[sel[i], :] <- X[sel[i], :] - eta s Y_K[i, :].
__global__ void __launch_bounds__(NT) k_update_rows(const MuMat* __restrict__ mats, const int* __restrict__ ts,
                                                    int nmat, int which, int bf16) {
  const int j = find_mat(ts, nmat, blockIdx.x);
  const MuMat& d = mats[j];
  const long long lb = blockIdx.x - ts[j];
  const long long tot = d.kr * d.n;
  for (int k = 0; k < EPB / NT; ++k) {
    const long long e = lb * EPB + (long long)k * NT + threadIdx.x;
    if (e < tot) {
      const float y = bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(d.Y[which])[e])
                           : static_cast<const float*>(d.Y[which])[e];
      float* xp = d.X + (long long)d.sel[e / d.n] * d.ldx + e % d.n;
      *xp = fmaf(-d.eta_s, y, *xp);
    }
  }
}

struct Group {
  long long m, n, k;       // shape of the orthogonalised block (kr x n) and the side of its Gram
  std::vector<int> mats;   // plan indices, in order
  size_t off_Y[2], off_A;  // workspace offsets
};

}  // namespace

struct muon_plan {
  std::vector<muon_matrix_desc> descs;
  int count = 0, iters = 0, precision = 0;
  float row_fraction = 1.f;
  bool select = false;                 // row-selection variant
  std::vector<long long> kr;           // rows orthogonalised per matrix
  std::vector<Group> groups;
  std::vector<int> ts;                 // block prefix sums of the streaming kernels (m x n)
  std::vector<int> ts_sel;             // ... over the selected blocks (kr x n)
  std::vector<int> rs;                 // row prefix sums (k_rownorm)
  std::vector<size_t> off_sel, off_rownorm;
  size_t t_ts_sel = 0, t_rs = 0;
  int max_rows = 0;
  std::vector<size_t> off_partial;
  size_t off_tables = 0, off_norm = 0, off_cublas = 0, ws_bytes = 0;
  size_t t_mats = 0, t_ts = 0, tables_bytes = 0;
  std::vector<unsigned char> image;
  const void* uploaded_ws = nullptr;
  cublasHandle_t handle = nullptr;
};

namespace {

dion_status_t cuda_err(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return dion_fail(DION_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DION_OK;
}

size_t esize(int precision) { return precision == MUON_NS_BF16 ? 2 : 4; }

dion_status_t upload(muon_plan* p, unsigned char* base, cudaStream_t s) {
  std::vector<MuMat> mats(p->count);
  for (int g = 0; g < (int)p->groups.size(); ++g) {
    const Group& gr = p->groups[g];
    for (size_t k = 0; k < gr.mats.size(); ++k) {
      const int i = gr.mats[k];
      const auto& d = p->descs[i];
      MuMat& x = mats[i];
      x.X = d.X; x.G = d.G; x.B = d.B;
      x.m = d.m; x.n = d.n; x.ldx = d.ld_x; x.ldg = d.ld_g; x.ldb = d.ld_b;
      x.kr = p->kr[i];
      x.sel = p->select ? reinterpret_cast<int*>(base + p->off_sel[i]) : nullptr;
      x.rownorm = p->select ? reinterpret_cast<float*>(base + p->off_rownorm[i]) : nullptr;
      for (int b = 0; b < 2; ++b)
        x.Y[b] = base + gr.off_Y[b] + k * (size_t)(x.kr * d.n) * esize(p->precision);
      x.partial = reinterpret_cast<float*>(base + p->off_partial[i]);
      x.inv_norm = reinterpret_cast<float*>(base + p->off_norm) + i;
      x.g_bf16 = d.g_dtype == DION_DTYPE_BF16;
      x.nblk = p->ts[i + 1] - p->ts[i];
      const float sc = d.scale > 0.f ? d.scale : (float)std::sqrt((double)d.m / (double)d.n);
      x.eta_s = d.eta * sc;
      x.mu = d.mu;
    }
  }
  p->image.assign(p->tables_bytes, 0);
  std::memcpy(p->image.data() + p->t_mats, mats.data(), sizeof(MuMat) * mats.size());
  std::memcpy(p->image.data() + p->t_ts, p->ts.data(), sizeof(int) * p->ts.size());
  std::memcpy(p->image.data() + p->t_ts_sel, p->ts_sel.data(), sizeof(int) * p->ts_sel.size());
  std::memcpy(p->image.data() + p->t_rs, p->rs.data(), sizeof(int) * p->rs.size());
  if (cudaMemcpyAsync(base + p->off_tables, p->image.data(), p->image.size(), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return cuda_err("muon table upload");
  p->uploaded_ws = base;
  return DION_OK;
}

}  // namespace

extern "C" {

dion_status_t muon_plan_create(const muon_matrix_desc* descs, int32_t count, int32_t ns_iters, int32_t precision,
                               float row_fraction, size_t* workspace_bytes, muon_plan** out) {
  if (!descs || !workspace_bytes || !out) return dion_fail(DION_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (count < 1 || count > (1 << 20)) return dion_fail(DION_ERR_INVALID_ARG, "count %d outside [1, 2^20]", count);
  if (ns_iters < 0 || ns_iters > 1000) return dion_fail(DION_ERR_INVALID_ARG, "ns_iters %d outside [0, 1000]", ns_iters);
  if (precision < MUON_NS_BF16 || precision > MUON_NS_FP32)
    return dion_fail(DION_ERR_INVALID_ARG, "unknown precision %d", precision);
  if (!(row_fraction > 0.f && row_fraction <= 1.f))
    return dion_fail(DION_ERR_INVALID_ARG, "row_fraction %g outside (0, 1]", (double)row_fraction);
  long long rows_total = 0;
  for (int i = 0; i < count; ++i) {
    const muon_matrix_desc& d = descs[i];
    if (!d.X || !d.G || !d.B) return dion_fail(DION_ERR_INVALID_ARG, "matrix %d: NULL pointer", i);
    if (d.m < 1 || d.n < 1 || d.m >= (1LL << 31) || d.n >= (1LL << 31))
      return dion_fail(DION_ERR_INVALID_ARG, "matrix %d: bad shape", i);
    if (d.ld_x < d.n || d.ld_g < d.n || d.ld_b < d.n)
      return dion_fail(DION_ERR_INVALID_ARG, "matrix %d: leading dimension below n", i);
    if (d.g_dtype != DION_DTYPE_F32 && d.g_dtype != DION_DTYPE_BF16)
      return dion_fail(DION_ERR_INVALID_ARG, "matrix %d: unknown g_dtype", i);
    if (!std::isfinite(d.eta) || !std::isfinite(d.mu) || !std::isfinite(d.scale))
      return dion_fail(DION_ERR_INVALID_ARG, "matrix %d: non-finite eta / mu / scale", i);
    if (row_fraction < 1.f && d.m > DION3_MAX_ROWS)
      return dion_fail(DION_ERR_UNSUPPORTED, "matrix %d: row selection needs m <= %d", i, DION3_MAX_ROWS);
    rows_total += d.m;
  }
  if (rows_total >= (1LL << 31)) return dion_fail(DION_ERR_UNSUPPORTED, "more than 2^31 rows in one plan");
  muon_plan* p = new muon_plan();
  p->descs.assign(descs, descs + count);
  p->count = count;
  p->iters = ns_iters;
  p->precision = precision;
  p->row_fraction = row_fraction;
  p->select = row_fraction < 1.f;
  p->kr.resize(count);
  for (int i = 0; i < count; ++i) {
    const long long m = descs[i].m;
    p->kr[i] = p->select ? std::min<long long>(m, std::max<long long>(1, (long long)std::ceil((double)row_fraction * m)))
                         : m;
    p->max_rows = std::max<int>(p->max_rows, (int)m);
  }
  // groups of equal orthogonalised shape (kr x n), in order of first appearance
  std::map<std::pair<long long, long long>, int> gid;
  for (int i = 0; i < count; ++i) {
    const auto key = std::make_pair(p->kr[i], (long long)descs[i].n);
    auto it = gid.find(key);
    if (it == gid.end()) {
      gid[key] = (int)p->groups.size();
      Group g;
      g.m = key.first; g.n = key.second; g.k = std::min(key.first, key.second);
      p->groups.push_back(g);
      it = gid.find(key);
    }
    p->groups[it->second].mats.push_back(i);
  }
  p->ts.assign(count + 1, 0);
  p->ts_sel.assign(count + 1, 0);
  p->rs.assign(count + 1, 0);
  for (int i = 0; i < count; ++i) {
    p->ts[i + 1] = p->ts[i] + (int)cdiv(descs[i].m * descs[i].n, EPB);
    p->ts_sel[i + 1] = p->ts_sel[i] + (int)cdiv(p->kr[i] * descs[i].n, EPB);
    p->rs[i + 1] = p->rs[i] + (int)descs[i].m;
  }
  // tables
  size_t off = 0;
  auto take = [&](size_t b) { size_t o = off; off = align_up(off + b, 128); return o; };
  p->t_mats = take(sizeof(MuMat) * count);
  p->t_ts = take(sizeof(int) * (count + 1));
  p->t_ts_sel = take(sizeof(int) * (count + 1));
  p->t_rs = take(sizeof(int) * (count + 1));
  p->tables_bytes = off;
  // workspace
  size_t ws = 0;
  auto region = [&](size_t b) { size_t o = ws; ws = align_up(ws + std::max<size_t>(b, 4), kAlign); return o; };
  p->off_tables = region(p->tables_bytes);
  p->off_norm = region(4 * (size_t)count);
  p->off_partial.resize(count);
  for (int i = 0; i < count; ++i) p->off_partial[i] = region(4 * (size_t)(p->ts[i + 1] - p->ts[i]));
  if (p->select) {
    p->off_sel.resize(count);
    p->off_rownorm.resize(count);
    for (int i = 0; i < count; ++i) {
      p->off_sel[i] = region(4 * (size_t)p->kr[i]);
      p->off_rownorm[i] = region(4 * (size_t)descs[i].m);
    }
  }
  const size_t es = esize(precision);
  for (Group& g : p->groups) {
    const size_t c = g.mats.size();
    g.off_Y[0] = region(c * (size_t)(g.m * g.n) * es);
    g.off_Y[1] = region(c * (size_t)(g.m * g.n) * es);
    g.off_A = region(c * (size_t)(g.k * g.k) * es);
  }
  p->off_cublas = region(kCublasWs);
  p->ws_bytes = ws;
  *workspace_bytes = ws;
  *out = p;
  return dion_ok();
}

void muon_plan_destroy(muon_plan* plan) {
  if (!plan) return;
  if (plan->handle) cublasDestroy(plan->handle);
  delete plan;
}

int32_t muon_plan_launches_per_step(const muon_plan* plan) {
  if (!plan) return -1;
  // momentum, norm, start, update (row selection: momentum, row norms, select, gather,
  // update); per iteration and group two GEMMs and the diagonal
  return (plan->select ? 5 : 4) + plan->iters * 3 * (int)plan->groups.size();
}

dion_status_t muon_plan_selected_rows(const muon_plan* plan, int32_t idx, size_t* byte_offset, int64_t* k) {
  if (!plan || !byte_offset || !k) return dion_fail(DION_ERR_INVALID_ARG, "NULL argument");
  if (!plan->select) return dion_fail(DION_ERR_INVALID_ARG, "the plan selects no rows (row_fraction = 1)");
  if (idx < 0 || idx >= plan->count) return dion_fail(DION_ERR_INVALID_ARG, "index %d outside the plan", idx);
  *byte_offset = plan->off_sel[idx];
  *k = plan->kr[idx];
  return dion_ok();
}

dion_status_t muon_step_batched(muon_plan* p, void* workspace, size_t ws_bytes, void* stream) {
  if (!p) return dion_fail(DION_ERR_INVALID_ARG, "NULL plan");
  if (!workspace || (uintptr_t)workspace % kAlign) return dion_fail(DION_ERR_WORKSPACE, "workspace NULL or misaligned");
  if (ws_bytes < p->ws_bytes)
    return dion_fail(DION_ERR_WORKSPACE, "workspace of %zu bytes, plan needs %zu", ws_bytes, p->ws_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  if (!p->handle) {
    if (cublasCreate(&p->handle) != CUBLAS_STATUS_SUCCESS) return dion_fail(DION_ERR_CUDA, "cublasCreate failed");
    if (p->select && cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, 8 * DION3_MAX_ROWS) !=
                         cudaSuccess)
      return cuda_err("kernel attributes");
  }
  if (p->uploaded_ws != workspace) {
    const dion_status_t st = upload(p, base, s);
    if (st) return st;
  }
  if (cublasSetStream(p->handle, s) != CUBLAS_STATUS_SUCCESS ||
      cublasSetWorkspace(p->handle, base + p->off_cublas, kCublasWs) != CUBLAS_STATUS_SUCCESS)
    return dion_fail(DION_ERR_CUDA, "cuBLAS stream / workspace");
  const MuMat* mats = reinterpret_cast<const MuMat*>(base + p->off_tables + p->t_mats);
  const int* ts = reinterpret_cast<const int*>(base + p->off_tables + p->t_ts);
  const int nblk = p->ts[p->count];
  const int bf16 = p->precision == MUON_NS_BF16;
  const int* ts_sel = reinterpret_cast<const int*>(base + p->off_tables + p->t_ts_sel);
  k_momentum<<<nblk, NT, 0, s>>>(mats, ts, p->count);
  if (p->select) {
    const long long rows = p->rs[p->count];
    k_rownorm<<<(int)cdiv(rows * 32, NT), NT, 0, s>>>(
        mats, reinterpret_cast<const int*>(base + p->off_tables + p->t_rs), p->count, rows);
    int P = 1;
    while (P < p->max_rows) P <<= 1;
    k_select<<<p->count, SEL_NT, 8 * (size_t)P, s>>>(mats);
    k_gather<<<p->ts_sel[p->count], NT, 0, s>>>(mats, ts_sel, p->count, bf16);
  } else {
    k_norm<<<p->count, NT, 0, s>>>(mats);
    k_start<<<nblk, NT, 0, s>>>(mats, ts, p->count, bf16);
  }
  dion_status_t st = cuda_err("muon launch");
  if (st) return st;
  const cudaDataType_t dt = bf16 ? CUDA_R_16BF : CUDA_R_32F;
  const cublasComputeType_t ct = p->precision == MUON_NS_TF32 ? CUBLAS_COMPUTE_32F_FAST_TF32 : CUBLAS_COMPUTE_32F;
  const float alpha_g = -0.5f, one = 1.f, zero = 0.f;
  for (int it = 0; it < p->iters; ++it) {
    for (const Group& g : p->groups) {
      const int c = (int)g.mats.size();
      void* Y = base + g.off_Y[it & 1];
      void* Yn = base + g.off_Y[(it + 1) & 1];
      void* A = base + g.off_A;
      const long long m = g.m, n = g.n, k = g.k;
      const long long sY = m * n, sA = k * k;
      // Row-major Y (m x n) is column-major Yc = Y^T (n x m, ld n).
      cublasStatus_t r1, r2;
      if (m <= n) {
        // A = -0.5 Y Y^T = -0.5 Yc^T Yc (m x m);  Y' = A Y, i.e. Y'c = Yc A
        r1 = cublasGemmStridedBatchedEx(p->handle, CUBLAS_OP_T, CUBLAS_OP_N, (int)k, (int)k, (int)n, &alpha_g, Y, dt,
                                        (int)n, sY, Y, dt, (int)n, sY, &zero, A, dt, (int)k, sA, c, ct,
                                        CUBLAS_GEMM_DEFAULT);
        k_add_diag<<<(int)cdiv(k * c, NT), NT, 0, s>>>(A, k, c, 1.5f, bf16);
        r2 = cublasGemmStridedBatchedEx(p->handle, CUBLAS_OP_N, CUBLAS_OP_N, (int)n, (int)m, (int)m, &one, Y, dt,
                                        (int)n, sY, A, dt, (int)k, sA, &zero, Yn, dt, (int)n, sY, c, ct,
                                        CUBLAS_GEMM_DEFAULT);
      } else {
        // A = -0.5 Y^T Y = -0.5 Yc Yc^T (n x n);  Y' = Y A, i.e. Y'c = A Yc
        r1 = cublasGemmStridedBatchedEx(p->handle, CUBLAS_OP_N, CUBLAS_OP_T, (int)k, (int)k, (int)m, &alpha_g, Y, dt,
                                        (int)n, sY, Y, dt, (int)n, sY, &zero, A, dt, (int)k, sA, c, ct,
                                        CUBLAS_GEMM_DEFAULT);
        k_add_diag<<<(int)cdiv(k * c, NT), NT, 0, s>>>(A, k, c, 1.5f, bf16);
        r2 = cublasGemmStridedBatchedEx(p->handle, CUBLAS_OP_N, CUBLAS_OP_N, (int)n, (int)m, (int)n, &one, A, dt,
                                        (int)k, sA, Y, dt, (int)n, sY, &zero, Yn, dt, (int)n, sY, c, ct,
                                        CUBLAS_GEMM_DEFAULT);
      }
      if (r1 != CUBLAS_STATUS_SUCCESS || r2 != CUBLAS_STATUS_SUCCESS)
        return dion_fail(DION_ERR_CUDA, "cuBLAS GEMM failed (%d, %d)", (int)r1, (int)r2);
    }
  }
  if (p->select)
    k_update_rows<<<p->ts_sel[p->count], NT, 0, s>>>(mats, ts_sel, p->count, p->iters & 1, bf16);
  else
    k_update<<<nblk, NT, 0, s>>>(mats, ts, p->count, p->iters & 1, bf16);
  st = cuda_err("muon launch");
  if (st) return st;
  return dion_ok();
}

}  // extern "C"
