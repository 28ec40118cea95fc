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

struct Group {
  long long m, n, k;       // shape and the side of the Gram (min(m, n))
  std::vector<int> mats;   // plan indices, in order
  size_t off_Y[2], off_A;  // workspace offsets
};

}  // namespace

struct muon_plan {
  std::vector<muon_matrix_desc> descs;
  int count = 0, iters = 0, precision = 0;
  std::vector<Group> groups;
  std::vector<int> ts;                 // block prefix sums of the streaming kernels
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
      for (int b = 0; b < 2; ++b)
        x.Y[b] = base + gr.off_Y[b] + k * (size_t)(d.m * d.n) * esize(p->precision);
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
  if (cudaMemcpyAsync(base + p->off_tables, p->image.data(), p->image.size(), cudaMemcpyHostToDevice, s) !=
      cudaSuccess)
    return cuda_err("muon table upload");
  p->uploaded_ws = base;
  return DION_OK;
}

}  // namespace

extern "C" {

dion_status_t muon_plan_create(const muon_matrix_desc* descs, int32_t count, int32_t ns_iters, int32_t precision,
                               size_t* workspace_bytes, muon_plan** out) {
  if (!descs || !workspace_bytes || !out) return dion_fail(DION_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (count < 1 || count > (1 << 20)) return dion_fail(DION_ERR_INVALID_ARG, "count %d outside [1, 2^20]", count);
  if (ns_iters < 0 || ns_iters > 1000) return dion_fail(DION_ERR_INVALID_ARG, "ns_iters %d outside [0, 1000]", ns_iters);
  if (precision < MUON_NS_BF16 || precision > MUON_NS_FP32)
    return dion_fail(DION_ERR_INVALID_ARG, "unknown precision %d", precision);
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
  }
  muon_plan* p = new muon_plan();
  p->descs.assign(descs, descs + count);
  p->count = count;
  p->iters = ns_iters;
  p->precision = precision;
  // groups of equal shape, in order of first appearance
  std::map<std::pair<long long, long long>, int> gid;
  for (int i = 0; i < count; ++i) {
    const auto key = std::make_pair((long long)descs[i].m, (long long)descs[i].n);
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
  for (int i = 0; i < count; ++i) p->ts[i + 1] = p->ts[i] + (int)cdiv(descs[i].m * descs[i].n, EPB);
  // tables
  size_t off = 0;
  auto take = [&](size_t b) { size_t o = off; off = align_up(off + b, 128); return o; };
  p->t_mats = take(sizeof(MuMat) * count);
  p->t_ts = take(sizeof(int) * (count + 1));
  p->tables_bytes = off;
  // workspace
  size_t ws = 0;
  auto region = [&](size_t b) { size_t o = ws; ws = align_up(ws + std::max<size_t>(b, 4), kAlign); return o; };
  p->off_tables = region(p->tables_bytes);
  p->off_norm = region(4 * (size_t)count);
  p->off_partial.resize(count);
  for (int i = 0; i < count; ++i) p->off_partial[i] = region(4 * (size_t)(p->ts[i + 1] - p->ts[i]));
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
  // momentum, norm, start, update; per iteration and group two GEMMs and the diagonal
  return 4 + plan->iters * 3 * (int)plan->groups.size();
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
  k_momentum<<<nblk, NT, 0, s>>>(mats, ts, p->count);
  k_norm<<<p->count, NT, 0, s>>>(mats);
  k_start<<<nblk, NT, 0, s>>>(mats, ts, p->count, bf16);
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
  k_update<<<nblk, NT, 0, s>>>(mats, ts, p->count, p->iters & 1, bf16);
  st = cuda_err("muon launch");
  if (st) return st;
  return dion_ok();
}

}  // extern "C"
