// Split of fp32 factors into the two tf32 operands of a 3xTF32 tensor-core
// product: x = hi + lo + O(2^-22 |x|), both stored as fp32 bit patterns whose
// low 13 mantissa bits are zero.  Columns c >= cols of the padded output are
// written as zero so that the K padding of the tensor-core kernels adds nothing.
// A job with lo == nullptr is a plain padded copy (hi = x).
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace tcsplit {

constexpr int NT = 256;
constexpr int ELEMS_PER_CTA = 4096;

struct SplitJob {
  const float* src;
  long long lds;        // leading dimension of src (elements)
  float* hi;
  float* lo;
  long long ldd;        // leading dimension of hi / lo (= padded columns)
  long long rows, cols; // valid region of src
  const unsigned* status;
  int tiled;            // 1: hi / lo in the update's operand tile layout (optile_idx, ldd = rp)
};

__global__ void __launch_bounds__(NT) k_split(const SplitJob* __restrict__ jobs, const int* __restrict__ tstart,
                                              int njob) {
  const int j = find_job(tstart, njob, blockIdx.x);
  const SplitJob& o = jobs[j];
  if (*o.status & ST_FATAL) return;
  const long long total = o.rows * o.ldd;
  const long long base = (long long)(blockIdx.x - tstart[j]) * ELEMS_PER_CTA;
  for (int e = threadIdx.x; e < ELEMS_PER_CTA; e += NT) {
    const long long idx = base + e;
    if (idx >= total) break;
    const long long row = idx / o.ldd, c = idx % o.ldd;
    const float v = c < o.cols ? o.src[row * o.lds + c] : 0.f;
    if (!o.lo) {
      o.hi[idx] = v;
      continue;
    }
    float h, l;
    tc::split_tf32(v, h, l);
    const long long d = o.tiled ? optile_idx(row, c, o.ldd) : idx;
    o.hi[d] = h;
    o.lo[d] = l;
  }
}

// Transposed split: dst[c][r] = src[r][c] for r < rows, c < cols_pad (zero for
// c >= cols), as hi / lo tf32 halves with leading dimension ldd (>= rows).
// 32 x 32 tiles through shared memory so that reads and writes coalesce; a CTA
// takes TROWS / 32 tiles down one 32-column strip (a launch of one tile per CTA
// spent its time in CTA start-up).
constexpr int TROWS = 128;
struct TJob {
  const float* src;
  long long lds;
  float* hi;
  float* lo;
  long long ldd;
  long long rows, cols, cols_pad;
  const unsigned* status;
};

__global__ void __launch_bounds__(NT) k_tsplit(const TJob* __restrict__ jobs, const int* __restrict__ tstart,
                                               int njob) {
  __shared__ float t[32][33];
  const int j = find_job(tstart, njob, blockIdx.x);
  const TJob& o = jobs[j];
  if (*o.status & ST_FATAL) return;
  const long long ntc = (o.cols_pad + 31) / 32;
  const long long local = blockIdx.x - tstart[j];
  const long long c0 = (local % ntc) * 32;
  const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
  for (long long r0 = (local / ntc) * TROWS, r1 = r0 + TROWS; r0 < r1 && r0 < o.rows; r0 += 32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long r = r0 + ty + 8 * k, c = c0 + tx;
      t[ty + 8 * k][tx] = (r < o.rows && c < o.cols) ? o.src[r * o.lds + c] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const long long c = c0 + ty + 8 * k, r = r0 + tx;
      if (r < o.rows && c < o.cols_pad) {
        float h, l;
        tc::split_tf32(t[tx][ty + 8 * k], h, l);
        o.hi[c * o.ldd + r] = h;
        o.lo[c * o.ldd + r] = l;
      }
    }
    __syncthreads();
  }
}

}  // namespace tcsplit
}  // namespace dion
