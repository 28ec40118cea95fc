// Gram partials of orth() on the 5th-generation tensor core: for every job and
// every 256-row chunk of its argument A (rows x r, fp32),
//
//     gpart[chunk] = A[chunk rows]^T A[chunk rows]          (rp x rp, 3xTF32;
//                    row a holds its 16-column blocks from the one with column a on)
//
// the first step of each CholeskyQR pass (orth() = thin QR with a positive
// diagonal; junaidaliop.github.io "Orth-Dion", symbol glossary).  Both MMA
// operands are the same converted tile A^T (rows a, K = the chunk's rows): the
// converter warps transpose 32-row TMA boxes of A into the 128-byte-swizzled
// K-major layout and split them into tf32 halves.  One chunk is one TMEM
// accumulation (256 of K), so the tensor core's truncating accumulation stays
// within ~2e-6 relative; the partials are summed in round-to-nearest fp32 by
// the Cholesky kernel.
//
// Warp roles: 0 TMA producer, 1 TMEM allocator + MMA issuer, 2..9 converters
// (one operand row each) and the drain to global memory.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace tcgram {

using namespace dion::tc;

constexpr int BK = 32;                 // rows of A per chunk (the MMA K step)
constexpr int CHUNK_ROWS = 256;        // rows of A per partial (one TMEM accumulation)
constexpr int RP_MAX = 192;            // widest job handled here
constexpr int OPROWS = 256;            // operand rows (two M = 128 blocks, zero padded)
constexpr int OSTAGES = 2, SSTAGES = 2;
constexpr int NCONV = 8;
constexpr int NTHREADS = (2 + NCONV) * 32;
constexpr uint32_t TMEM_COLS = 512;    // block b of the Gram at columns [b * RP_MAX, b * RP_MAX + rp)

constexpr uint32_t OP_BYTES = OPROWS * BK * 4;          // 32 KB (hi or lo)
constexpr uint32_t OST_BYTES = 2 * OP_BYTES;             // 64 KB
constexpr uint32_t SST_BYTES = RP_MAX * BK * 4;          // 24 KB: rp / 32 boxes of 32 x 32
constexpr uint32_t SMEM_BYTES = 1024 + OSTAGES * OST_BYTES + SSTAGES * SST_BYTES + 512;

// One 256-row chunk `chunk` of job `job` (host-built table).
struct GItem {
  int job, chunk, pad0, pad1;
};

struct GJob {
  CUtensorMap mA;            // A (rows x rp fp32), box 32 (columns) x 32 (rows), 128-byte swizzle
  float* gpart;              // nchunk x rp x rp
  int rows, rp, nchunk;
  int pass;                  // CholeskyQR pass; pass 2 runs only for flagged jobs
  const unsigned* flag;
  unsigned* status;
  int pad[8];
};
static_assert(sizeof(GJob) % 64 == 0, "GJob must keep 64-byte alignment of its map");

__device__ __forceinline__ bool skip(const GJob& j) {
  return (*j.status & ST_FATAL) != 0 || (j.pass == 2 && !*j.flag);
}

__global__ void __launch_bounds__(NTHREADS, 1)
k_gram(const GJob* __restrict__ jobs, const GItem* __restrict__ items, int nitems) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* ost = smem;
  unsigned char* sst = smem + OSTAGES * OST_BYTES;
  uint64_t* bars = (uint64_t*)(sst + SSTAGES * SST_BYTES);
  uint64_t* o_full = bars;                 // NCONV converter arrivals
  uint64_t* o_empty = o_full + OSTAGES;    // MMA commit
  uint64_t* s_full = o_empty + OSTAGES;    // TMA bytes
  uint64_t* s_empty = s_full + SSTAGES;    // NCONV arrivals
  uint64_t* acc_full = s_empty + SSTAGES;  // MMA commit per item
  uint64_t* acc_empty = acc_full + 1;      // NCONV drain arrivals
  uint64_t* drain = acc_empty + 1;
  uint32_t* tslot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < OSTAGES; ++i) { mbar_init(&o_full[i], NCONV); mbar_init(&o_empty[i], 1); }
    for (int i = 0; i < SSTAGES; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], NCONV); }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, NCONV);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tslot, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  int failed = -1;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    int ss = 0; uint32_t sph = 0;
    uint32_t slast[SSTAGES] = {0, 0}; bool sused[SSTAGES] = {false, false};
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const int jb = items[t].job;
      const GJob& j = jobs[jb];
      if (skip(j)) continue;
      const int r0 = items[t].chunk * CHUNK_ROWS;
      const int nk = (min(j.rows - r0, CHUNK_ROWS) + BK - 1) / BK;
      const int nbox = j.rp / 32;
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait(&s_empty[ss], sph ^ 1, abort_flag)) { failed = jb; goto prod_done; }
        mbar_arrive_expect_tx(&s_full[ss], nbox * 4096);
        for (int b = 0; b < nbox; ++b)
          tma_load_2d(sst + ss * SST_BYTES + b * 4096, &j.mA, &s_full[ss], b * 32, r0 + kc * BK);
        sused[ss] = true; slast[ss] = sph;
        if (++ss == SSTAGES) { ss = 0; sph ^= 1; }
      }
    }
  prod_done:
    if (*abort_flag)
      for (int i = 0; i < SSTAGES; ++i) if (sused[i]) mbar_wait_drain(&s_full[i], slast[i]);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int os = 0; uint32_t oph = 0; uint32_t aph = 0;
    bool issued = false;
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const int jb = items[t].job;
      const GJob& j = jobs[jb];
      if (skip(j)) continue;
      const int r0 = items[t].chunk * CHUNK_ROWS;
      const int nk = (min(j.rows - r0, CHUNK_ROWS) + BK - 1) / BK;
      const int nblk = j.rp > 128 ? 2 : 1;
      const uint32_t idesc = idesc_tf32(128, j.rp);
      if (!mbar_wait(&acc_empty[0], aph ^ 1, abort_flag)) { failed = jb; goto mma_done; }
      tc_fence_after();
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait(&o_full[os], oph, abort_flag)) { failed = jb; goto mma_done; }
        tc_fence_after();
        const uint32_t hi = smem_u32(ost + os * OST_BYTES), lo = hi + OP_BYTES;
        for (int blk = 0; blk < nblk; ++blk) {
          const uint32_t d = tmem + blk * RP_MAX;
          const uint32_t ab = blk * 128 * 128;   // byte offset of operand row blk * 128
#pragma unroll
          for (int kk = 0; kk < BK / 8; ++kk) {
            const uint32_t o = kk * 32;
            mma_tf32(d, sdesc_k_sw128(lo + ab + o), sdesc_k_sw128(hi + o), idesc, (kc | kk) != 0);
            mma_tf32(d, sdesc_k_sw128(hi + ab + o), sdesc_k_sw128(lo + o), idesc, 1);
            mma_tf32(d, sdesc_k_sw128(hi + ab + o), sdesc_k_sw128(hi + o), idesc, 1);
          }
        }
        issued = true;
        mma_commit(&o_empty[os]);
        if (++os == OSTAGES) { os = 0; oph ^= 1; }
      }
      mma_commit(&acc_full[0]);
      aph ^= 1;
    }
  mma_done:
    if (*abort_flag && issued) { mma_commit(drain); mbar_wait_drain(drain, 0); }
  } else if (warp >= 2) {
    // ------------------------------------------------------------ converters + drain
    const int cw = warp - 2;                 // 0..7
    const int arow = cw * 32 + lane;         // operand row (a) converted by this thread
    const int quarter = warp & 3;            // TMEM lane quarter
    const int blk = cw >> 2;                 // Gram block drained by this warp
    int os = 0, ss = 0; uint32_t oph = 0, sph = 0; uint32_t aph = 0;
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const int jb = items[t].job;
      const GJob& j = jobs[jb];
      if (skip(j)) continue;
      const int ch = items[t].chunk;
      const int r0 = ch * CHUNK_ROWS;
      const int nk = (min(j.rows - r0, CHUNK_ROWS) + BK - 1) / BK;
      bool ok = true;
      for (int kc = 0; kc < nk; ++kc) {
        if (!mbar_wait_warp(&s_full[ss], sph, abort_flag)) { failed = jb; ok = false; break; }
        if (!mbar_wait_warp(&o_empty[os], oph ^ 1, abort_flag)) { failed = jb; ok = false; break; }
        const unsigned char* src = sst + ss * SST_BYTES;
        unsigned char* hp = ost + os * OST_BYTES;
        unsigned char* lp = hp + OP_BYTES;
        const bool live = arow < j.rp;
        const int bx = arow >> 5, ax = arow & 31;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          float4 h4 = make_float4(0.f, 0.f, 0.f, 0.f), l4 = h4;
          if (live) {
            float v[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = 4 * c + e;   // row of A within the chunk (K index)
              v[e] = *reinterpret_cast<const float*>(src + bx * 4096 + i * 128 + ((((ax >> 2) ^ i) & 7) << 4) +
                                                     ((ax & 3) << 2));
            }
            split_tf32(v[0], h4.x, l4.x);
            split_tf32(v[1], h4.y, l4.y);
            split_tf32(v[2], h4.z, l4.z);
            split_tf32(v[3], h4.w, l4.w);
          }
          const uint32_t off = sw128_off(arow, 4 * c);
          *reinterpret_cast<float4*>(hp + off) = h4;
          *reinterpret_cast<float4*>(lp + off) = l4;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_empty[ss]);
          mbar_arrive(&o_full[os]);
        }
        if (++ss == SSTAGES) { ss = 0; sph ^= 1; }
        if (++os == OSTAGES) { os = 0; oph ^= 1; }
      }
      if (!ok) break;
      // drain: warp (quarter, blk) holds Gram rows a = blk * 128 + quarter * 32 + lane
      if (!mbar_wait_warp(&acc_full[0], aph, abort_flag)) { failed = jb; break; }
      tc_fence_after();
      const int nblk = j.rp > 128 ? 2 : 1;
      if (blk < nblk) {
        const int a = blk * 128 + quarter * 32 + lane;
        float* dst = j.gpart + (long long)ch * j.rp * j.rp + (long long)a * j.rp;
        // the Gram is symmetric and its consumers read the upper triangle: only the
        // 16-column blocks that reach the diagonal or above are written (the warp's
        // first row decides which blocks it loads at all)
        const int a0 = blk * 128 + quarter * 32;
        for (int cb = a0 / 16; cb < j.rp / 16; ++cb) {
          float v[16];
          tmem_ld16(tmem + ((uint32_t)(quarter * 32) << 16) + blk * RP_MAX + cb * 16, v);
          tmem_wait_ld();
          if (a < j.rp && cb * 16 + 15 >= a) {
#pragma unroll
            for (int k = 0; k < 16; k += 4)
              *reinterpret_cast<float4*>(dst + cb * 16 + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[0]);
      aph ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, TMEM_COLS); }
  if (failed >= 0) atomicOr(jobs[failed].status, ST_TIMEOUT);
  // after an abort this CTA left items unfinished: every job it had items of is incomplete
  if (threadIdx.x == 0 && *abort_flag)
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) atomicOr(jobs[items[t].job].status, ST_TIMEOUT);
}

}  // namespace tcgram
}  // namespace dion
