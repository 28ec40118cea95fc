// Phases (a) and (c) on the 5th-generation tensor core: the two streaming
// contractions with the error-feedback buffer M = G + R (junaidaliop.github.io
// "Orth-Dion", update equations for U and W):
//
//     (a)  P = M V       rows i of M, K = n      (TRANS = false)
//     (c)  W = M^T U     rows j of M^T, K = m    (TRANS = true, K split over CTAs)
//
// M is never stored: every CTA streams G and R tiles by TMA into a staging
// ring, and 16 converter warps form M = G + R in fp32, split it into the two
// tf32 halves of a 3xTF32 product and store them in tensor memory (one thread
// per operand row, i.e. per TMEM lane; for M^T a thread gathers one column of the
// staged rows), where the MMA reads its A operand.  A from TMEM keeps the
// operand halves out of shared memory: the tensor core's operand reads from
// shared memory, three products per K step, were what bounded this kernel.  The
// second operand (V^T or U^T, already split) comes in by TMA.  Chunks of 16 along K
// keep four operand stages and eight staging slots in flight.  The same kernel
// runs the A T products of orth(); its final pass also writes the tf32 halves
// of the result for the next tensor-core kernels.
//
// The tensor core's fp32 accumulation truncates: its bias grows with the
// number of accumulation steps (measured -1e-5 relative per 1024 of K).  So a
// tile accumulates at most 256 of K in TMEM (a "slice", 2 TMEM buffers) and the
// converter warps, between conversions, add finished slices into registers in
// round-to-nearest fp32; the bias then stays near 2e-6.
//
// Warp roles: 0 TMA producer of the staged G / R tiles, 1 TMEM allocator + MMA
// issuer, 2..17 converters (four groups of four, alternating chunks) and slice
// drain, 18 TMA producer of the B operand halves.  The two producers run
// independently, so a full operand ring never holds back the HBM loads of the
// staging ring (and the other way round).  One CTA per SM, persistent over
// (row tile, K range, column block) items of every matrix.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace tcstream {

using namespace dion::tc;

constexpr int BM = 128;              // output rows per tile (TMEM lanes)
constexpr int BK = 16;               // K per chunk: one 64-byte swizzle row of fp32
constexpr int SLICE = 16;            // chunks per TMEM slice (256 of K)
constexpr int OSTAGES = 4;           // operand stages (A hi/lo in TMEM by the converters, B by TMA)
constexpr int SSTAGES = 8;           // staging slots of G and R (HBM latency)
constexpr int NCONV = 16;            // converter / drain warps: four groups of four
constexpr int NGROUP = 4;            // converter groups; group g converts the chunks numbered g (mod 4)
constexpr int BWARP = 2 + NCONV;      // warp of the B-operand producer
constexpr int NTHREADS = (3 + NCONV) * 32;
constexpr int BN_MAX = 192;          // widest column block (TMEM: 2 x 192 <= 512)
constexpr int QMAX = BN_MAX / 4;     // accumulator columns per converter thread (one column quarter)
constexpr uint32_t TMEM_COLS = 512;
// TMEM columns: accumulator slices at [0, 2 BN_MAX), then per operand stage the A
// halves (hi: BK columns, lo: BK columns)
constexpr uint32_t TMEM_A = 2 * BN_MAX;
static_assert(TMEM_A + OSTAGES * 2 * BK <= TMEM_COLS, "accumulators and A stages fit in TMEM");

constexpr uint32_t B_BYTES_MAX = BN_MAX * BK * 4;        // 12 KB
constexpr uint32_t OST_BYTES = 2 * B_BYTES_MAX;          // 24 KB: B hi | B lo
constexpr uint32_t SST_BYTES = 16384;                    // staging slot: G (<= 8 KB) | R (8 KB)
constexpr uint32_t SST_R = 8192;                         // offset of the R tile in a slot
constexpr uint32_t SMEM_BYTES = 1024 + OSTAGES * OST_BYTES + SSTAGES * SST_BYTES + 512;
// Converter group g waits on the chunks numbered g mod NGROUP only.  mbarrier
// parity waits are exact only when a waiter sees every phase of the barrier it
// waits on, so every stage and slot must belong to a single group: chunk numbers
// map to stages and slots modulo a multiple of NGROUP.
static_assert(OSTAGES % NGROUP == 0 && SSTAGES % NGROUP == 0, "stages must be owned by one converter group");

// gmode: what the staged tiles hold.  G_BF16 / G_F32: M = G + R (phases a, c);
// G_NONE: a single fp32 matrix in the R slot (the A T product of orth()).
enum { G_NONE = 0, G_BF16 = 1, G_F32 = 2 };

struct SJob {
  CUtensorMap mG, mR, mBh, mBl;   // G, R (staging boxes); B operand hi / lo (box 32 x bn)
  float* out;                     // P (a), W or its partials (c), or the final result of orth()
  long long ld_out;               // leading dimension of out
  long long split_stride;         // elements between the K-range partials of out
  float* q1;                      // orth(): pass-0 result (ld rp)
  float* q2;                      // orth(): pass-1 result of a three-pass job (ld rp)
  const unsigned* flag;           // orth(): three-pass flag of the job
  int pass;                       // orth(): CholeskyQR pass 0..2; -1 for phases (a), (c) and a
                                  // Gram of pass 0 / 1, -2 for the Gram of a third pass
  int out_cols;                   // columns of out to write (rp, or r for Vbar into V)
  int rows;                       // output rows: m (a) or n (c), rows of A (orth)
  int kdim;                       // K extent: n (a), m (c), rp (orth)
  int ksplit, kchunk;             // K ranges (multiple of BK)
  int ncb, bn;                    // column blocks of width bn (multiple of 32, <= BN_MAX)
  int rp, gmode;
  unsigned* status;
  // tf32 halves of the final result for the tensor-core kernels that read it next
  // (null: none): in the update's operand tile layout (optile_idx with rp), and
  // (th / tl) transposed with leading dimension ld_t; columns hcols..rp-1 are
  // written as zero
  float* sh;
  float* sl;
  float* th;
  float* tl;
  long long ld_t;
  int hcols;
  float mu;                       // M = G + mu R: 1 for Dion / Orth-Dion, the momentum coefficient otherwise
  int tr_fin, tr_inter;           // write th / tl for the final result, for an intermediate factor
};
static_assert(sizeof(SJob) % 64 == 0, "SJob must keep 64-byte alignment of its maps");

// One work item (host-built table, heaviest first): output rows row0..row0+127 of
// job `job`, K range [k0, k0 + 16 nk) (partial `ks`), output columns from c0.
struct Item {
  int job, row0, ks, c0, k0, nk, pad0, pad1;
};

// pass 2 (an A T job) and pass -2 (the Gram of a third CholeskyQR pass) run only for
// jobs whose first pass took the shifted branch
__device__ __forceinline__ bool skip(const SJob& j) {
  return (*j.status & ST_FATAL) != 0 || ((j.pass == 2 || j.pass == -2) && !*j.flag);
}

// Drain one finished TMEM slice (columns [col0, col0 + quarter) of this
// thread's lane, a multiple of 8) into the register accumulator: two batches of
// three 8-column loads, one wait each (a wait per load cost a TMEM round trip per
// 8 columns; the wait names the loaded registers so that no add moves above it).
__device__ __forceinline__ void drain_add(uint32_t taddr, int quarter, float (&acc)[QMAX]) {
  static_assert(QMAX % 24 == 0, "batches of three 8-column loads");
#pragma unroll
  for (int h = 0; h < QMAX / 24; ++h) {
    if (h * 24 < quarter) {
      float v0[8], v1[8], v2[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) { v0[k] = 0.f; v1[k] = 0.f; v2[k] = 0.f; }
      tmem_ld8(taddr + h * 24, v0);
      if (h * 24 + 8 < quarter) tmem_ld8(taddr + h * 24 + 8, v1);
      if (h * 24 + 16 < quarter) tmem_ld8(taddr + h * 24 + 16, v2);
      tmem_wait_ld_dep(v0, v1, v2);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[h * 24 + k] += v0[k];
        acc[h * 24 + 8 + k] += v1[k];
        acc[h * 24 + 16 + k] += v2[k];
      }
    }
  }
}

template <bool TRANS>
__global__ void __launch_bounds__(NTHREADS, 1)
k_stream(const SJob* __restrict__ jobs, const Item* __restrict__ items, int nitems) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* ost = smem;
  unsigned char* sst = smem + OSTAGES * OST_BYTES;
  uint64_t* bars = (uint64_t*)(sst + SSTAGES * SST_BYTES);
  uint64_t* o_full = bars;                 // B bytes (TMA) + NCONV / NGROUP converter arrivals
  uint64_t* o_empty = o_full + OSTAGES;    // MMA commit
  uint64_t* s_full = o_empty + OSTAGES;    // staging bytes (TMA)
  uint64_t* s_empty = s_full + SSTAGES;    // NCONV / NGROUP converter arrivals
  uint64_t* acc_full = s_empty + SSTAGES;  // MMA commit per slice
  uint64_t* acc_empty = acc_full + 2;      // NCONV drain arrivals
  uint64_t* drain = acc_empty + 2;
  uint32_t* tslot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // a chunk is converted by one group of NCONV / NGROUP warps
    for (int i = 0; i < OSTAGES; ++i) { mbar_init(&o_full[i], 1 + NCONV / NGROUP); mbar_init(&o_empty[i], 1); }
    for (int i = 0; i < SSTAGES; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], NCONV / NGROUP); }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], NCONV); }
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
    // ------------------------------------------------------------ TMA producer: staged G / R
    int ss = 0; uint32_t sph = 0;
    uint32_t slast[SSTAGES];
    bool sused[SSTAGES];
    for (int i = 0; i < SSTAGES; ++i) { slast[i] = 0; sused[i] = false; }
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const Item it = items[t];
      const SJob& j = jobs[it.job];
      if (skip(j)) continue;
      const uint32_t gbytes = j.gmode == G_NONE ? 0u : BM * BK * (j.gmode == G_BF16 ? 2 : 4);
      for (int kc = 0; kc < it.nk; ++kc) {
        const int k = it.k0 + kc * BK;
        // staging: G and R tiles of M
        if (!mbar_wait(&s_empty[ss], sph ^ 1, abort_flag)) { failed = it.job; goto prod_done; }
        mbar_arrive_expect_tx(&s_full[ss], gbytes + BM * BK * 4);
        {
          unsigned char* gdst = sst + ss * SST_BYTES;
          unsigned char* rdst = gdst + SST_R;
          if (!TRANS) {
            if (j.gmode != G_NONE) tma_load_2d(gdst, &j.mG, &s_full[ss], k, it.row0);
            tma_load_2d(rdst, &j.mR, &s_full[ss], k, it.row0);
          } else {
            // rows k..k+15 of M, columns row0..row0+127, in boxes of 128 bytes per row
            if (j.gmode != G_NONE) {
              const int gbox = j.gmode == G_BF16 ? 64 : 32;
              for (int b = 0; b < BM / gbox; ++b)
                tma_load_2d(gdst + b * 2048, &j.mG, &s_full[ss], it.row0 + b * gbox, k);
            }
            for (int b = 0; b < BM / 32; ++b)
              tma_load_2d(rdst + b * 2048, &j.mR, &s_full[ss], it.row0 + b * 32, k);
          }
        }
        sused[ss] = true; slast[ss] = sph;
        if (++ss == SSTAGES) { ss = 0; sph ^= 1; }
      }
    }
  prod_done:
    if (*abort_flag)
      for (int i = 0; i < SSTAGES; ++i) if (sused[i]) mbar_wait_drain(&s_full[i], slast[i]);
  } else if (warp == BWARP && lane == 0) {
    // ------------------------------------------------------------ TMA producer: B operand halves
    int os = 0; uint32_t oph = 0;
    uint32_t olast[OSTAGES];
    bool oused[OSTAGES];
    for (int i = 0; i < OSTAGES; ++i) { olast[i] = 0; oused[i] = false; }
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const Item it = items[t];
      const SJob& j = jobs[it.job];
      if (skip(j)) continue;
      const uint32_t bbytes = j.bn * BK * 4;
      for (int kc = 0; kc < it.nk; ++kc) {
        const int k = it.k0 + kc * BK;
        // operand stage: the B half (already split), bn rows
        if (!mbar_wait(&o_empty[os], oph ^ 1, abort_flag)) { failed = it.job; goto bprod_done; }
        mbar_arrive_expect_tx(&o_full[os], 2 * bbytes);
        unsigned char* b = ost + os * OST_BYTES;
        tma_load_2d(b, &j.mBh, &o_full[os], k, it.c0);
        tma_load_2d(b + B_BYTES_MAX, &j.mBl, &o_full[os], k, it.c0);
        oused[os] = true; olast[os] = oph;
        if (++os == OSTAGES) { os = 0; oph ^= 1; }
      }
    }
  bprod_done:
    if (*abort_flag)
      for (int i = 0; i < OSTAGES; ++i) if (oused[i]) mbar_wait_drain(&o_full[i], olast[i]);
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    int os = 0; uint32_t oph = 0; int b = 0; uint32_t aph[2] = {0, 0};
    bool issued = false;
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const Item it = items[t];
      const SJob& j = jobs[it.job];
      if (skip(j)) continue;
      const uint32_t idesc = idesc_tf32(BM, j.bn);
      for (int kc = 0; kc < it.nk; ++kc) {
        if (kc % SLICE == 0) {
          if (!mbar_wait(&acc_empty[b], aph[b] ^ 1, abort_flag)) { failed = it.job; goto mma_done; }
          tc_fence_after();
        }
        if (!mbar_wait(&o_full[os], oph, abort_flag)) { failed = it.job; goto mma_done; }
        tc_fence_after();
        const uint32_t d = tmem + b * BN_MAX;
        const uint32_t ah = tmem + TMEM_A + os * 2 * BK, al = ah + BK;   // A halves in TMEM (columns)
        const uint32_t bh = smem_u32(ost + os * OST_BYTES), bl = bh + B_BYTES_MAX;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint32_t o = kk * 32;        // B: 8 fp32 of K = 32 bytes; A: 8 columns
          mma_tf32_ts(d, al + kk * 8, sdesc_k_sw64(bh + o), idesc, ((kc % SLICE) | kk) != 0);
          mma_tf32_ts(d, ah + kk * 8, sdesc_k_sw64(bl + o), idesc, 1);
          mma_tf32_ts(d, ah + kk * 8, sdesc_k_sw64(bh + o), idesc, 1);
        }
        issued = true;
        mma_commit(&o_empty[os]);
        if (++os == OSTAGES) { os = 0; oph ^= 1; }
        if (kc % SLICE == SLICE - 1 || kc == it.nk - 1) {
          mma_commit(&acc_full[b]);
          aph[b] ^= 1; b ^= 1;
        }
      }
    }
  mma_done:
    if (*abort_flag && issued) { mma_commit(drain); mbar_wait_drain(drain, 0); }
  } else if (warp >= 2 && warp < BWARP) {
    // ------------------------------------------------------------ converters + slice drain
    // Four groups of four warps; group g converts the chunks whose sequence number
    // is g mod 4, so four chunks are in conversion at once.  For the drain every
    // warp owns TMEM lane quarter (warp % 4) and column quarter g.
    const int cw = warp - 2;                 // 0..15
    const int quarter = warp & 3;            // TMEM lane quarter of this warp
    const int g = cw >> 2;                   // converter group; column quarter for the drain
    const int row = quarter * 32 + lane;     // output row within the tile (TMEM lane)
    uint32_t seq = (uint32_t)g;              // sequence number of this group's next chunk
    int b = 0; uint32_t aph[2] = {0, 0};
    uint32_t base_seq = 0;                   // sequence number of the current item's first chunk
    float acc[QMAX];
    for (int t = blockIdx.x; t < nitems; t += gridDim.x) {
      const Item it = items[t];
      const SJob& j = jobs[it.job];
      if (skip(j)) continue;
      const int qw = j.bn >> 2;              // columns per quarter
      const int nslices = (it.nk + SLICE - 1) / SLICE;
      int drained = 0;
#pragma unroll
      for (int k = 0; k < QMAX; ++k) acc[k] = 0.f;
      bool ok = true;
      for (; ok && seq < base_seq + (uint32_t)it.nk; seq += NGROUP) {
        const int kc = (int)(seq - base_seq);
        // before converting a chunk of slice s, fold every slice up to s - 2 into the registers
        while (drained < kc / SLICE - 1) {
          if (!mbar_wait_warp(&acc_full[b], aph[b], abort_flag)) { failed = it.job; ok = false; break; }
          tc_fence_after();
          drain_add(tmem + ((uint32_t)(quarter * 32) << 16) + b * BN_MAX + g * qw, qw, acc);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[b]);
          aph[b] ^= 1; b ^= 1; ++drained;
        }
        if (!ok) break;
        const int ss = (int)(seq % SSTAGES), os = (int)(seq % OSTAGES);
        const uint32_t sph = (seq / SSTAGES) & 1u, oph = (seq / OSTAGES) & 1u;
        if (!mbar_wait_warp(&s_full[ss], sph, abort_flag)) { failed = it.job; ok = false; break; }
        if (!mbar_wait_warp(&o_empty[os], oph ^ 1, abort_flag)) { failed = it.job; ok = false; break; }
        const unsigned char* gsrc = sst + ss * SST_BYTES;
        const unsigned char* rsrc = gsrc + SST_R;
        const float mu = j.mu;                // M = G + mu R (mu = 1: the error-feedback buffer)
        float mv[16];                         // this thread's operand row: 16 of K
        if (!TRANS) {
          // row `row` of M, the chunk's 16 K elements (64-byte rows, 64-byte swizzle)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 r = *reinterpret_cast<const float4*>(rsrc + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
            mv[4 * c] = r.x; mv[4 * c + 1] = r.y; mv[4 * c + 2] = r.z; mv[4 * c + 3] = r.w;
          }
          if (j.gmode == G_BF16) {
            // 32-byte rows, 32-byte swizzle: 8 bf16 per 16-byte chunk
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const uint4 v = *reinterpret_cast<const uint4*>(gsrc + row * 32 + ((c ^ ((row >> 2) & 1)) << 4));
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                mv[8 * c + 2 * k] = fmaf(mu, mv[8 * c + 2 * k], __uint_as_float(w[k] << 16));
                mv[8 * c + 2 * k + 1] = fmaf(mu, mv[8 * c + 2 * k + 1], __uint_as_float(w[k] & 0xFFFF0000u));
              }
            }
          } else if (j.gmode == G_F32) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const float4 gv = *reinterpret_cast<const float4*>(gsrc + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
              mv[4 * c] = fmaf(mu, mv[4 * c], gv.x);
              mv[4 * c + 1] = fmaf(mu, mv[4 * c + 1], gv.y);
              mv[4 * c + 2] = fmaf(mu, mv[4 * c + 2], gv.z);
              mv[4 * c + 3] = fmaf(mu, mv[4 * c + 3], gv.w);
            }
          }
        } else {
          // column `row` of M (row of the M^T operand), the chunk's 16 rows of M as K:
          // scalar loads walk one staged row across the warp (conflict-free)
          const int jb = row >> 5, jj = row & 31;
#pragma unroll
          for (int i = 0; i < 16; ++i)
            mv[i] = *reinterpret_cast<const float*>(rsrc + jb * 2048 + i * 128 + ((((jj >> 2) ^ i) & 7) << 4) +
                                                    ((jj & 3) << 2));
          if (j.gmode == G_BF16) {
            const int gb = row >> 6, gj = row & 63;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const uint16_t gv = *reinterpret_cast<const uint16_t*>(
                  gsrc + gb * 2048 + i * 128 + ((((gj >> 3) ^ i) & 7) << 4) + ((gj & 7) << 1));
              mv[i] = fmaf(mu, mv[i], __uint_as_float((uint32_t)gv << 16));
            }
          } else if (j.gmode == G_F32) {
#pragma unroll
            for (int i = 0; i < 16; ++i)
              mv[i] = fmaf(mu, mv[i],
                           *reinterpret_cast<const float*>(gsrc + jb * 2048 + i * 128 + ((((jj >> 2) ^ i) & 7) << 4) +
                                                           ((jj & 3) << 2)));
          }
        }
        // the tf32 halves into this stage's TMEM columns, lane `row` (the warp's own
        // lane quarter); the MMA that last read these columns has completed (o_empty)
        {
          float hv[16], lv[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) split_tf32(mv[k], hv[k], lv[k]);
          tc_fence_after();
          const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16) + TMEM_A + os * 2 * BK;
          tmem_st16(ta, hv);
          tmem_st16(ta + BK, lv);
          tmem_wait_st();
          tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&s_empty[ss]);
          mbar_arrive(&o_full[os]);
        }
      }
      // the remaining slices
      while (ok && drained < nslices) {
        if (!mbar_wait_warp(&acc_full[b], aph[b], abort_flag)) { failed = it.job; ok = false; break; }
        tc_fence_after();
        drain_add(tmem + ((uint32_t)(quarter * 32) << 16) + b * BN_MAX + g * qw, qw, acc);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[b]);
        aph[b] ^= 1; b ^= 1; ++drained;
      }
      base_seq += (uint32_t)it.nk;
      if (!ok) break;
      const int grow = it.row0 + row;
      // destination: phases (a) / (c) write out (+ the K-range partial); orth() passes
      // write their intermediate factor, or the final result after the last pass
      float* dst = j.out + (long long)it.ks * j.split_stride;
      long long ld = j.ld_out;
      int cols = j.out_cols;
      bool fin = true;                       // writing the job's final result
      if (j.pass == 0 || (j.pass == 1 && *j.flag)) {
        dst = j.pass == 0 ? j.q1 : j.q2;
        ld = j.rp;
        cols = j.rp;
        fin = false;
      }
      if (grow < j.rows) {
        dst += (long long)grow * ld;
        const int cbase = it.c0 + g * qw;
        // 16-byte stores where the row is 16-byte aligned (leading dimension rp);
        // element stores for Vbar written into V (leading dimension r)
        const bool vec = ((ld & 3) == 0) && ((((uintptr_t)dst) & 15) == 0);
#pragma unroll
        for (int cb = 0; cb < QMAX / 8; ++cb)
          if (cb * 8 < qw) {
            const int c = cbase + cb * 8;
            if (vec && c + 8 <= cols) {
              *reinterpret_cast<float4*>(dst + c) =
                  make_float4(acc[cb * 8], acc[cb * 8 + 1], acc[cb * 8 + 2], acc[cb * 8 + 3]);
              *reinterpret_cast<float4*>(dst + c + 4) =
                  make_float4(acc[cb * 8 + 4], acc[cb * 8 + 5], acc[cb * 8 + 6], acc[cb * 8 + 7]);
            } else {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                if (c + k < cols) dst[c + k] = acc[cb * 8 + k];
            }
          }
        // tf32 halves for the next tensor-core kernel: row-major ones of the final
        // result, transposed ones of the final result (tr_fin) or of an intermediate
        // CholeskyQR factor (tr_inter: the next pass's Gram reads them)
        const bool want_rm = fin && j.sh;
        const bool want_tr = j.th && (fin ? j.tr_fin : j.tr_inter);
        if (want_rm || want_tr) {
          // c is a multiple of 8 and rp of 32, so a block of 8 is in or out
#pragma unroll
          for (int cb = 0; cb < QMAX / 8; ++cb)
            if (cb * 8 < qw && cbase + cb * 8 < j.rp) {
              const int c = cbase + cb * 8;
              float h[8], l[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) split_tf32(c + k < j.hcols ? acc[cb * 8 + k] : 0.f, h[k], l[k]);
              if (want_rm) {
                // two 16-byte pieces of the row in the update's operand tiles
                const long long o0 = optile_idx(grow, c, j.rp), o1 = optile_idx(grow, c + 4, j.rp);
                *reinterpret_cast<float4*>(j.sh + o0) = make_float4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<float4*>(j.sh + o1) = make_float4(h[4], h[5], h[6], h[7]);
                *reinterpret_cast<float4*>(j.sl + o0) = make_float4(l[0], l[1], l[2], l[3]);
                *reinterpret_cast<float4*>(j.sl + o1) = make_float4(l[4], l[5], l[6], l[7]);
              }
              if (want_tr) {
                // transposed: the 32 lanes of a warp hold 32 consecutive rows, so each
                // column is one 128-byte segment
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                  j.th[(long long)(c + k) * j.ld_t + grow] = h[k];
                  j.tl[(long long)(c + k) * j.ld_t + grow] = l[k];
                }
              }
            }
        }
      }
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

}  // namespace tcstream
}  // namespace dion
