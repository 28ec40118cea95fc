// Phase (e) on the 5th-generation tensor core: the fused parameter / residual
// update of every matrix of the plan (junaidaliop.github.io "Orth-Dion",
// update equations for X and R):
//
//     T1 = U Vbar^T,  T2 = U W^T            (K = r, 3xTF32, fp32 accumulation in TMEM)
//     X <- X - eta s T1,   R <- beta (G + R - T2)
//
// (In the momentum form of the low-rank Muon variant M = G + mu R and R <- M:
// the kernel computes R <- beta (G + mu R - gamma T2) with mu = beta = gamma = 1
// for Dion and mu = momentum, beta = 1, gamma = 0 for that variant.)
//
// The tensor core's fp32 accumulation truncates (its bias grows with the number
// of accumulation steps, about -1e-5 relative per 1024 of K), and R can be a
// small difference of large terms.  So one launch accumulates at most KPASS of
// K: a matrix with r > KPASS takes several launches ("K passes"), the first
// one as above with the first KPASS of K, every later one
//     X <- X - eta s T1',  R <- R - beta T2'
// with the next KPASS of K, the partial results carried in HBM in fp32.
//
// One CTA per SM, persistent over 128 x 128 tiles of every m x n matrix.
// Warp roles:
//   0  producer of the MMA operands (U hi/lo rows; [Vbar; W] hi/lo rows): each
//      128 x 16 operand tile is one contiguous 8 KB bulk copy (optile_idx layout)
//   1  TMEM allocator and MMA issuer (one thread)
//   2  TMA producer of the streamed state (G, R, X in 16-column sub-chunks)
//   3  idle
//   4-7 epilogue: TMEM -> registers, update in the staging buffers, TMA store
// The accumulator is double-buffered in TMEM (2 x 256 columns: T1 | T2) so the
// MMAs of the next tile overlap the epilogue of this one.  Operand stages hold
// 16 of K (64-byte swizzle), three in flight.
#pragma once

#include "common.cuh"
#include "tc.cuh"

namespace dion {
namespace tcepi {

using namespace dion::tc;

constexpr int BM = 128;          // rows of X per tile (TMEM lanes)
constexpr int BNJ = 128;         // columns of X per tile
constexpr int NMMA = 2 * BNJ;    // MMA N: [Vbar rows | W rows]
constexpr int BK = 16;           // K per operand stage (one 64-byte swizzle row of fp32)
constexpr int OSTAGES = 3;       // operand ring
constexpr int SUB = 16;          // columns per streamed sub-chunk
constexpr int QSTAGES_MAX = 4;   // streamed-state ring; the slot count is chosen per launch
constexpr int NTHREADS = 256;
constexpr uint32_t TMEM_COLS = 512;   // 2 accumulators x NMMA
constexpr int KPASS = 256;            // K accumulated per launch (per K pass)

constexpr uint32_t A_BYTES = BM * BK * 4;            // 8 KB
constexpr uint32_t BH_BYTES = NMMA * BK * 4;         // 16 KB ([Vbar; W] 256 rows)
constexpr uint32_t OST_BYTES = 2 * A_BYTES + 2 * BH_BYTES;   // 48 KB
constexpr uint32_t RX_BYTES = BM * SUB * 4;          // 8 KB
// Streamed-state region, cut per launch into slots of [G | R (8 KB) | X (8 KB)]:
// three slots of 20 KB (bf16 gradients) or 24 KB (fp32).  A fourth bf16 slot fits but
// was measured slower (its loads compete with the operand copies).
constexpr uint32_t QREG_BYTES = 81920;
constexpr uint32_t SMEM_BYTES = 1024 + OSTAGES * OST_BYTES + QREG_BYTES + 512;

enum { MAP_G, MAP_R, MAP_X, NMAPS };
static_assert(BM == OPT_ROWS && BNJ == OPT_ROWS && BK == OPT_K, "operand tiles are whole optile tiles");

struct EpiMat {
  CUtensorMap map[NMAPS];
  const float* uh;      // tf32 halves of U, Vbar and W in the optile layout (rows padded to 128)
  const float* ul;
  const float* vh;
  const float* vl;
  const float* wh;
  const float* wl;
  int m, n, rp, g_bf16;
  float eta_s, beta;
  unsigned* status;
  float mu, gamma;      // M = G + mu R;  R <- beta (M - gamma U W^T)
  int pad[8];
};
static_assert(sizeof(EpiMat) % 64 == 0, "EpiMat must keep 64-byte alignment of its maps");

// One 128 x 128 tile of matrix `mat` at rows i0.., columns j0.. (host-built table,
// one per K pass holding the matrices with rp > KPASS * pass).
struct Tile {
  int mat, i0, j0, pad;
};

__device__ __forceinline__ bool skip(const EpiMat& e) { return (*e.status & ST_FATAL) != 0; }

// Testing hook (dion_debug_expire_wait): the operand producer stops issuing at the
// first tile of this matrix, so that the MMA issuer's wait on it runs out (-1: off).
static __device__ int g_withhold_epi_matrix = -1;

__device__ __forceinline__ int nsub(const EpiMat& e, int j0) {
  const int left = e.n - j0;
  return left >= BNJ ? BNJ / SUB : (left + SUB - 1) / SUB;
}

__global__ void __launch_bounds__(NTHREADS, 1)
k_epi(const EpiMat* __restrict__ mats, const Tile* __restrict__ tiles, int ntiles, int qslot, int nq, int kpass) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = (unsigned char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  unsigned char* ost = smem;                                   // operand ring
  unsigned char* qst = smem + OSTAGES * OST_BYTES;             // streamed-state ring
  const int QSTAGES = nq;                  // streamed-state slots of this launch (<= QSTAGES_MAX)
  const int QST_BYTES = qslot;
  const int Q_R = qslot - 2 * RX_BYTES;    // offsets of R and X in a slot (G first)
  const int kc0 = kpass * (KPASS / BK);    // first K chunk of this pass
  uint64_t* bars = (uint64_t*)(qst + QREG_BYTES);
  uint64_t* op_full = bars;
  uint64_t* op_empty = op_full + OSTAGES;
  uint64_t* acc_full = op_empty + OSTAGES;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* q_full = acc_empty + 2;
  uint64_t* q_empty = q_full + QSTAGES_MAX;
  uint64_t* drain = q_empty + QSTAGES_MAX;
  uint32_t* tslot = (uint32_t*)(drain + 1);
  volatile int* abort_flag = (volatile int*)(tslot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < OSTAGES; ++i) { mbar_init(&op_full[i], 1); mbar_init(&op_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], 4); }
    for (int i = 0; i < QSTAGES; ++i) { mbar_init(&q_full[i], 1); mbar_init(&q_empty[i], 1); }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) { tmem_alloc(tslot, TMEM_COLS); tmem_relinquish(); }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  int failed_mat = -1;   // matrix whose wait timed out in this thread, if any

  if (warp == 0 && lane == 0) {
    // ---------------------------------------------------------- operand producer
    int s = 0; uint32_t ph = 0;
    uint32_t last_ph[OSTAGES] = {0, 0, 0}; bool used[OSTAGES] = {false, false, false};
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tiles[t];
      const EpiMat& e = mats[tl.mat];
      if (skip(e) || kc0 * BK >= e.rp) continue;
      if (tl.mat == g_withhold_epi_matrix) goto prod_done;
      const int kc1 = min((e.rp + BK - 1) / BK, kc0 + KPASS / BK);
      const int kt = e.rp / OPT_K;                          // tiles per 128 rows
      const long long tu = (long long)(tl.i0 / OPT_ROWS) * kt, tv = (long long)(tl.j0 / OPT_ROWS) * kt;
      for (int kc = kc0; kc < kc1; ++kc) {
        if (!mbar_wait(&op_empty[s], ph ^ 1, abort_flag)) { failed_mat = tl.mat; goto prod_done; }
        mbar_arrive_expect_tx(&op_full[s], OST_BYTES);
        unsigned char* b = ost + s * OST_BYTES;
        const long long ou = (tu + kc) * OPT_FLOATS, ov = (tv + kc) * OPT_FLOATS;
        bulk_load(b, e.uh + ou, A_BYTES, &op_full[s]);
        bulk_load(b + A_BYTES, e.ul + ou, A_BYTES, &op_full[s]);
        bulk_load(b + 2 * A_BYTES, e.vh + ov, A_BYTES, &op_full[s]);
        bulk_load(b + 2 * A_BYTES + BH_BYTES / 2, e.wh + ov, A_BYTES, &op_full[s]);
        bulk_load(b + 2 * A_BYTES + BH_BYTES, e.vl + ov, A_BYTES, &op_full[s]);
        bulk_load(b + 2 * A_BYTES + BH_BYTES + BH_BYTES / 2, e.wl + ov, A_BYTES, &op_full[s]);
        used[s] = true; last_ph[s] = ph;
        if (++s == OSTAGES) { s = 0; ph ^= 1; }
      }
    }
  prod_done:
    if (*abort_flag)
      for (int i = 0; i < OSTAGES; ++i) if (used[i]) mbar_wait_drain(&op_full[i], last_ph[i]);
  } else if (warp == 1 && lane == 0) {
    // ---------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_tf32(BM, NMMA);
    int s = 0; uint32_t ph = 0; int b = 0; uint32_t aph[2] = {0, 0};
    bool issued = false;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tiles[t];
      const EpiMat& e = mats[tl.mat];
      if (skip(e) || kc0 * BK >= e.rp) continue;
      const int kc1 = min((e.rp + BK - 1) / BK, kc0 + KPASS / BK);
      if (!mbar_wait(&acc_empty[b], aph[b] ^ 1, abort_flag)) { failed_mat = tl.mat; goto mma_done; }
      tc_fence_after();
      const uint32_t d = tmem + b * NMMA;
      for (int kc = kc0; kc < kc1; ++kc) {
        if (!mbar_wait(&op_full[s], ph, abort_flag)) { failed_mat = tl.mat; goto mma_done; }
        tc_fence_after();
        const uint32_t ah = smem_u32(ost + s * OST_BYTES), al = ah + A_BYTES;
        const uint32_t bh = ah + 2 * A_BYTES, bl = bh + BH_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 8; ++kk) {
          const uint32_t o = kk * 32;
          mma_tf32(d, sdesc_k_sw64(al + o), sdesc_k_sw64(bh + o), idesc, ((kc - kc0) | kk) != 0);
          mma_tf32(d, sdesc_k_sw64(ah + o), sdesc_k_sw64(bl + o), idesc, 1);
          mma_tf32(d, sdesc_k_sw64(ah + o), sdesc_k_sw64(bh + o), idesc, 1);
        }
        issued = true;
        mma_commit(&op_empty[s]);
        if (++s == OSTAGES) { s = 0; ph ^= 1; }
      }
      mma_commit(&acc_full[b]);
      aph[b] ^= 1; b ^= 1;
    }
  mma_done:
    if (*abort_flag && issued) { mma_commit(drain); mbar_wait_drain(drain, 0); }
  } else if (warp == 2 && lane == 0) {
    // ---------------------------------------------------------- streamed-state producer
    int q = 0; uint32_t ph = 0;
    uint32_t last_ph[QSTAGES_MAX] = {0, 0, 0, 0}; bool used[QSTAGES_MAX] = {false, false, false, false};
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tiles[t];
      const EpiMat& e = mats[tl.mat];
      if (skip(e) || kc0 * BK >= e.rp) continue;
      // later K passes read the carried R and X only
      const uint32_t gbytes = kpass > 0 ? 0u : (e.g_bf16 ? BM * SUB * 2 : BM * SUB * 4);
      const int ns = nsub(e, tl.j0);
      for (int sc = 0; sc < ns; ++sc) {
        if (!mbar_wait(&q_empty[q], ph ^ 1, abort_flag)) { failed_mat = tl.mat; goto stream_done; }
        mbar_arrive_expect_tx(&q_full[q], gbytes + 2 * RX_BYTES);
        unsigned char* b = qst + q * QST_BYTES;
        const int x = tl.j0 + sc * SUB;
        if (kpass == 0) tma_load_2d(b, &e.map[MAP_G], &q_full[q], x, tl.i0);
        tma_load_2d(b + Q_R, &e.map[MAP_R], &q_full[q], x, tl.i0);
        tma_load_2d(b + Q_R + RX_BYTES, &e.map[MAP_X], &q_full[q], x, tl.i0);
        used[q] = true; last_ph[q] = ph;
        if (++q == QSTAGES) { q = 0; ph ^= 1; }
      }
    }
  stream_done:
    if (*abort_flag)
      for (int i = 0; i < QSTAGES_MAX; ++i) if (used[i]) mbar_wait_drain(&q_full[i], last_ph[i]);
  } else if (warp >= 4) {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;         // TMEM lane = row of the tile
    const bool leader = (warp == 4 && lane == 0);
    int b = 0; uint32_t aph[2] = {0, 0};
    int q = 0; uint32_t ph = 0;
    int prev_q = -1;   // staging slot whose TMA stores are still reading it (leader only)
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      const Tile tl = tiles[t];
      const EpiMat& e = mats[tl.mat];
      if (skip(e) || kc0 * BK >= e.rp) continue;
      // every wait is followed by a vote of the 128 epilogue threads, so that
      // they leave together and nobody is left behind at a named barrier
      bool ok = mbar_wait(&acc_full[b], aph[b], abort_flag);
      if (!ok) failed_mat = tl.mat;
      if (!named_sync_all(1, 128, ok)) break;
      tc_fence_after();
      const int ns = nsub(e, tl.j0);
      const float eta_s = e.eta_s, beta = e.beta, mu = e.mu, gamma = e.gamma;
      for (int sc = 0; sc < ns; ++sc) {
        ok = mbar_wait(&q_full[q], ph, abort_flag);
        if (!ok) failed_mat = tl.mat;
        if (!named_sync_all(1, 128, ok)) { ok = false; break; }
        float t1[16], t2[16];
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16) + b * NMMA + sc * SUB;
        tmem_ld16(lane_addr, t1);
        tmem_ld16(lane_addr + BNJ, t2);
        tmem_wait_ld();
        unsigned char* gb = qst + q * QST_BYTES;
        unsigned char* rb = gb + Q_R;
        unsigned char* xb = rb + RX_BYTES;
        float g[16];
        if (kpass > 0) {
          // a later K pass: R already holds beta (G + R - T2 of the earlier passes)
#pragma unroll
          for (int k = 0; k < 16; ++k) g[k] = 0.f;
        } else if (e.g_bf16) {
          // 32-byte rows, 32-byte swizzle: 16-byte chunk c of row t at c ^ ((t >> 2) & 1)
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const uint4 v = *reinterpret_cast<const uint4*>(gb + row * 32 + ((c ^ ((row >> 2) & 1)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              g[c * 8 + 2 * k] = __uint_as_float(w[k] << 16);
              g[c * 8 + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const float4 v = *reinterpret_cast<const float4*>(gb + row * 64 + ((c ^ ((row >> 1) & 3)) << 4));
            g[4 * c] = v.x; g[4 * c + 1] = v.y; g[4 * c + 2] = v.z; g[4 * c + 3] = v.w;
          }
        }
        // 64-byte rows, 64-byte swizzle: chunk c of row t at c ^ ((t >> 1) & 3)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = row * 64 + ((c ^ ((row >> 1) & 3)) << 4);
          float4 r = *reinterpret_cast<float4*>(rb + off);
          float4 x = *reinterpret_cast<float4*>(xb + off);
          const int k = 4 * c;
          x.x = fmaf(-eta_s, t1[k], x.x);
          x.y = fmaf(-eta_s, t1[k + 1], x.y);
          x.z = fmaf(-eta_s, t1[k + 2], x.z);
          x.w = fmaf(-eta_s, t1[k + 3], x.w);
          if (kpass == 0) {
            r.x = beta * (fmaf(mu, r.x, g[k]) - gamma * t2[k]);
            r.y = beta * (fmaf(mu, r.y, g[k + 1]) - gamma * t2[k + 1]);
            r.z = beta * (fmaf(mu, r.z, g[k + 2]) - gamma * t2[k + 2]);
            r.w = beta * (fmaf(mu, r.w, g[k + 3]) - gamma * t2[k + 3]);
          } else {
            r.x = fmaf(-beta * gamma, t2[k], r.x);
            r.y = fmaf(-beta * gamma, t2[k + 1], r.y);
            r.z = fmaf(-beta * gamma, t2[k + 2], r.z);
            r.w = fmaf(-beta * gamma, t2[k + 3], r.w);
          }
          *reinterpret_cast<float4*>(rb + off) = r;
          *reinterpret_cast<float4*>(xb + off) = x;
        }
        fence_async_smem();
        named_sync(1, 128);
        if (leader) {
          // stores of this slot go out now; the previous slot is released once
          // its own stores have read the shared memory (all but the newest group)
          const int x = tl.j0 + sc * SUB;
          tma_store_2d(&e.map[MAP_R], rb, x, tl.i0);
          tma_store_2d(&e.map[MAP_X], xb, x, tl.i0);
          tma_store_commit();
          tma_store_wait_read<1>();
          if (prev_q >= 0) mbar_arrive(&q_empty[prev_q]);
          prev_q = q;
        }
        if (++q == QSTAGES) { q = 0; ph ^= 1; }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[b]);
      aph[b] ^= 1; b ^= 1;
    }
    if (leader) {
      tma_store_wait_all<0>();
      if (prev_q >= 0) mbar_arrive(&q_empty[prev_q]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) { tc_fence_after(); tmem_dealloc(tmem, TMEM_COLS); }
  if (failed_mat >= 0) atomicOr(mats[failed_mat].status, ST_TIMEOUT);
  // after an abort this CTA left tiles unfinished: every matrix it had tiles of is incomplete
  if (threadIdx.x == 0 && *abort_flag)
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) atomicOr(mats[tiles[t].mat].status, ST_TIMEOUT);
}

}  // namespace tcepi
}  // namespace dion
