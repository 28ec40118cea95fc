// Host side of libdion: descriptor validation, workspace layout, device
// tables, and the grouped launches of each phase of the Dion / Orth-Dion step
// (junaidaliop.github.io "Orth-Dion", update equations and glossary).
#include "dion.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "common.cuh"
#include "host_errors.h"
#include "simt.cuh"
#include "tc_epilogue.cuh"
#include "tc_split.cuh"
#include "tc_stream.cuh"
#include "tc_gram.cuh"
#include "bchol.cuh"

using namespace dion;

namespace {
thread_local std::string g_err;
}  // namespace

// Error text of the calling host thread, shared by every translation unit of the
// library (host_errors.h).
dion_status_t dion_fail(dion_status_t s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

dion_status_t dion_ok() {
  g_err.clear();
  return DION_OK;
}

namespace {

template <class... A>
dion_status_t fail(dion_status_t s, const char* fmt, A... a) { return dion_fail(s, fmt, a...); }
dion_status_t ok() { return dion_ok(); }

constexpr size_t kAlign = 256;
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

// rank padding granule: one 128-byte row of fp32 operands (the tensor-core K step)
constexpr long long kRankGranule = 32;

}  // namespace

// ---- scratch of dion_orth_noalloc (see include/dion.h): a fixed device array
// inside the library, for callers that cannot allocate device memory.
namespace noalloc {
constexpr long long kRowsMax = DION_NOALLOC_MAX_ROWS;
constexpr long long kRankMax = DION_NOALLOC_MAX_RANK;        // rp == kRankMax at most
constexpr long long kChunksMax = 32;                           // Gram partials (CUDA-core chunking)
constexpr size_t kJobBytes = 512;                              // OrthJob + two launch tables + status words
constexpr size_t kGpartFloats = (size_t)kChunksMax * kRankMax * kRankMax;
constexpr size_t kSFloats = (size_t)kRankMax * kRankMax + kRankMax + 32 * kRankMax;
constexpr size_t kTFloats = (size_t)kRankMax * kRankMax;
constexpr size_t kQFloats = (size_t)kRowsMax * kRankMax;
constexpr size_t kBytes = kJobBytes + 4 * (kGpartFloats + kSFloats + kTFloats + 2 * kQFloats);
constexpr int kMaxDevices = 64;                                // per-device address cache
}  // namespace noalloc
static __device__ __align__(256) unsigned char g_noalloc_scratch[noalloc::kBytes];

struct dion_plan {
  std::vector<dion_matrix_desc> descs;
  int count = 0;
  std::vector<long long> rp;
  std::vector<int> ksplit, kchunk;
  std::vector<int> nchunk_p, chunk_p, nchunk_w, chunk_w;
  std::vector<int> orth_idx, dion_idx;   // matrices by right-factor variant

  // workspace layout (byte offsets from the workspace base)
  size_t ws_bytes = 0;
  // exchange regions of the row-sharded step: the reduced Grams of orth(P) of every
  // matrix, and every W, each back to back (dion_plan_exchange)
  size_t off_gx = 0, gx_bytes = 0, off_wx = 0, wx_bytes = 0;
  std::vector<size_t> off_gsum;
  // tf32 halves of W recomputed from the exchanged W (row-sharded stage 4)
  size_t t_wsplit = 0, t_ts_wsplit = 0;
  std::vector<int> ts_wsplit;
  size_t off_tables = 0, tables_bytes = 0, off_status = 0;
  std::vector<size_t> off_P, off_Q, off_Q2, off_U, off_W, off_Wpart, off_gpart, off_S, off_T, off_Vo;

  // table image layout (byte offsets inside the tables region)
  size_t t_mats = 0, t_jobs_p = 0, t_jobs_w = 0, t_jobs_v = 0, t_ts_gram_v = 0, t_ts_trmm_v = 0;
  size_t t_ts_gram_p = 0, t_ts_trmm_p = 0, t_ts_wred = 0, t_ts_gram_w = 0, t_ts_trmm_w = 0, t_ts_coln = 0,
         t_coln_idx = 0;
  std::vector<int> ts_gram_p, ts_trmm_p, ts_wred, ts_gram_w, ts_trmm_w, ts_coln;
  std::vector<int> ts_gram_v, ts_trmm_v;   // orth(V) of the Dion matrices
  bool any_split = false;

  // tensor-core path: split (hi/lo tf32) operand copies and the phase (e) tables
  std::vector<size_t> off_Uh, off_Ul, off_Vh, off_Vl, off_Wh, off_Wl;
  size_t t_epi = 0, t_split = 0, t_ts_split = 0;
  std::vector<int> ts_split;
  int n_split = 0;
  // k_split jobs (matrix, 0: U / 1: Vbar): the halves that no earlier kernel wrote
  std::vector<std::pair<int, int>> split_list;
  int num_sms = 0;
  // phases (a) and (c): streaming jobs, transposed split copies V^T, U^T
  std::vector<int> ncb, bn;
  std::vector<long long> ldt_n, ldt_m;
  std::vector<size_t> off_VTh, off_VTl, off_UTh, off_UTl;
  size_t t_sj_a = 0, t_sj_c = 0, t_tj_v = 0, t_tj_u = 0, t_ts_tv = 0, t_ts_tu = 0;
  std::vector<int> ts_tv, ts_tu;
  // tensor-core orth(): per list (0 = P, 1 = W, 2 = V) and pass, Gram and A T jobs
  bool tc_orth = true;
  // ranks above 192: Gram by the streaming kernel (transposed mode, K split over rows),
  // blocked Cholesky + inverse, T^T halves by the transposed split
  bool big_orth = false;
  std::vector<int> gks[3], gkc[3];                 // per list and job: K split and chunk of the Gram
  std::vector<tcstream::Item> it_gs[3];            // Gram work items per list
  size_t t_gsj[3][3] = {}, t_it_gs[3] = {}, t_atj[3] = {}, t_ts_atj[3] = {}, t_ttj[3] = {}, t_ts_ttj[3] = {};
  std::vector<int> ts_atj[3], ts_ttj[3];
  long long rmax_l[3] = {0, 0, 0};                 // largest rank of each list
  bool any_g_f32 = false;   // a gradient in fp32: larger staging slots
  std::vector<size_t> off_Tth, off_Ttl;
  size_t t_gj[3][3] = {}, t_tj[3][3] = {};
  std::vector<int> ts_gred[3];
  std::vector<int> chol_order[3];          // jobs of each orth list, largest rank first
  size_t t_chol_order[3] = {};
  size_t t_ts_gred[3] = {};
  size_t t_vcopy = 0, t_ts_vcopy = 0;
  std::vector<int> ts_vcopy;
  // work-item tables of the persistent tensor-core kernels (built on the host, heaviest first)
  std::vector<tcstream::Item> it_sa, it_sc, it_tr[3];
  std::vector<std::vector<tcepi::Tile>> it_epi;   // per K pass of the update
  std::vector<tcgram::GItem> it_g[3];
  size_t t_it_sa = 0, t_it_sc = 0, t_it_tr[3] = {}, t_it_g[3] = {};
  std::vector<size_t> t_it_epi;

  std::vector<unsigned char> image;
  const void* uploaded_ws = nullptr;
  bool dirty = true;
};

namespace {

dion_status_t validate(const dion_matrix_desc* d, int count) {
  struct Range { uintptr_t lo, hi; bool writable; int idx; };
  std::vector<Range> ranges;
  ranges.reserve((size_t)count * 4);
  for (int i = 0; i < count; ++i) {
    const dion_matrix_desc& x = d[i];
    if (!x.X || !x.G || !x.R || !x.V)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: NULL pointer", i);
    if (x.m < 1 || x.n < 1 || x.m >= (1LL << 31) || x.n >= (1LL << 31))   // rows index as int32 on the device
      return fail(DION_ERR_INVALID_ARG, "matrix %d: bad shape %lld x %lld", i, (long long)x.m, (long long)x.n);
    if (x.r < 1 || x.r > std::min(x.m, x.n))
      return fail(DION_ERR_INVALID_ARG, "matrix %d: rank %lld outside [1, min(m, n) = %lld]", i,
                  (long long)x.r, (long long)std::min(x.m, x.n));
    if (x.ld_x < x.n || x.ld_g < x.n || x.ld_r < x.n)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: leading dimension below n", i);
    if (x.g_dtype != DION_DTYPE_F32 && x.g_dtype != DION_DTYPE_BF16)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: unknown g_dtype %d", i, x.g_dtype);
    if (x.variant != DION_VARIANT_DION && x.variant != DION_VARIANT_ORTH && x.variant != DION_VARIANT_LOWRANK_MUON)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: unknown variant %d", i, x.variant);
    if (!std::isfinite(x.eta) || !std::isfinite(x.beta) || !std::isfinite(x.scale))
      return fail(DION_ERR_INVALID_ARG, "matrix %d: non-finite eta / beta / scale", i);
    if (x.reserved != 0.f)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: reserved field must be 0", i);
    const size_t gsz = x.g_dtype == DION_DTYPE_BF16 ? 2 : 4;
    if (((uintptr_t)x.X | (uintptr_t)x.G | (uintptr_t)x.R | (uintptr_t)x.V) & 15)
      return fail(DION_ERR_UNSUPPORTED, "matrix %d: pointers must be 16-byte aligned", i);
    if ((x.ld_x * 4) % 16 || (x.ld_r * 4) % 16 || (x.ld_g * (long long)gsz) % 16)
      return fail(DION_ERR_UNSUPPORTED, "matrix %d: row pitch of X, G, R must be a multiple of 16 bytes", i);
    auto span = [](const void* p, long long rows, long long cols, long long ld, size_t es) {
      const uintptr_t lo = (uintptr_t)p;
      return Range{lo, lo + (uintptr_t)(((rows - 1) * ld + cols) * (long long)es), false, 0};
    };
    Range rx = span(x.X, x.m, x.n, x.ld_x, 4); rx.writable = true; rx.idx = i;
    Range rr = span(x.R, x.m, x.n, x.ld_r, 4); rr.writable = true; rr.idx = i;
    Range rv = span(x.V, x.n, x.r, x.r, 4); rv.writable = true; rv.idx = i;
    Range rg = span(x.G, x.m, x.n, x.ld_g, gsz); rg.writable = false; rg.idx = i;
    ranges.push_back(rx); ranges.push_back(rr); ranges.push_back(rv); ranges.push_back(rg);
  }
  std::sort(ranges.begin(), ranges.end(), [](const Range& a, const Range& b) { return a.lo < b.lo; });
  uintptr_t end_any = 0, end_w = 0;
  for (const Range& g : ranges) {
    if (g.writable ? g.lo < end_any : g.lo < end_w)
      return fail(DION_ERR_INVALID_ARG, "matrix %d: buffer overlaps another matrix's buffer", g.idx);
    end_any = std::max(end_any, g.hi);
    if (g.writable) end_w = std::max(end_w, g.hi);
  }
  return DION_OK;
}

template <class T>
void put(std::vector<unsigned char>& img, size_t off, const T* src, size_t n) {
  std::memcpy(img.data() + off, src, n * sizeof(T));
}

void layout(dion_plan* p) {
  const int cnt = p->count;
  p->rp.resize(cnt); p->ksplit.resize(cnt); p->kchunk.resize(cnt);
  p->nchunk_p.resize(cnt); p->chunk_p.resize(cnt); p->nchunk_w.resize(cnt); p->chunk_w.resize(cnt);
  for (int i = 0; i < cnt; ++i) {
    const auto& d = p->descs[i];
    p->rp[i] = cdiv(d.r, kRankGranule) * kRankGranule;
    (d.variant == DION_VARIANT_DION ? p->dion_idx : p->orth_idx).push_back(i);
  }
  // column blocks of the streaming kernels (TMEM holds two slices of bn <= 192 columns)
  p->ncb.resize(cnt); p->bn.resize(cnt); p->ldt_n.resize(cnt); p->ldt_m.resize(cnt);
  for (int i = 0; i < cnt; ++i) {
    p->ncb[i] = (int)cdiv(p->rp[i], tcstream::BN_MAX);
    p->bn[i] = (int)(cdiv(cdiv(p->rp[i], p->ncb[i]), 32) * 32);
    p->ldt_n[i] = cdiv(p->descs[i].n, 32) * 32;
    p->ldt_m[i] = cdiv(p->descs[i].m, 32) * 32;
  }
  // phase (c) splits the rows of M (its K) into ranges when the batch has too few
  // items to fill the GPU (then of at most 2048 rows), and otherwise only where an
  // item would exceed a third of a CTA's share of the work (or 2048 rows, if more):
  // a split costs the write and the reduction of its K-range partials of W
  long long items_c = 0, work_c = 0;
  for (int i = 0; i < cnt; ++i) {
    items_c += cdiv(p->descs[i].n, tcstream::BM) * p->ncb[i];
    work_c += cdiv(p->descs[i].n, tcstream::BM) * p->ncb[i] * p->descs[i].m;
  }
  const long long want = 2LL * 148;
  const long long split = items_c >= want ? 1 : cdiv(want, items_c);
  const long long cap = split > 1 ? 2048 : std::max<long long>(2048, cdiv(work_c / (3 * 148), 256) * 256);
  for (int i = 0; i < cnt; ++i) {
    const long long m = p->descs[i].m;
    long long ch = cdiv(cdiv(m, split), 256) * 256;
    ch = std::min<long long>(ch, cap);
    ch = std::min<long long>(ch, cdiv(m, 32) * 32);
    p->kchunk[i] = (int)ch;
    p->ksplit[i] = (int)cdiv(m, ch);
    if (p->ksplit[i] > 1) p->any_split = true;
  }
  p->any_g_f32 = false;
  for (int i = 0; i < cnt; ++i) p->any_g_f32 = p->any_g_f32 || p->descs[i].g_dtype == DION_DTYPE_F32;
  p->tc_orth = true;
  p->big_orth = false;
  for (int i = 0; i < cnt; ++i) p->big_orth = p->big_orth || p->rp[i] > tcgram::RP_MAX;
  for (int i = 0; i < cnt; ++i) {
    // tensor-core Gram of ranks <= 192: one partial per 256 rows
    p->chunk_p[i] = p->chunk_w[i] = tcgram::CHUNK_ROWS;
    p->nchunk_p[i] = (int)cdiv(p->descs[i].m, tcgram::CHUNK_ROWS);
    p->nchunk_w[i] = (int)cdiv(p->descs[i].n, tcgram::CHUNK_ROWS);
  }
  {
    const std::vector<int>* lists[3] = {nullptr, &p->orth_idx, &p->dion_idx};
    for (int L = 0; L < 3; ++L) {
      const size_t nj = L == 0 ? (size_t)cnt : lists[L]->size();
      auto mat = [&](size_t k) { return L == 0 ? (int)k : (*lists[L])[k]; };
      p->rmax_l[L] = 0;
      for (size_t k = 0; k < nj; ++k) p->rmax_l[L] = std::max<long long>(p->rmax_l[L], p->descs[mat(k)].r);
      p->gks[L].assign(nj, 1);
      p->gkc[L].assign(nj, 0);
      p->it_gs[L].clear();
      if (!p->big_orth) continue;
      // Gram by the streaming kernel: output rows rp (128-row tiles) x column blocks, the
      // rows of the factor as K, split into ranges of at most 2048 until the GPU is full
      long long items = 0;
      for (size_t k = 0; k < nj; ++k) items += cdiv(p->rp[mat(k)], tcstream::BM) * p->ncb[mat(k)];
      const long long want = 2LL * 148;
      const long long split = items >= want ? 1 : cdiv(want, std::max<long long>(1, items));
      for (size_t k = 0; k < nj; ++k) {
        const int i = mat(k);
        const long long rows = L == 0 ? p->descs[i].m : p->descs[i].n;
        long long ch = cdiv(cdiv(rows, split), 256) * 256;
        ch = std::min<long long>(ch, 2048);
        ch = std::min<long long>(ch, cdiv(rows, 32) * 32);
        p->gkc[L][k] = (int)ch;
        p->gks[L][k] = (int)cdiv(rows, ch);
        (L == 0 ? p->nchunk_p[i] : p->nchunk_w[i]) = p->gks[L][k];
        (L == 0 ? p->chunk_p[i] : p->chunk_w[i]) = (int)ch;
        // the Gram is symmetric and its consumers read the upper triangle only: tiles
        // wholly below the diagonal (first row past the block's last column) are skipped
        for (long long r0 = 0; r0 < p->rp[i]; r0 += tcstream::BM)
          for (int ks = 0; ks < p->gks[L][k]; ++ks)
            for (int cb = 0; cb < p->ncb[i]; ++cb) {
              if (r0 >= (long long)(cb + 1) * p->bn[i]) continue;
              const long long k0 = (long long)ks * ch, k1 = std::min<long long>(rows, k0 + ch);
              p->it_gs[L].push_back(tcstream::Item{(int)k, (int)r0, ks, cb * p->bn[i], (int)k0,
                                                   (int)cdiv(k1 - k0, tcstream::BK), 0, 0});
            }
      }
      std::stable_sort(p->it_gs[L].begin(), p->it_gs[L].end(), [](const tcstream::Item& a, const tcstream::Item& b) {
        return a.nk > b.nk; });
    }
  }

  // ---- tile prefix sums
  auto prefix = [&](std::vector<int>& ts, const std::vector<int>& ids, auto tiles_of) {
    ts.assign(ids.size() + 1, 0);
    for (size_t k = 0; k < ids.size(); ++k) ts[k + 1] = ts[k] + (int)tiles_of(ids[k]);
  };
  std::vector<int> all(cnt);
  for (int i = 0; i < cnt; ++i) all[i] = i;
  auto D = [&](int i) -> const dion_matrix_desc& { return p->descs[i]; };
  prefix(p->ts_gram_p, all, [&](int i) { long long t = cdiv(p->rp[i], simt::TN); return p->nchunk_p[i] * t * t; });
  prefix(p->ts_trmm_p, all, [&](int i) { return cdiv(D(i).m, simt::TM) * cdiv(p->rp[i], simt::TN); });
  prefix(p->ts_wred, all, [&](int i) { return p->ksplit[i] > 1 ? cdiv(D(i).n * p->rp[i], 1024) : 1; });
  prefix(p->ts_gram_w, p->orth_idx, [&](int i) { long long t = cdiv(p->rp[i], simt::TN); return p->nchunk_w[i] * t * t; });
  prefix(p->ts_trmm_w, p->orth_idx, [&](int i) { return cdiv(D(i).n, simt::TM) * cdiv(p->rp[i], simt::TN); });
  prefix(p->ts_coln, p->dion_idx, [&](int i) { return cdiv(D(i).r, 32); });
  prefix(p->ts_gram_v, p->dion_idx, [&](int i) { long long t = cdiv(p->rp[i], simt::TN); return p->nchunk_w[i] * t * t; });
  prefix(p->ts_trmm_v, p->dion_idx, [&](int i) { return cdiv(D(i).n, simt::TM) * cdiv(p->rp[i], simt::TN); });

  // ---- tables region
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 128); return o; };
  // tensor-core tables first: they hold CUtensorMaps (64-byte alignment)
  // tf32 halves for the update: the tensor-core orth() writes those of U and of an
  // Orth-Dion Vbar itself, phase (c) those of W; the rest come from k_split
  p->split_list.clear();
  for (int i = 0; i < cnt; ++i)
    if (D(i).variant == DION_VARIANT_DION) p->split_list.push_back({i, 1});
  p->n_split = (int)p->split_list.size();
  {
    std::vector<int> jobs(p->n_split);
    for (int k = 0; k < p->n_split; ++k) jobs[k] = k;
    prefix(p->ts_split, jobs, [&](int k) {
      const int i = p->split_list[k].first;
      const long long rows = p->split_list[k].second == 0 ? D(i).m : D(i).n;
      return cdiv(rows * p->rp[i], tcsplit::ELEMS_PER_CTA);
    });
  }
  prefix(p->ts_wsplit, all, [&](int i) { return cdiv(D(i).n * p->rp[i], tcsplit::ELEMS_PER_CTA); });
  prefix(p->ts_tv, all, [&](int i) { return cdiv(D(i).n, tcsplit::TROWS) * cdiv(p->rp[i], 32); });
  prefix(p->ts_tu, all, [&](int i) { return cdiv(D(i).m, tcsplit::TROWS) * cdiv(p->rp[i], 32); });
  {
    const std::vector<int>* lists[3] = {&all, &p->orth_idx, &p->dion_idx};
    for (int L = 0; L < 3; ++L) {
      const size_t nj = std::max<size_t>(1, lists[L]->size());
      prefix(p->ts_gred[L], *lists[L], [&](int i) { return cdiv(p->rp[i] * p->rp[i], simt::GRED_ELEMS); });
      for (int ps = 0; ps < 3; ++ps) {
        p->t_gj[L][ps] = take(sizeof(tcgram::GJob) * nj);
        p->t_tj[L][ps] = take(sizeof(tcstream::SJob) * nj);
      }
    }
    prefix(p->ts_vcopy, p->dion_idx, [&](int i) { return cdiv(D(i).n * p->rp[i], tcsplit::ELEMS_PER_CTA); });
    p->t_vcopy = take(sizeof(tcsplit::SplitJob) * std::max<size_t>(1, p->dion_idx.size()));
    for (int L = 0; L < 3; ++L) {
      p->t_ts_gred[L] = take(4 * p->ts_gred[L].size());
    }
    p->t_ts_vcopy = take(4 * p->ts_vcopy.size());
  }
  // ---- work-item tables
  {
    auto by_cost = [](std::vector<tcstream::Item>& v, const std::vector<int>& bnv, bool job_is_matrix,
                      const std::vector<int>* list) {
      std::stable_sort(v.begin(), v.end(), [&](const tcstream::Item& a, const tcstream::Item& b) {
        const int ia = job_is_matrix ? a.job : (*list)[a.job], ib = job_is_matrix ? b.job : (*list)[b.job];
        return (long long)a.nk * bnv[ia] > (long long)b.nk * bnv[ib];
      });
    };
    p->it_sa.clear();
    p->it_sc.clear();
    for (int i = 0; i < cnt; ++i) {
      const long long m = D(i).m, n = D(i).n;
      for (long long r0 = 0; r0 < m; r0 += tcstream::BM)
        for (int cb = 0; cb < p->ncb[i]; ++cb)
          p->it_sa.push_back(tcstream::Item{i, (int)r0, 0, cb * p->bn[i], 0, (int)cdiv(n, tcstream::BK), 0, 0});
      for (long long r0 = 0; r0 < n; r0 += tcstream::BM)
        for (int ks = 0; ks < p->ksplit[i]; ++ks)
          for (int cb = 0; cb < p->ncb[i]; ++cb) {
            const long long k0 = (long long)ks * p->kchunk[i];
            const long long k1 = std::min<long long>(m, k0 + p->kchunk[i]);
            p->it_sc.push_back(tcstream::Item{i, (int)r0, ks, cb * p->bn[i], (int)k0,
                                              (int)cdiv(k1 - k0, tcstream::BK), 0, 0});
          }
    }
    by_cost(p->it_sa, p->bn, true, nullptr);
    by_cost(p->it_sc, p->bn, true, nullptr);
    const std::vector<int>* lists[3] = {&all, &p->orth_idx, &p->dion_idx};
    for (int L = 0; L < 3; ++L) {
      p->it_tr[L].clear();
      p->it_g[L].clear();
      for (size_t k = 0; k < lists[L]->size(); ++k) {
        const int i = (*lists[L])[k];
        const long long rows = L == 0 ? D(i).m : D(i).n;
        for (long long r0 = 0; r0 < rows; r0 += tcstream::BM)
          for (int cb = 0; cb < p->ncb[i]; ++cb)
            // T is upper triangular: output columns below c0 + bn need K below c0 + bn only
            p->it_tr[L].push_back(tcstream::Item{
                (int)k, (int)r0, 0, cb * p->bn[i], 0,
                (int)(std::min<long long>(p->rp[i], (long long)(cb + 1) * p->bn[i]) / tcstream::BK), 0, 0});
        for (long long c = 0; c < cdiv(rows, tcgram::CHUNK_ROWS); ++c)
          p->it_g[L].push_back(tcgram::GItem{(int)k, (int)c, 0, 0});
      }
      by_cost(p->it_tr[L], p->bn, false, lists[L]);
    }
    // update tiles per K pass: pass k holds the matrices with rp > k * KPASS
    long long rpmax = 0;
    for (int i = 0; i < cnt; ++i) rpmax = std::max<long long>(rpmax, p->rp[i]);
    const int npass = (int)cdiv(rpmax, tcepi::KPASS);
    p->it_epi.assign(npass, {});
    for (int k = 0; k < npass; ++k) {
      for (int i = 0; i < cnt; ++i) {
        if (p->rp[i] <= (long long)k * tcepi::KPASS) continue;
        for (long long i0 = 0; i0 < D(i).m; i0 += tcepi::BM)
          for (long long j0 = 0; j0 < D(i).n; j0 += tcepi::BNJ)
            p->it_epi[k].push_back(tcepi::Tile{i, (int)i0, (int)j0, 0});
      }
      std::stable_sort(p->it_epi[k].begin(), p->it_epi[k].end(), [&](const tcepi::Tile& a, const tcepi::Tile& b) {
        return p->rp[a.mat] > p->rp[b.mat]; });
    }
    p->t_it_sa = take(sizeof(tcstream::Item) * std::max<size_t>(1, p->it_sa.size()));
    p->t_it_sc = take(sizeof(tcstream::Item) * std::max<size_t>(1, p->it_sc.size()));
    for (int L = 0; L < 3; ++L) {
      p->t_it_tr[L] = take(sizeof(tcstream::Item) * std::max<size_t>(1, p->it_tr[L].size()));
      p->t_it_g[L] = take(sizeof(tcgram::GItem) * std::max<size_t>(1, p->it_g[L].size()));
    }
    p->t_it_epi.resize(p->it_epi.size());
    for (size_t k = 0; k < p->it_epi.size(); ++k)
      p->t_it_epi[k] = take(sizeof(tcepi::Tile) * std::max<size_t>(1, p->it_epi[k].size()));
    for (int L = 0; L < 3; ++L) {
      const size_t nj = lists[L]->size();
      p->chol_order[L].resize(nj);
      for (size_t k = 0; k < nj; ++k) p->chol_order[L][k] = (int)k;
      std::stable_sort(p->chol_order[L].begin(), p->chol_order[L].end(), [&](int a, int b) {
        return D((*lists[L])[a]).r > D((*lists[L])[b]).r; });
      p->t_chol_order[L] = take(4 * std::max<size_t>(1, nj));
    }
    // ranks above 192: Gram jobs and items, transposed splits of A (pass 0) and of T
    for (int L = 0; L < 3; ++L) {
      const size_t nj = std::max<size_t>(1, lists[L]->size());
      for (int ps = 0; ps < 3; ++ps) p->t_gsj[L][ps] = take(sizeof(tcstream::SJob) * nj);
      p->t_it_gs[L] = take(sizeof(tcstream::Item) * std::max<size_t>(1, p->it_gs[L].size()));
      p->t_atj[L] = take(sizeof(tcsplit::TJob) * nj);
      p->t_ttj[L] = take(sizeof(tcsplit::TJob) * nj);
      prefix(p->ts_atj[L], *lists[L], [&](int i) {
        const long long rows = L == 0 ? D(i).m : D(i).n;
        return cdiv(rows, tcsplit::TROWS) * cdiv(p->rp[i], 32); });
      prefix(p->ts_ttj[L], *lists[L],
             [&](int i) { return cdiv(p->rp[i], tcsplit::TROWS) * cdiv(p->rp[i], 32); });
      p->t_ts_atj[L] = take(4 * p->ts_atj[L].size());
      p->t_ts_ttj[L] = take(4 * p->ts_ttj[L].size());
    }
  }
  p->t_sj_a = take(sizeof(tcstream::SJob) * cnt);
  p->t_sj_c = take(sizeof(tcstream::SJob) * cnt);
  p->t_epi = take(sizeof(tcepi::EpiMat) * cnt);
  p->t_split = take(sizeof(tcsplit::SplitJob) * std::max(1, p->n_split));
  p->t_wsplit = take(sizeof(tcsplit::SplitJob) * cnt);
  p->t_ts_wsplit = take(4 * p->ts_wsplit.size());
  p->t_ts_split = take(4 * p->ts_split.size());
  p->t_tj_v = take(sizeof(tcsplit::TJob) * cnt);
  p->t_tj_u = take(sizeof(tcsplit::TJob) * cnt);
  p->t_ts_tv = take(4 * p->ts_tv.size());
  p->t_ts_tu = take(4 * p->ts_tu.size());
  p->t_mats = take(sizeof(MatDev) * cnt);
  p->t_jobs_p = take(sizeof(OrthJob) * cnt);
  p->t_jobs_w = take(sizeof(OrthJob) * std::max<size_t>(1, p->orth_idx.size()));
  p->t_jobs_v = take(sizeof(OrthJob) * std::max<size_t>(1, p->dion_idx.size()));
  p->t_ts_gram_v = take(4 * p->ts_gram_v.size());
  p->t_ts_trmm_v = take(4 * p->ts_trmm_v.size());
  p->t_ts_gram_p = take(4 * p->ts_gram_p.size());
  p->t_ts_trmm_p = take(4 * p->ts_trmm_p.size());
  p->t_ts_wred = take(4 * p->ts_wred.size());
  p->t_ts_gram_w = take(4 * p->ts_gram_w.size());
  p->t_ts_trmm_w = take(4 * p->ts_trmm_w.size());
  p->t_ts_coln = take(4 * p->ts_coln.size());
  p->t_coln_idx = take(4 * std::max<size_t>(1, p->dion_idx.size()));
  p->tables_bytes = off;

  // ---- workspace regions
  size_t ws = 0;
  auto region = [&](size_t bytes) { size_t o = ws; ws = align_up(ws + std::max<size_t>(bytes, 4), kAlign); return o; };
  p->off_tables = region(p->tables_bytes);
  // status words, then the three-pass flags of the orth() of P, W and V
  p->off_status = region(16 * (size_t)cnt);
  p->off_Q2.resize(cnt);
  p->off_P.resize(cnt); p->off_Q.resize(cnt); p->off_U.resize(cnt); p->off_W.resize(cnt);
  p->off_Wpart.resize(cnt); p->off_gpart.resize(cnt); p->off_S.resize(cnt); p->off_T.resize(cnt);
  p->off_Vo.resize(cnt); p->off_gsum.resize(cnt);
  // every W (n x rp, a multiple of 128 bytes) and every reduced Gram of orth(P)
  // (rp x rp) back to back: one exchange region each
  {
    size_t wb = 0, gb = 0;
    for (int i = 0; i < cnt; ++i) {
      wb += 4 * (size_t)(D(i).n * p->rp[i]);
      gb += 4 * (size_t)(p->rp[i] * p->rp[i]);
    }
    p->off_wx = region(wb);
    p->wx_bytes = wb;
    p->off_gx = region(gb);
    p->gx_bytes = gb;
    size_t wo = p->off_wx, go = p->off_gx;
    for (int i = 0; i < cnt; ++i) {
      p->off_W[i] = wo;
      wo += 4 * (size_t)(D(i).n * p->rp[i]);
      p->off_gsum[i] = go;
      go += 4 * (size_t)(p->rp[i] * p->rp[i]);
    }
  }
  for (int i = 0; i < cnt; ++i) {
    const long long m = D(i).m, n = D(i).n, rp = p->rp[i];
    p->off_P[i] = region(4 * (size_t)(m * rp));
    p->off_Q[i] = region(4 * (size_t)(std::max(m, n) * rp));
    p->off_Q2[i] = region(4 * (size_t)(std::max(m, n) * rp));
    p->off_U[i] = region(4 * (size_t)(m * rp));
    p->off_Wpart[i] = region(p->ksplit[i] > 1 ? 4 * (size_t)p->ksplit[i] * (size_t)(n * rp) : 4);
    p->off_gpart[i] = region(4 * (size_t)std::max(p->nchunk_p[i], p->nchunk_w[i]) * (size_t)(rp * rp));
    p->off_S[i] = region(4 * (size_t)(rp * rp + rp + 32 * rp));
    p->off_T[i] = region(4 * (size_t)(rp * rp));
    p->off_Vo[i] = region(D(i).variant == DION_VARIANT_DION ? 4 * (size_t)(n * rp) : 4);
  }
  p->off_Tth.resize(cnt); p->off_Ttl.resize(cnt);
  for (int i = 0; i < cnt; ++i) {
    p->off_Tth[i] = region(4 * (size_t)(p->rp[i] * p->rp[i]));
    p->off_Ttl[i] = region(4 * (size_t)(p->rp[i] * p->rp[i]));
  }
  p->off_VTh.resize(cnt); p->off_VTl.resize(cnt); p->off_UTh.resize(cnt); p->off_UTl.resize(cnt);
  for (int i = 0; i < cnt; ++i) {
    const long long rp = p->rp[i];
    p->off_VTh[i] = region(4 * (size_t)(rp * p->ldt_n[i]));
    p->off_VTl[i] = region(4 * (size_t)(rp * p->ldt_n[i]));
    p->off_UTh[i] = region(4 * (size_t)(rp * p->ldt_m[i]));
    p->off_UTl[i] = region(4 * (size_t)(rp * p->ldt_m[i]));
  }
  p->off_Uh.resize(cnt); p->off_Ul.resize(cnt); p->off_Vh.resize(cnt); p->off_Vl.resize(cnt);
  p->off_Wh.resize(cnt); p->off_Wl.resize(cnt);
  for (int i = 0; i < cnt; ++i) {
    // the update's operand tiles: rows padded to a multiple of 128 (optile_idx)
    const long long m = cdiv(D(i).m, OPT_ROWS) * OPT_ROWS, n = cdiv(D(i).n, OPT_ROWS) * OPT_ROWS, rp = p->rp[i];
    p->off_Uh[i] = region(4 * (size_t)(m * rp));
    p->off_Ul[i] = region(4 * (size_t)(m * rp));
    p->off_Vh[i] = region(4 * (size_t)(n * rp));
    p->off_Vl[i] = region(4 * (size_t)(n * rp));
    p->off_Wh[i] = region(4 * (size_t)(n * rp));
    p->off_Wl[i] = region(4 * (size_t)(n * rp));
  }
  p->ws_bytes = ws;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda link).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  // resolved once per process: a function-local static is initialised by exactly one
  // thread, so host threads creating plans at the same time do not race on it
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(f);
    return nullptr;
  }();
  return fn;
}

// 2-D row-major tensor map: `cols` elements per row (the contiguous dimension),
// `rows` rows `pitch_bytes` apart; box of box_cols x box_rows elements.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, long long cols, long long rows,
              long long pitch_bytes, int box_cols, int box_rows, CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Host check of the work tables that layout() built, before any kernel can use
// them: every output tile of every launch covered exactly once, K ranges that
// tile K without gaps or overlap, and every TMA x coordinate on a 16-byte
// boundary (x * element size % 16 == 0; an unaligned x is an illegal
// instruction on the device).  Returns an empty string or what is wrong.
std::string verify_tables(const dion_plan* p) {
  char buf[256];
  auto bad = [&](const char* what, int i) {
    std::snprintf(buf, sizeof buf, "%s (matrix %d)", what, i);
    return std::string(buf);
  };
  const int cnt = p->count;
  // (a): rows x column blocks, the whole of K; staging x = k (multiple of 16)
  {
    std::vector<std::vector<int>> seen(cnt);
    for (int i = 0; i < cnt; ++i) seen[i].assign(cdiv(p->descs[i].m, tcstream::BM) * p->ncb[i], 0);
    for (const auto& it : p->it_sa) {
      const int i = it.job;
      if (i < 0 || i >= cnt) return bad("phase (a) item of an unknown matrix", i);
      const auto& d = p->descs[i];
      if (it.row0 % tcstream::BM || it.row0 >= d.m || it.c0 % p->bn[i] || it.c0 >= p->rp[i] || it.k0 != 0 ||
          (long long)it.nk * tcstream::BK < d.n || (long long)(it.nk - 1) * tcstream::BK >= d.n)
        return bad("phase (a) item out of range", i);
      if (++seen[i][(it.row0 / tcstream::BM) * p->ncb[i] + it.c0 / p->bn[i]] != 1)
        return bad("phase (a) tile covered twice", i);
    }
    for (int i = 0; i < cnt; ++i)
      for (int v : seen[i]) if (v != 1) return bad("phase (a) tile not covered", i);
  }
  // (c): rows of M^T x K ranges x column blocks; G / R boxes start at x = row0 + 32 b
  // (row0 a multiple of 128), K ranges on multiples of 32
  {
    std::vector<std::vector<int>> seen(cnt);
    for (int i = 0; i < cnt; ++i)
      seen[i].assign(cdiv(p->descs[i].n, tcstream::BM) * p->ksplit[i] * p->ncb[i], 0);
    for (const auto& it : p->it_sc) {
      const int i = it.job;
      if (i < 0 || i >= cnt) return bad("phase (c) item of an unknown matrix", i);
      const auto& d = p->descs[i];
      if (it.row0 % tcstream::BM || it.row0 >= d.n || it.c0 % p->bn[i] || it.c0 >= p->rp[i] ||
          it.ks < 0 || it.ks >= p->ksplit[i] || it.k0 != (long long)it.ks * p->kchunk[i] || it.k0 % 32)
        return bad("phase (c) item out of range", i);
      const long long k1 = std::min<long long>(d.m, (long long)it.k0 + p->kchunk[i]);
      if ((long long)it.nk != cdiv(k1 - it.k0, tcstream::BK)) return bad("phase (c) K range", i);
      if (++seen[i][((it.row0 / tcstream::BM) * p->ksplit[i] + it.ks) * p->ncb[i] + it.c0 / p->bn[i]] != 1)
        return bad("phase (c) tile covered twice", i);
    }
    for (int i = 0; i < cnt; ++i) {
      for (int v : seen[i]) if (v != 1) return bad("phase (c) tile not covered", i);
      if (p->kchunk[i] % 32 || (long long)p->ksplit[i] * p->kchunk[i] < p->descs[i].m ||
          (long long)(p->ksplit[i] - 1) * p->kchunk[i] >= p->descs[i].m)
        return bad("phase (c) K split", i);
    }
  }
  // orth(): A T items cover the rows, Gram items the 256-row chunks, of every job
  {
    const std::vector<int>* lists[3] = {nullptr, &p->orth_idx, &p->dion_idx};
    for (int L = 0; L < 3; ++L) {
      const size_t nj = L == 0 ? (size_t)cnt : lists[L]->size();
      std::vector<std::vector<int>> seen(nj), gseen(nj);
      auto mat = [&](size_t k) { return L == 0 ? (int)k : (*lists[L])[k]; };
      auto rows = [&](size_t k) { return L == 0 ? p->descs[mat(k)].m : p->descs[mat(k)].n; };
      for (size_t k = 0; k < nj; ++k) {
        seen[k].assign(cdiv(rows(k), tcstream::BM) * p->ncb[mat(k)], 0);
        gseen[k].assign(cdiv(rows(k), tcgram::CHUNK_ROWS), 0);
      }
      for (const auto& it : p->it_tr[L]) {
        if (it.job < 0 || (size_t)it.job >= nj) return bad("orth() item of an unknown job", it.job);
        const int i = mat(it.job);
        if (it.row0 % tcstream::BM || it.row0 >= rows(it.job) || it.c0 % p->bn[i] || it.c0 >= p->rp[i] ||
            it.k0 != 0 || (long long)it.nk * tcstream::BK != std::min<long long>(p->rp[i], (long long)it.c0 + p->bn[i]))
          return bad("orth() item out of range", i);
        if (++seen[it.job][(it.row0 / tcstream::BM) * p->ncb[i] + it.c0 / p->bn[i]] != 1)
          return bad("orth() tile covered twice", i);
      }
      for (const auto& g : p->it_g[L]) {
        if (g.job < 0 || (size_t)g.job >= nj || g.chunk < 0 || (size_t)g.chunk >= gseen[g.job].size())
          return bad("Gram item out of range", g.job);
        if (++gseen[g.job][g.chunk] != 1) return bad("Gram chunk covered twice", mat(g.job));
      }
      for (size_t k = 0; k < nj; ++k) {
        for (int v : seen[k]) if (v != 1) return bad("orth() tile not covered", mat(k));
        for (int v : gseen[k]) if (v != 1) return bad("Gram chunk not covered", mat(k));
      }
    }
  }
  // Gram items of ranks above 192 (streaming kernel, transposed mode): rows rp in
  // tiles of 128 x K ranges x column blocks, every K range on a multiple of 256 rows
  for (int L = 0; L < 3 && p->big_orth; ++L) {
    const std::vector<int>* lists[3] = {nullptr, &p->orth_idx, &p->dion_idx};
    const size_t nj = L == 0 ? (size_t)cnt : lists[L]->size();
    auto mat = [&](size_t k) { return L == 0 ? (int)k : (*lists[L])[k]; };
    std::vector<std::vector<int>> seen(nj);
    for (size_t k = 0; k < nj; ++k)
      seen[k].assign(cdiv(p->rp[mat(k)], tcstream::BM) * p->gks[L][k] * p->ncb[mat(k)], 0);
    for (const auto& it : p->it_gs[L]) {
      if (it.job < 0 || (size_t)it.job >= nj) return bad("Gram item of an unknown job", it.job);
      const int i = mat(it.job);
      const long long rows = L == 0 ? p->descs[i].m : p->descs[i].n;
      const int ks = it.ks, ch = p->gkc[L][it.job];
      if (it.row0 % tcstream::BM || it.row0 >= p->rp[i] || it.c0 % p->bn[i] || it.c0 >= p->rp[i] || ks < 0 ||
          ks >= p->gks[L][it.job] || it.k0 != (long long)ks * ch || it.k0 % 256 ||
          (long long)it.nk != cdiv(std::min<long long>(rows, (long long)it.k0 + ch) - it.k0, tcstream::BK))
        return bad("Gram item out of range", i);
      if (++seen[it.job][((it.row0 / tcstream::BM) * p->gks[L][it.job] + ks) * p->ncb[i] + it.c0 / p->bn[i]] != 1)
        return bad("Gram tile covered twice", i);
    }
    for (size_t k = 0; k < nj; ++k) {
      const int i = mat(k);
      for (size_t t = 0; t < seen[k].size(); ++t) {
        const long long r0 = (long long)(t / ((size_t)p->gks[L][k] * p->ncb[i])) * tcstream::BM;
        const long long cb = (long long)(t % p->ncb[i]);
        const int want = r0 >= (cb + 1) * p->bn[i] ? 0 : 1;   // below the diagonal: skipped
        if (seen[k][t] != want) return bad("Gram tile coverage", i);
      }
    }
  }
  // (e): every K pass covers the m x n tiles of exactly the matrices with rp > KPASS * pass
  for (size_t k = 0; k < p->it_epi.size(); ++k) {
    std::vector<std::vector<int>> seen(cnt);
    for (int i = 0; i < cnt; ++i)
      if (p->rp[i] > (long long)k * tcepi::KPASS)
        seen[i].assign(cdiv(p->descs[i].m, tcepi::BM) * cdiv(p->descs[i].n, tcepi::BNJ), 0);
    for (const auto& t : p->it_epi[k]) {
      const int i = t.mat;
      if (i < 0 || i >= cnt || seen[i].empty()) return bad("update tile of a matrix without this K pass", i);
      const auto& d = p->descs[i];
      if (t.i0 % tcepi::BM || t.i0 >= d.m || t.j0 % tcepi::BNJ || t.j0 >= d.n)
        return bad("update tile out of range", i);
      if (++seen[i][(t.i0 / tcepi::BM) * cdiv(d.n, tcepi::BNJ) + t.j0 / tcepi::BNJ] != 1)
        return bad("update tile covered twice", i);
    }
    for (int i = 0; i < cnt; ++i)
      for (int v : seen[i]) if (v != 1) return bad("update tile not covered", i);
  }
  // widths the kernels assume: rp and bn multiples of 32 (fp32 operand boxes of
  // 16 along K, 128-byte Gram boxes), bn within the TMEM budget
  for (int i = 0; i < cnt; ++i)
    if (p->rp[i] % 32 || p->bn[i] % 32 || p->bn[i] > tcstream::BN_MAX || (long long)p->ncb[i] * p->bn[i] < p->rp[i])
      return bad("rank padding or column blocks", i);
  return std::string();
}

dion_status_t build_image(dion_plan* p, unsigned char* base) {
  const int cnt = p->count;
  p->image.assign(p->tables_bytes, 0);
  std::vector<MatDev> mats(cnt);
  std::vector<OrthJob> jp(cnt), jw(std::max<size_t>(1, p->orth_idx.size())),
      jv(std::max<size_t>(1, p->dion_idx.size()));
  unsigned* status = reinterpret_cast<unsigned*>(base + p->off_status);
  for (int i = 0; i < cnt; ++i) {
    const auto& d = p->descs[i];
    MatDev& x = mats[i];
    x.X = d.X; x.G = d.G; x.R = d.R; x.V = d.V;
    // Dion's warm start Vbar = W diag(1/|w_j|) can be far from orthonormal; phase (a)
    // then reads orth(V) instead, which leaves U = orth(M V) unchanged (orth(A T) = orth(A)
    // for T upper triangular with a positive diagonal) and keeps M V well conditioned.
    const bool dn = d.variant == DION_VARIANT_DION;
    x.Vin = dn ? reinterpret_cast<const float*>(base + p->off_Vo[i]) : d.V;
    x.ldvin = dn ? p->rp[i] : d.r;
    x.m = d.m; x.n = d.n; x.r = d.r; x.rp = p->rp[i];
    x.ldx = d.ld_x; x.ldg = d.ld_g; x.ldr = d.ld_r;
    x.g_bf16 = d.g_dtype == DION_DTYPE_BF16;
    x.variant = d.variant;
    const float s = d.scale > 0.f ? d.scale : (float)std::sqrt((double)d.m / (double)d.n);
    x.eta_s = d.eta * s;
    x.beta = d.beta;
    x.mu = d.variant == DION_VARIANT_LOWRANK_MUON ? d.beta : 1.f;
    x.P = reinterpret_cast<float*>(base + p->off_P[i]);
    x.U = reinterpret_cast<float*>(base + p->off_U[i]);
    x.W = reinterpret_cast<float*>(base + p->off_W[i]);
    x.Wpart = reinterpret_cast<float*>(base + p->off_Wpart[i]);
    x.Wh = reinterpret_cast<float*>(base + p->off_Wh[i]);
    x.Wl = reinterpret_cast<float*>(base + p->off_Wl[i]);
    x.ksplit = p->ksplit[i];
    x.kchunk = p->kchunk[i];
    x.status = status + i;
    auto job = [&](OrthJob& o, const float* A, long long rows, float* out, long long ldo,
                   long long ocols, int nch, int ch) {
      o.A = A; o.lda = x.rp;
      o.Q = reinterpret_cast<float*>(base + p->off_Q[i]);
      o.Q2 = reinterpret_cast<float*>(base + p->off_Q2[i]);
      o.out = out; o.ldo = ldo; o.out_cols = ocols;
      o.gpart = reinterpret_cast<float*>(base + p->off_gpart[i]);
      o.gsum = o.gpart;
      o.S = reinterpret_cast<float*>(base + p->off_S[i]);
      o.T = reinterpret_cast<float*>(base + p->off_T[i]);
      o.Tt_hi = reinterpret_cast<float*>(base + p->off_Tth[i]);
      o.Tt_lo = reinterpret_cast<float*>(base + p->off_Ttl[i]);
      o.rows = rows; o.r = x.r; o.rp = x.rp;
      o.nchunk = nch; o.chunk = ch;
      o.status = x.status;
    };
    job(jp[i], x.P, x.m, x.U, x.rp, x.rp, p->nchunk_p[i], p->chunk_p[i]);
    jp[i].flag = status + cnt + i;
    jp[i].gsum = reinterpret_cast<float*>(base + p->off_gsum[i]);   // the exchange region
  }
  for (size_t k = 0; k < p->orth_idx.size(); ++k) {
    const int i = p->orth_idx[k];
    const MatDev& x = mats[i];
    OrthJob& o = jw[k];
    o = jp[i];
    o.gsum = o.gpart;
    o.A = x.W; o.lda = x.rp; o.rows = x.n;
    o.out = x.V; o.ldo = x.r; o.out_cols = x.r;
    o.nchunk = p->nchunk_w[i]; o.chunk = p->chunk_w[i];
    o.flag = status + 2 * cnt + i;
  }
  for (size_t k = 0; k < p->dion_idx.size(); ++k) {
    const int i = p->dion_idx[k];
    const MatDev& x = mats[i];
    OrthJob& o = jv[k];
    o = jp[i];
    o.gsum = o.gpart;
    o.A = x.Vin; o.lda = x.rp; o.rows = x.n;
    o.out = const_cast<float*>(x.Vin); o.ldo = x.rp; o.out_cols = x.rp;
    o.nchunk = p->nchunk_w[i]; o.chunk = p->chunk_w[i];
    o.flag = status + 3 * cnt + i;
  }
  put(p->image, p->t_mats, mats.data(), mats.size());
  put(p->image, p->t_jobs_v, jv.data(), jv.size());
  put(p->image, p->t_ts_gram_v, p->ts_gram_v.data(), p->ts_gram_v.size());
  put(p->image, p->t_ts_trmm_v, p->ts_trmm_v.data(), p->ts_trmm_v.size());
  put(p->image, p->t_jobs_p, jp.data(), jp.size());
  put(p->image, p->t_jobs_w, jw.data(), jw.size());
  put(p->image, p->t_ts_gram_p, p->ts_gram_p.data(), p->ts_gram_p.size());
  put(p->image, p->t_ts_trmm_p, p->ts_trmm_p.data(), p->ts_trmm_p.size());
  put(p->image, p->t_ts_wred, p->ts_wred.data(), p->ts_wred.size());
  put(p->image, p->t_ts_gram_w, p->ts_gram_w.data(), p->ts_gram_w.size());
  put(p->image, p->t_ts_trmm_w, p->ts_trmm_w.data(), p->ts_trmm_w.size());
  put(p->image, p->t_ts_coln, p->ts_coln.data(), p->ts_coln.size());
  if (!p->dion_idx.empty()) put(p->image, p->t_coln_idx, p->dion_idx.data(), p->dion_idx.size());

  // ---- tensor-core phase (e): operand maps (split copies in the workspace) and state maps
  std::vector<tcepi::EpiMat> epi(cnt);
  std::vector<tcsplit::SplitJob> sj(std::max(1, p->n_split));
  const CUtensorMapDataType F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  for (int i = 0; i < cnt; ++i) {
    const auto& d = p->descs[i];
    const MatDev& x = mats[i];
    const long long rp = p->rp[i];
    float* Uh = reinterpret_cast<float*>(base + p->off_Uh[i]);
    float* Ul = reinterpret_cast<float*>(base + p->off_Ul[i]);
    float* Vh = reinterpret_cast<float*>(base + p->off_Vh[i]);
    float* Vl = reinterpret_cast<float*>(base + p->off_Vl[i]);
    float* Wh = reinterpret_cast<float*>(base + p->off_Wh[i]);
    float* Wl = reinterpret_cast<float*>(base + p->off_Wl[i]);
    tcepi::EpiMat& e = epi[i];
    std::memset(&e, 0, sizeof e);
    bool okm = true;
    // the operand halves are read as whole tiles (optile_idx layout) by bulk copies
    e.uh = Uh; e.ul = Ul; e.vh = Vh; e.vl = Vl; e.wh = Wh; e.wl = Wl;
    if (d.g_dtype == DION_DTYPE_BF16)
      okm &= make_map(&e.map[tcepi::MAP_G], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d.G, d.n, d.m, d.ld_g * 2, tcepi::SUB,
                      tcepi::BM, CU_TENSOR_MAP_SWIZZLE_32B);
    else
      okm &= make_map(&e.map[tcepi::MAP_G], F32, d.G, d.n, d.m, d.ld_g * 4, tcepi::SUB, tcepi::BM,
                      CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&e.map[tcepi::MAP_R], F32, d.R, d.n, d.m, d.ld_r * 4, tcepi::SUB, tcepi::BM, CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&e.map[tcepi::MAP_X], F32, d.X, d.n, d.m, d.ld_x * 4, tcepi::SUB, tcepi::BM, CU_TENSOR_MAP_SWIZZLE_64B);
    if (!okm) return fail(DION_ERR_CUDA, "matrix %d: cuTensorMapEncodeTiled failed", i);
    e.m = (int)d.m; e.n = (int)d.n; e.rp = (int)rp; e.g_bf16 = x.g_bf16;
    e.eta_s = x.eta_s; e.beta = x.beta; e.status = x.status;
    // low-rank Muon: M = G + mu R with the descriptor's beta as mu, and R <- M
    const bool momentum = d.variant == DION_VARIANT_LOWRANK_MUON;
    e.mu = x.mu;
    e.gamma = momentum ? 0.f : 1.f;
    if (momentum) e.beta = 1.f;
  }
  // split jobs: U (workspace, ld rp), Vbar (= V after phase (d), ld r)
  for (int k = 0; k < p->n_split; ++k) {
    const int i = p->split_list[k].first;
    const auto& d = p->descs[i];
    const MatDev& x = mats[i];
    const long long rp = p->rp[i];
    if (p->split_list[k].second == 0)
      sj[k] = tcsplit::SplitJob{x.U, rp, reinterpret_cast<float*>(base + p->off_Uh[i]),
                                reinterpret_cast<float*>(base + p->off_Ul[i]), rp, d.m, d.r, x.status, 1};
    else
      sj[k] = tcsplit::SplitJob{d.V, d.r, reinterpret_cast<float*>(base + p->off_Vh[i]),
                                reinterpret_cast<float*>(base + p->off_Vl[i]), rp, d.n, d.r, x.status, 1};
  }
  // ---- tensor-core phases (a) and (c)
  std::vector<tcstream::SJob> sa(cnt), sc(cnt);
  std::vector<tcsplit::TJob> tv(cnt), tu(cnt);
  for (int i = 0; i < cnt; ++i) {
    const auto& d = p->descs[i];
    const MatDev& x = mats[i];
    const long long rp = p->rp[i];
    const bool gb = d.g_dtype == DION_DTYPE_BF16;
    const CUtensorMapDataType gdt = gb ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : F32;
    const long long gpitch = d.ld_g * (gb ? 2 : 4);
    float* VTh = reinterpret_cast<float*>(base + p->off_VTh[i]);
    float* VTl = reinterpret_cast<float*>(base + p->off_VTl[i]);
    float* UTh = reinterpret_cast<float*>(base + p->off_UTh[i]);
    float* UTl = reinterpret_cast<float*>(base + p->off_UTl[i]);
    tcstream::SJob& a = sa[i];
    std::memset(&a, 0, sizeof a);
    bool okm = true;
    // staging boxes of 16 columns (64-byte rows for fp32, 32-byte rows for bf16) and
    // operand boxes of 16 along K (64-byte swizzle)
    okm &= make_map(&a.mG, gdt, d.G, d.n, d.m, gpitch, tcstream::BK, tcstream::BM,
                    gb ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&a.mR, F32, d.R, d.n, d.m, d.ld_r * 4, tcstream::BK, tcstream::BM, CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&a.mBh, F32, VTh, d.n, rp, p->ldt_n[i] * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&a.mBl, F32, VTl, d.n, rp, p->ldt_n[i] * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
    a.out = x.P; a.ld_out = rp; a.split_stride = 0; a.rows = (int)d.m; a.kdim = (int)d.n;
    a.ksplit = 1; a.kchunk = (int)(cdiv(d.n, 32) * 32); a.ncb = p->ncb[i]; a.bn = p->bn[i];
    a.rp = (int)rp; a.gmode = gb ? tcstream::G_BF16 : tcstream::G_F32; a.status = x.status;
    a.pass = -1; a.out_cols = (int)rp;
    a.mu = x.mu;
    tcstream::SJob& c = sc[i];
    std::memset(&c, 0, sizeof c);
    okm &= make_map(&c.mG, gdt, d.G, d.n, d.m, gpitch, gb ? 64 : 32, tcstream::BK, CU_TENSOR_MAP_SWIZZLE_128B);
    okm &= make_map(&c.mR, F32, d.R, d.n, d.m, d.ld_r * 4, 32, tcstream::BK, CU_TENSOR_MAP_SWIZZLE_128B);
    okm &= make_map(&c.mBh, F32, UTh, d.m, rp, p->ldt_m[i] * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
    okm &= make_map(&c.mBl, F32, UTl, d.m, rp, p->ldt_m[i] * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
    if (!okm) return fail(DION_ERR_CUDA, "matrix %d: cuTensorMapEncodeTiled failed (streaming maps)", i);
    c.out = p->ksplit[i] > 1 ? x.Wpart : x.W; c.ld_out = rp; c.split_stride = d.n * rp;
    c.rows = (int)d.n; c.kdim = (int)d.m; c.ksplit = p->ksplit[i]; c.kchunk = p->kchunk[i];
    c.ncb = p->ncb[i]; c.bn = p->bn[i]; c.rp = (int)rp; c.gmode = gb ? tcstream::G_BF16 : tcstream::G_F32;
    c.status = x.status; c.pass = -1; c.out_cols = (int)rp;
    c.mu = x.mu;
    if (p->ksplit[i] == 1) {
      // W written whole by this launch: its halves too (else by the reduction)
      c.sh = x.Wh; c.sl = x.Wl; c.hcols = (int)d.r;
    }
    tv[i] = tcsplit::TJob{x.Vin, x.ldvin, VTh, VTl, p->ldt_n[i], d.n, d.r, rp, x.status};
    tu[i] = tcsplit::TJob{x.U, rp, UTh, UTl, p->ldt_m[i], d.m, d.r, rp, x.status};
  }
  // ---- tensor-core orth(): Gram and A T jobs per list and pass
  if (p->tc_orth) {
    const std::vector<OrthJob>* ojs[3] = {&jp, &jw, &jv};
    const std::vector<int>* lists[3] = {nullptr, &p->orth_idx, &p->dion_idx};
    for (int L = 0; L < 3; ++L) {
      const size_t nj = L == 0 ? (size_t)cnt : lists[L]->size();
      for (int ps = 0; ps < 3; ++ps) {
        std::vector<tcgram::GJob> gj(std::max<size_t>(1, nj));
        std::vector<tcstream::SJob> tj(std::max<size_t>(1, nj));
        for (size_t k = 0; k < nj; ++k) {
          const int i = L == 0 ? (int)k : (*lists[L])[k];
          const OrthJob& o = (*ojs[L])[k];
          const long long rp = p->rp[i];
          const float* src = ps == 0 ? o.A : (ps == 1 ? o.Q : o.Q2);
          const long long lds = ps == 0 ? o.lda : rp;
          tcgram::GJob& g = gj[k];
          std::memset(&g, 0, sizeof g);
          bool okm = make_map(&g.mA, F32, src, rp, o.rows, lds * 4, 32, tcgram::BK, CU_TENSOR_MAP_SWIZZLE_128B);
          g.gpart = o.gpart; g.rows = (int)o.rows; g.rp = (int)rp;
          g.nchunk = (int)cdiv(o.rows, tcgram::CHUNK_ROWS); g.pass = ps; g.flag = o.flag; g.status = o.status;
          tcstream::SJob& t = tj[k];
          std::memset(&t, 0, sizeof t);
          okm &= make_map(&t.mR, F32, src, rp, o.rows, lds * 4, tcstream::BK, tcstream::BM, CU_TENSOR_MAP_SWIZZLE_64B);
          okm &= make_map(&t.mBh, F32, o.Tt_hi, rp, rp, rp * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
          okm &= make_map(&t.mBl, F32, o.Tt_lo, rp, rp, rp * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
          if (!okm) return fail(DION_ERR_CUDA, "matrix %d: cuTensorMapEncodeTiled failed (orth maps)", i);
          t.out = o.out; t.ld_out = o.ldo; t.split_stride = 0; t.q1 = o.Q; t.q2 = o.Q2; t.flag = o.flag;
          t.pass = ps; t.out_cols = (int)o.out_cols; t.rows = (int)o.rows; t.kdim = (int)rp;
          t.ksplit = 1; t.kchunk = (int)rp; t.ncb = p->ncb[i]; t.bn = p->bn[i]; t.rp = (int)rp;
          t.gmode = tcstream::G_NONE; t.status = o.status;
          if (L == 0) {
            // U: halves for the update, transposed halves for W = M^T U
            t.sh = reinterpret_cast<float*>(base + p->off_Uh[i]);
            t.sl = reinterpret_cast<float*>(base + p->off_Ul[i]);
            t.th = reinterpret_cast<float*>(base + p->off_UTh[i]);
            t.tl = reinterpret_cast<float*>(base + p->off_UTl[i]);
            t.ld_t = p->ldt_m[i];
            t.hcols = (int)p->descs[i].r;
            t.tr_fin = 1;
            t.tr_inter = p->big_orth;
          } else {
            if (L == 1) {
              // Orth-Dion Vbar: halves for the update
              t.sh = reinterpret_cast<float*>(base + p->off_Vh[i]);
              t.sl = reinterpret_cast<float*>(base + p->off_Vl[i]);
              t.hcols = (int)p->descs[i].r;
            }
            if (p->big_orth) {
              // transposed halves of the intermediate factors, read by the next pass's
              // Gram: V^T's halves buffers are free while W and V are orthonormalised
              t.th = reinterpret_cast<float*>(base + p->off_VTh[i]);
              t.tl = reinterpret_cast<float*>(base + p->off_VTl[i]);
              t.ld_t = p->ldt_n[i];
              t.hcols = (int)p->descs[i].r;
              t.tr_fin = 0;
              t.tr_inter = 1;
            }
          }
        }
        put(p->image, p->t_gj[L][ps], gj.data(), gj.size());
        put(p->image, p->t_tj[L][ps], tj.data(), tj.size());
      }
      put(p->image, p->t_ts_gred[L], p->ts_gred[L].data(), p->ts_gred[L].size());
    }
    // ranks above 192: Gram jobs of the streaming kernel (transposed mode: output rows
    // = the factor's columns, K = its rows, B = its transposed halves), the split of
    // the pass-0 argument into those halves, and the split of T into T^T halves
    for (int L = 0; L < 3 && p->big_orth; ++L) {
      const size_t nj = L == 0 ? (size_t)cnt : lists[L]->size();
      std::vector<tcsplit::TJob> at(std::max<size_t>(1, nj)), tt(std::max<size_t>(1, nj));
      for (int ps = 0; ps < 3; ++ps) {
        std::vector<tcstream::SJob> gs(std::max<size_t>(1, nj));
        for (size_t k = 0; k < nj; ++k) {
          const int i = L == 0 ? (int)k : (*lists[L])[k];
          const OrthJob& o = (*ojs[L])[k];
          const long long rp = p->rp[i];
          const long long ldt = L == 0 ? p->ldt_m[i] : p->ldt_n[i];
          float* Th = reinterpret_cast<float*>(base + (L == 0 ? p->off_UTh[i] : p->off_VTh[i]));
          float* Tl = reinterpret_cast<float*>(base + (L == 0 ? p->off_UTl[i] : p->off_VTl[i]));
          const float* src = ps == 0 ? o.A : (ps == 1 ? o.Q : o.Q2);
          const long long lds = ps == 0 ? o.lda : rp;
          tcstream::SJob& g = gs[k];
          std::memset(&g, 0, sizeof g);
          bool okm = make_map(&g.mR, F32, src, rp, o.rows, lds * 4, 32, tcstream::BK, CU_TENSOR_MAP_SWIZZLE_128B);
          okm &= make_map(&g.mBh, F32, Th, o.rows, rp, ldt * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
          okm &= make_map(&g.mBl, F32, Tl, o.rows, rp, ldt * 4, tcstream::BK, p->bn[i], CU_TENSOR_MAP_SWIZZLE_64B);
          if (!okm) return fail(DION_ERR_CUDA, "matrix %d: cuTensorMapEncodeTiled failed (Gram maps)", i);
          g.out = o.gpart; g.ld_out = rp; g.split_stride = rp * rp;
          g.flag = o.flag;
          g.pass = ps == 2 ? -2 : -1;   // -2: the Gram of a third (shifted) pass, flagged jobs only
          g.out_cols = (int)rp; g.rows = (int)rp; g.kdim = (int)o.rows;
          g.ksplit = p->gks[L][k]; g.kchunk = p->gkc[L][k]; g.ncb = p->ncb[i]; g.bn = p->bn[i];
          g.rp = (int)rp; g.gmode = tcstream::G_NONE; g.status = o.status; g.mu = 1.f;
          if (ps == 0) {
            at[k] = tcsplit::TJob{o.A, o.lda, Th, Tl, ldt, o.rows, p->descs[i].r, rp, o.status};
            tt[k] = tcsplit::TJob{o.T, rp, o.Tt_hi, o.Tt_lo, rp, rp, rp, rp, o.status};
          }
        }
        put(p->image, p->t_gsj[L][ps], gs.data(), gs.size());
      }
      put(p->image, p->t_atj[L], at.data(), at.size());
      put(p->image, p->t_ttj[L], tt.data(), tt.size());
      put(p->image, p->t_ts_atj[L], p->ts_atj[L].data(), p->ts_atj[L].size());
      put(p->image, p->t_ts_ttj[L], p->ts_ttj[L].data(), p->ts_ttj[L].size());
      if (!p->it_gs[L].empty()) put(p->image, p->t_it_gs[L], p->it_gs[L].data(), p->it_gs[L].size());
    }
    std::vector<tcsplit::SplitJob> vc(std::max<size_t>(1, p->dion_idx.size()));
    for (size_t k = 0; k < p->dion_idx.size(); ++k) {
      const int i = p->dion_idx[k];
      vc[k] = tcsplit::SplitJob{mats[i].V, p->descs[i].r, const_cast<float*>(mats[i].Vin), nullptr, p->rp[i],
                                p->descs[i].n, p->descs[i].r, mats[i].status, 0};
    }
    put(p->image, p->t_vcopy, vc.data(), vc.size());
    put(p->image, p->t_ts_vcopy, p->ts_vcopy.data(), p->ts_vcopy.size());
  }
  if (!p->it_sa.empty()) put(p->image, p->t_it_sa, p->it_sa.data(), p->it_sa.size());
  if (!p->it_sc.empty()) put(p->image, p->t_it_sc, p->it_sc.data(), p->it_sc.size());
  for (int L = 0; L < 3; ++L) {
    if (!p->it_tr[L].empty()) put(p->image, p->t_it_tr[L], p->it_tr[L].data(), p->it_tr[L].size());
    if (!p->it_g[L].empty()) put(p->image, p->t_it_g[L], p->it_g[L].data(), p->it_g[L].size());
  }
  for (size_t k = 0; k < p->it_epi.size(); ++k)
    if (!p->it_epi[k].empty()) put(p->image, p->t_it_epi[k], p->it_epi[k].data(), p->it_epi[k].size());
  for (int L = 0; L < 3; ++L)
    if (!p->chol_order[L].empty()) put(p->image, p->t_chol_order[L], p->chol_order[L].data(), p->chol_order[L].size());
  put(p->image, p->t_sj_a, sa.data(), sa.size());
  put(p->image, p->t_sj_c, sc.data(), sc.size());
  put(p->image, p->t_tj_v, tv.data(), tv.size());
  put(p->image, p->t_tj_u, tu.data(), tu.size());
  put(p->image, p->t_ts_tv, p->ts_tv.data(), p->ts_tv.size());
  put(p->image, p->t_ts_tu, p->ts_tu.data(), p->ts_tu.size());
  put(p->image, p->t_epi, epi.data(), epi.size());
  put(p->image, p->t_split, sj.data(), sj.size());
  put(p->image, p->t_ts_split, p->ts_split.data(), p->ts_split.size());
  {
    std::vector<tcsplit::SplitJob> ws(cnt);
    for (int i = 0; i < cnt; ++i)
      ws[i] = tcsplit::SplitJob{mats[i].W, p->rp[i], mats[i].Wh, mats[i].Wl, p->rp[i], p->descs[i].n,
                                p->descs[i].r, mats[i].status, 1};
    put(p->image, p->t_wsplit, ws.data(), ws.size());
    put(p->image, p->t_ts_wsplit, p->ts_wsplit.data(), p->ts_wsplit.size());
  }
  return DION_OK;
}

dion_status_t check_ws(const dion_plan* p, const void* ws, size_t bytes) {
  if (!p) return fail(DION_ERR_INVALID_ARG, "NULL plan");
  if (!ws) return fail(DION_ERR_WORKSPACE, "NULL workspace");
  if ((uintptr_t)ws % kAlign) return fail(DION_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  if (bytes < p->ws_bytes)
    return fail(DION_ERR_WORKSPACE, "workspace of %zu bytes, plan needs %zu", bytes, p->ws_bytes);
  return DION_OK;
}

dion_status_t cuda_check(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DION_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return DION_OK;
}

template <class T>
const T* tab(const dion_plan* p, unsigned char* base, size_t off) {
  return reinterpret_cast<const T*>(base + p->off_tables + off);
}

// One CholeskyQR pass `ps` of orth() over list L (0: P, 1: W, 2: V) is three
// pieces, kept apart so that the row-sharded step can exchange the Gram between them:
//   orth_gram   the Gram of the pass's argument, summed into each job's gsum
//   orth_chol   Cholesky + inverse of gsum, and T^T's tf32 halves for the tensor core
//   orth_apply  argument T on the tensor core: the next factor, or the result
// Ranks up to 192: tensor-core Gram partials per 256 rows and the one-CTA Cholesky.
// Above 192 (any job of the plan): the Gram on the streaming kernel (transposed mode)
// and the blocked Cholesky of bchol.cuh.  A pass-2 piece only works on jobs whose
// pass 0 took the shifted branch.
struct OrthList {
  const OrthJob* jobs;
  int njob;
};

OrthList orth_list(const dion_plan* p, unsigned char* base, int L) {
  const size_t t = L == 0 ? p->t_jobs_p : (L == 1 ? p->t_jobs_w : p->t_jobs_v);
  const int n = L == 0 ? p->count : (int)(L == 1 ? p->orth_idx.size() : p->dion_idx.size());
  return OrthList{tab<OrthJob>(p, base, t), n};
}

void orth_gram(const dion_plan* p, unsigned char* base, cudaStream_t s, int L, int ps) {
  const OrthList ol = orth_list(p, base, L);
  if (ol.njob == 0) return;
  if (p->big_orth) {
    if (ps == 0)   // the argument's transposed halves (later passes get them from the A T drain)
      tcsplit::k_tsplit<<<p->ts_atj[L][ol.njob], tcsplit::NT, 0, s>>>(
          tab<tcsplit::TJob>(p, base, p->t_atj[L]), tab<int>(p, base, p->t_ts_atj[L]), ol.njob);
    const int ni = (int)p->it_gs[L].size();
    tcstream::k_stream<true><<<std::min(ni, p->num_sms), tcstream::NTHREADS, tcstream::SMEM_BYTES, s>>>(
        tab<tcstream::SJob>(p, base, p->t_gsj[L][ps]), tab<tcstream::Item>(p, base, p->t_it_gs[L]), ni);
  } else {
    const int ng = (int)p->it_g[L].size();
    tcgram::k_gram<<<std::min(ng, p->num_sms), tcgram::NTHREADS, tcgram::SMEM_BYTES, s>>>(
        tab<tcgram::GJob>(p, base, p->t_gj[L][ps]), tab<tcgram::GItem>(p, base, p->t_it_g[L]), ng);
  }
  simt::k_gram_reduce<<<p->ts_gred[L][ol.njob], 256, 0, s>>>(ol.jobs, tab<int>(p, base, p->t_ts_gred[L]),
                                                              ol.njob, ps);
}

void orth_chol(const dion_plan* p, unsigned char* base, cudaStream_t s, int L, int ps) {
  const OrthList ol = orth_list(p, base, L);
  if (ol.njob == 0) return;
  const OrthJob* jobs = ol.jobs;
  const int njob = ol.njob;
  if (!p->big_orth) {
    gj::k_chol_gj<<<njob, gj::NT, gj::SMEM_BYTES, s>>>(jobs, ps, tab<int>(p, base, p->t_chol_order[L]));
    return;
  }
  const long long rmax = p->rmax_l[L];
  long long rpmax = 0;
  for (int k = 0; k < njob; ++k) {
    const int i = L == 0 ? k : (L == 1 ? p->orth_idx[k] : p->dion_idx[k]);
    rpmax = std::max<long long>(rpmax, p->rp[i]);
  }
  const int np = (int)cdiv(rmax, bchol::NB);
  const int ncopy = (int)cdiv(rpmax * rpmax, bchol::COPY_ELEMS);
  auto factor = [&](int retry) {
    bchol::k_stats<<<njob, bchol::NT, 0, s>>>(jobs, ps, retry);
    bchol::k_copy<<<njob * ncopy, bchol::NT, 0, s>>>(jobs, ps, retry, ncopy);
    for (int pp = 0; pp < np; ++pp) {
      bchol::k_diag_gj<<<njob, gj::NT, gj::SMEM_BYTES, s>>>(jobs, ps, retry, pp);
      const long long trail = rmax - (long long)(pp + 1) * bchol::NB;   // columns right of the panel
      if (trail <= 0) continue;
      const int nslab = (int)cdiv(trail, bchol::SLAB);
      const int tdim = (int)cdiv(trail, simt::TM);
      bchol::k_panel<<<njob * nslab, bchol::NT, bchol::PANEL_SMEM, s>>>(jobs, ps, retry, pp, nslab);
      bchol::k_update<<<njob * (tdim * (tdim + 1) / 2), simt::NT, 0, s>>>(jobs, ps, retry, pp,
                                                                          tdim * (tdim + 1) / 2);
    }
    bchol::k_check<<<(int)cdiv(njob, 128), 128, 0, s>>>(jobs, njob, ps, retry);
  };
  factor(0);
  if (ps == 0) factor(1);   // the shifted repetition, for the jobs whose pivots asked for it
  // off-diagonal blocks of T by recursive doubling: two launches per level
  for (int lv = 0; ((long long)bchol::NB << lv) < rmax; ++lv) {
    const long long sz = (long long)bchol::NB << lv, tps = sz / simt::TM;
    const int ntile = (int)(cdiv(rmax, 2 * sz) * tps * tps);
    for (int step = 0; step < 2; ++step)
      bchol::k_inv_pairs<<<njob * ntile, simt::NT, 0, s>>>(jobs, ps, lv, step, ntile);
  }
  tcsplit::k_tsplit<<<p->ts_ttj[L][njob], tcsplit::NT, 0, s>>>(tab<tcsplit::TJob>(p, base, p->t_ttj[L]),
                                                               tab<int>(p, base, p->t_ts_ttj[L]), njob);
}

void orth_apply(const dion_plan* p, unsigned char* base, cudaStream_t s, int L, int ps) {
  const OrthList ol = orth_list(p, base, L);
  if (ol.njob == 0) return;
  const int nt = (int)p->it_tr[L].size();
  tcstream::k_stream<false><<<std::min(nt, p->num_sms), tcstream::NTHREADS, tcstream::SMEM_BYTES, s>>>(
      tab<tcstream::SJob>(p, base, p->t_tj[L][ps]), tab<tcstream::Item>(p, base, p->t_it_tr[L]), nt);
}

// orth() of every job of list L: up to three CholeskyQR passes.
dion_status_t launch_orth(const dion_plan* p, unsigned char* base, cudaStream_t s, int L) {
  for (int ps = 0; ps < 3; ++ps) {
    orth_gram(p, base, s, L, ps);
    orth_chol(p, base, s, L, ps);
    orth_apply(p, base, s, L, ps);
  }
  return cuda_check("orth launch");
}

// Kernel launches of launch_orth(L) (a pass-2 launch returns at once for jobs
// without the shifted branch).
int orth_launches(const dion_plan* p, int L) {
  const int njob = L == 0 ? p->count : (int)(L == 1 ? p->orth_idx.size() : p->dion_idx.size());
  if (njob == 0) return 0;
  if (!p->big_orth) return 3 * 4;
  const int np = (int)cdiv(p->rmax_l[L], bchol::NB);
  int fac = 2 + 1;                                       // stats, copy, check
  for (int pp = 0; pp < np; ++pp) fac += (p->rmax_l[L] > (long long)(pp + 1) * bchol::NB) ? 3 : 1;
  int lv = 0;
  while (((long long)bchol::NB << lv) < p->rmax_l[L]) ++lv;
  const int chol = fac + 2 * lv + 1;                     // + inverse levels (two launches each) + T^T split
  return 3 * (2 + chol + 1) + 1 + fac;                   // gram + reduce, chol, apply; pass-0 split and repetition
}

dion_status_t run_phases(dion_plan* p, void* workspace, size_t ws_bytes, int first, int last,
                         void* stream) {
  dion_status_t st = check_ws(p, workspace, ws_bytes);
  if (st) return st;
  if (first < 0 || last > 4 || first > last)
    return fail(DION_ERR_INVALID_ARG, "phase range %d..%d outside 0..4", first, last);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  if (p->dirty || p->uploaded_ws != workspace) {
    st = dion_plan_upload(p, workspace, ws_bytes, stream);
    if (st) return st;
  }
  const MatDev* mats = tab<MatDev>(p, base, p->t_mats);
  const int cnt = p->count;
  // one NVTX range per phase, so that timeline tools show the step's structure
  static const char* const kPhaseNames[5] = {
      "dion (a) P = (G + R) V", "dion (b) U = orth(P)", "dion (c) W = (G + R)^T U",
      "dion (d) Vbar = orth(W) | colnorm(W)", "dion (e) X, R update"};
  struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
  };
  for (int ph = first; ph <= last; ++ph) {
    const Range range(kPhaseNames[ph]);
    switch (ph) {
      case 0:
        if (cudaMemsetAsync(base + p->off_status, 0, 16 * (size_t)cnt, s) != cudaSuccess)
          return cuda_check("status reset");
        if (!p->dion_idx.empty()) {
          // Dion's warm start: a padded copy of V, orthonormalised (orth(M V) = orth(M orth(V)))
          tcsplit::k_split<<<p->ts_vcopy[p->dion_idx.size()], tcsplit::NT, 0, s>>>(
              tab<tcsplit::SplitJob>(p, base, p->t_vcopy), tab<int>(p, base, p->t_ts_vcopy),
              (int)p->dion_idx.size());
          st = launch_orth(p, base, s, 2);
          if (st) return st;
        }
        tcsplit::k_tsplit<<<p->ts_tv[cnt], tcsplit::NT, 0, s>>>(
            tab<tcsplit::TJob>(p, base, p->t_tj_v), tab<int>(p, base, p->t_ts_tv), cnt);
        tcstream::k_stream<false><<<std::min((int)p->it_sa.size(), p->num_sms), tcstream::NTHREADS,
                                    tcstream::SMEM_BYTES, s>>>(tab<tcstream::SJob>(p, base, p->t_sj_a),
                                                               tab<tcstream::Item>(p, base, p->t_it_sa),
                                                               (int)p->it_sa.size());
        break;
      case 1:
        st = launch_orth(p, base, s, 0);
        if (st) return st;
        break;
      case 2:
        // (the last A T pass of orth(P) wrote U^T's halves)
        tcstream::k_stream<true><<<std::min((int)p->it_sc.size(), p->num_sms), tcstream::NTHREADS,
                                   tcstream::SMEM_BYTES, s>>>(tab<tcstream::SJob>(p, base, p->t_sj_c),
                                                              tab<tcstream::Item>(p, base, p->t_it_sc),
                                                              (int)p->it_sc.size());
        if (p->any_split)
          simt::k_wreduce<<<p->ts_wred[cnt], simt::NT, 0, s>>>(mats, tab<int>(p, base, p->t_ts_wred), cnt);
        break;
      case 3:
        st = launch_orth(p, base, s, 1);
        if (st) return st;
        if (!p->dion_idx.empty())
          simt::k_colnorm<<<p->ts_coln[p->dion_idx.size()], simt::NT, 0, s>>>(
              mats, tab<int>(p, base, p->t_ts_coln), tab<int>(p, base, p->t_coln_idx),
              (int)p->dion_idx.size());
        // tf32 halves of the update's operands that no earlier kernel wrote
        if (p->n_split > 0)
          tcsplit::k_split<<<p->ts_split[p->n_split], tcsplit::NT, 0, s>>>(
              tab<tcsplit::SplitJob>(p, base, p->t_split), tab<int>(p, base, p->t_ts_split), p->n_split);
        break;
      case 4: {
        // one launch per K pass (K <= KPASS accumulated in TMEM per launch); three slots
        // of streamed state also with bf16 gradients (measured: 4 slots 12.85, 3 slots
        // 12.48, 2 slots 14.85 ms on the Llama-3B update)
        for (size_t k = 0; k < p->it_epi.size(); ++k) {
          const int tiles = (int)p->it_epi[k].size();
          const int grid = std::min(tiles, p->num_sms);
          tcepi::k_epi<<<grid, tcepi::NTHREADS, tcepi::SMEM_BYTES, s>>>(
              tab<tcepi::EpiMat>(p, base, p->t_epi), tab<tcepi::Tile>(p, base, p->t_it_epi[k]), tiles,
              p->any_g_f32 ? 24576 : 20480, 3, (int)k);
        }
        break;
      }
    }
    st = cuda_check("phase launch");
    if (st) return st;
  }
  return ok();
}

// ---- row-sharded step: the step of phases (a)-(e) cut at its three exchange points
//
// A rank holds rows of X, G and R (V replicated).  P's rows are local, but orth(P)
// needs the Gram P^T P of all rows, and W = M^T U sums over all rows; so the
// step stops after every Gram of orth(P)'s CholeskyQR passes (the reduced Grams in
// the exchange region, all-reduced by the caller between stages) and after the
// local W (the W region).  Stage k:
//   0  status reset, orth(V) (Dion), P = M V, Gram of P (pass 0)
//   1  Cholesky + inverse of the exchanged Gram, Q1 = P T, Gram of Q1 (pass 1)
//   2  Cholesky + inverse, U = Q1 T2 (or Q2 for a shifted job), Gram of Q2 (shifted jobs)
//   3  Cholesky + inverse and U = Q2 T3 (shifted jobs), W = M^T U over the local rows
//   4  W's tf32 halves from the exchanged W, Vbar = orth(W) | colnorm(W), X and R update
// Every rank computes the same Cholesky factors and Vbar from the same exchanged
// data (the kernels are deterministic), and the shifted-pass decision with them.
dion_status_t run_shard_stage(dion_plan* p, void* workspace, size_t ws_bytes, int stage, void* stream) {
  dion_status_t st = check_ws(p, workspace, ws_bytes);
  if (st) return st;
  if (stage < 0 || stage > 4) return fail(DION_ERR_INVALID_ARG, "shard stage %d outside 0..4", stage);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned char* base = static_cast<unsigned char*>(workspace);
  if (p->dirty || p->uploaded_ws != workspace) {
    st = dion_plan_upload(p, workspace, ws_bytes, stream);
    if (st) return st;
  }
  const int cnt = p->count;
  const MatDev* mats = tab<MatDev>(p, base, p->t_mats);
  switch (stage) {
    case 0: {
      // phase (a) as in the fused step, then the first Gram into the exchange region
      st = run_phases(p, workspace, ws_bytes, 0, 0, stream);
      if (st) return st;
      orth_gram(p, base, s, 0, 0);
      break;
    }
    case 1:
    case 2:
      orth_chol(p, base, s, 0, stage - 1);
      orth_apply(p, base, s, 0, stage - 1);
      orth_gram(p, base, s, 0, stage);
      break;
    case 3:
      orth_chol(p, base, s, 0, 2);
      orth_apply(p, base, s, 0, 2);
      tcstream::k_stream<true><<<std::min((int)p->it_sc.size(), p->num_sms), tcstream::NTHREADS,
                                 tcstream::SMEM_BYTES, s>>>(tab<tcstream::SJob>(p, base, p->t_sj_c),
                                                            tab<tcstream::Item>(p, base, p->t_it_sc),
                                                            (int)p->it_sc.size());
      if (p->any_split)
        simt::k_wreduce<<<p->ts_wred[cnt], simt::NT, 0, s>>>(mats, tab<int>(p, base, p->t_ts_wred), cnt);
      break;
    case 4:
      tcsplit::k_split<<<p->ts_wsplit[cnt], tcsplit::NT, 0, s>>>(
          tab<tcsplit::SplitJob>(p, base, p->t_wsplit), tab<int>(p, base, p->t_ts_wsplit), cnt);
      st = cuda_check("shard stage launch");
      if (st) return st;
      return run_phases(p, workspace, ws_bytes, 3, 4, stream);
  }
  st = cuda_check("shard stage launch");
  if (st) return st;
  return ok();
}

// ---- dion_orth_noalloc: one orth() on the CUDA-core kernels, scratch in g_noalloc_scratch

// Writes the job and its launch tables into the scratch and clears the status
// and three-pass flag (kernel arguments carry them, so no host buffer is read
// after the call returns).
__global__ void k_noalloc_setup(OrthJob job, int ngram, int ntrmm, unsigned char* base) {
  if (threadIdx.x == 0) {
    *reinterpret_cast<OrthJob*>(base) = job;
    int* ts = reinterpret_cast<int*>(base + 256);
    ts[0] = 0; ts[1] = ngram; ts[2] = 0; ts[3] = ntrmm;
    *job.status = 0u;
    *job.flag = 0u;
  }
}

dion_status_t orth_noalloc_impl(const float* A, long long rows, long long r, long long lda, float* Q, long long ldq,
                                uint32_t* status_out, void* stream) {
  if (!A || !Q) return fail(DION_ERR_INVALID_ARG, "NULL matrix pointer");
  if (rows < 1 || r < 1 || r > rows) return fail(DION_ERR_INVALID_ARG, "need 1 <= r <= rows");
  if (lda < r || ldq < r) return fail(DION_ERR_INVALID_ARG, "leading dimension below r");
  if (rows > noalloc::kRowsMax || r > noalloc::kRankMax)
    return fail(DION_ERR_UNSUPPORTED, "%lld x %lld exceeds the fixed scratch (rows <= %d, r <= %d)", rows, r,
                DION_NOALLOC_MAX_ROWS, DION_NOALLOC_MAX_RANK);
  // Device address of the scratch, looked up once per device with that device
  // current.  Host threads may race on a first call: each entry is an atomic, and a
  // second lookup of the same device stores the same address.  The cache is not
  // refreshed after cudaDeviceReset().
  static std::atomic<void*> dev_ptr[noalloc::kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_check("device query");
  if (dev < 0 || dev >= noalloc::kMaxDevices)
    return fail(DION_ERR_UNSUPPORTED, "device %d: the scratch address cache covers devices 0..%d", dev,
                noalloc::kMaxDevices - 1);
  void* cached = dev_ptr[dev].load(std::memory_order_acquire);
  if (!cached) {
    if (cudaGetSymbolAddress(&cached, g_noalloc_scratch) != cudaSuccess || !cached)
      return cuda_check("scratch address lookup");
    dev_ptr[dev].store(cached, std::memory_order_release);
  }
  unsigned char* base = static_cast<unsigned char*>(cached);
  const long long rp = cdiv(r, kRankGranule) * kRankGranule;
  long long nch = std::min<long long>(noalloc::kChunksMax, std::max<long long>(1, cdiv(rows, 512)));
  const long long chunk = cdiv(cdiv(rows, nch), 64) * 64;
  nch = cdiv(rows, chunk);
  float* fbase = reinterpret_cast<float*>(base + noalloc::kJobBytes);
  OrthJob job;
  std::memset(&job, 0, sizeof job);
  job.A = A; job.lda = lda;
  job.gpart = fbase;
  job.S = job.gpart + noalloc::kGpartFloats;
  job.T = job.S + noalloc::kSFloats;
  job.Q = job.T + noalloc::kTFloats;
  job.Q2 = job.Q + noalloc::kQFloats;
  job.out = Q; job.ldo = ldq; job.out_cols = r;
  job.rows = rows; job.r = r; job.rp = rp;
  job.nchunk = (int)nch; job.chunk = (int)chunk;
  job.status = reinterpret_cast<unsigned*>(base + 256 + 32);
  job.flag = job.status + 1;
  job.Tt_hi = job.Tt_lo = nullptr;
  job.gsum = job.gpart;
  const long long nt = cdiv(rp, simt::TN);
  const int ngram = (int)(nch * nt * nt);
  const int ntrmm = (int)(cdiv(rows, simt::TM) * nt);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  k_noalloc_setup<<<1, 32, 0, s>>>(job, ngram, ntrmm, base);
  const OrthJob* jobs = reinterpret_cast<const OrthJob*>(base);
  const int* tg = reinterpret_cast<const int*>(base + 256);
  const int* tt = tg + 2;
  const size_t chol_smem = (size_t)((r * (r + 1) + r + 32 * r) * 4);   // <= 25 KB at r = 64
  for (int pass = 0; pass < 3; ++pass) {
    simt::k_gram<<<ngram, simt::NT, 0, s>>>(jobs, tg, 1, pass);
    simt::k_chol_inv<true><<<1, simt::CHOL_NT, chol_smem, s>>>(jobs, pass, 0, nullptr);
    simt::k_trmm<<<ntrmm, simt::NT, 0, s>>>(jobs, tt, 1, pass);
  }
  dion_status_t st = cuda_check("orth launch");
  if (st) return st;
  if (status_out) {
    if (cudaMemcpyAsync(status_out, job.status, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return cuda_check("status copy");
    if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_check("status sync");
  }
  return ok();
}

}  // namespace

extern "C" {

int32_t dion_abi_version(void) { return DION_ABI_VERSION; }

const char* dion_status_string(dion_status_t s) {
  switch (s) {
    case DION_OK: return "DION_OK";
    case DION_ERR_INVALID_ARG: return "DION_ERR_INVALID_ARG";
    case DION_ERR_CUDA: return "DION_ERR_CUDA";
    case DION_ERR_WORKSPACE: return "DION_ERR_WORKSPACE";
    case DION_ERR_UNSUPPORTED: return "DION_ERR_UNSUPPORTED";
  }
  return "DION_ERR_UNKNOWN";
}

const char* dion_last_error(void) { return g_err.c_str(); }

dion_status_t dion_plan_create(const dion_matrix_desc* descs, int32_t count, size_t* workspace_bytes,
                               dion_plan** out) {
  if (!descs || !workspace_bytes || !out) return fail(DION_ERR_INVALID_ARG, "NULL argument");
  *out = nullptr;
  if (count < 1 || count > (1 << 20)) return fail(DION_ERR_INVALID_ARG, "count %d outside [1, 2^20]", count);
  dion_status_t st = validate(descs, count);
  if (st) return st;
  dion_plan* p = new dion_plan();
  p->descs.assign(descs, descs + count);
  p->count = count;
  layout(p);
  const std::string wrong = verify_tables(p);
  if (!wrong.empty()) {
    delete p;
    return fail(DION_ERR_UNSUPPORTED, "internal: work tables failed their check: %s", wrong.c_str());
  }
  // every grouped launch must fit in one grid dimension
  const long long grids[] = {p->ts_wred[count], p->ts_split[p->n_split], p->ts_tv[count], p->ts_wsplit[count],
                             p->ts_atj[0].empty() ? 0 : p->ts_atj[0].back()};
  for (long long g : grids)
    if (g >= (1LL << 31)) {
      delete p;
      return fail(DION_ERR_UNSUPPORTED, "batch too large for one grouped launch");
    }
  *workspace_bytes = p->ws_bytes;
  *out = p;
  return ok();
}

void dion_plan_destroy(dion_plan* plan) { delete plan; }

int32_t dion_plan_count(const dion_plan* plan) { return plan ? plan->count : -1; }

dion_status_t dion_plan_set_hparams(dion_plan* plan, int32_t idx, float eta, float beta) {
  if (!plan) return fail(DION_ERR_INVALID_ARG, "NULL plan");
  if (idx < 0 || idx >= plan->count) return fail(DION_ERR_INVALID_ARG, "index %d outside the plan", idx);
  if (!std::isfinite(eta) || !std::isfinite(beta)) return fail(DION_ERR_INVALID_ARG, "non-finite eta / beta");
  plan->descs[idx].eta = eta;
  plan->descs[idx].beta = beta;
  plan->dirty = true;
  return ok();
}

dion_status_t dion_plan_upload(dion_plan* plan, void* workspace, size_t ws_bytes, void* stream) {
  dion_status_t st = check_ws(plan, workspace, ws_bytes);
  if (st) return st;
  unsigned char* base = static_cast<unsigned char*>(workspace);
  if (plan->num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&plan->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return cuda_check("device query");
    if (cudaFuncSetAttribute(tcepi::k_epi, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tcepi::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(tcstream::k_stream<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tcstream::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(tcstream::k_stream<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tcstream::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(simt::k_chol_inv<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             simt::CHOL_SMEM_MAX) != cudaSuccess ||
        cudaFuncSetAttribute(tcgram::k_gram, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tcgram::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(bchol::k_panel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bchol::PANEL_SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(gj::k_chol_gj, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gj::SMEM_BYTES) != cudaSuccess ||
        cudaFuncSetAttribute(bchol::k_diag_gj, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)gj::SMEM_BYTES) != cudaSuccess)
      return cuda_check("kernel attributes");
  }
  st = build_image(plan, base);
  if (st) return st;
  if (cudaMemcpyAsync(base + plan->off_tables, plan->image.data(), plan->image.size(),
                      cudaMemcpyHostToDevice, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_check("table upload");
  plan->uploaded_ws = workspace;
  plan->dirty = false;
  return ok();
}

dion_status_t dion_step_batched(dion_plan* plan, void* workspace, size_t ws_bytes, void* stream) {
  return run_phases(plan, workspace, ws_bytes, 0, 4, stream);
}

dion_status_t dion_step_phases(dion_plan* plan, void* workspace, size_t ws_bytes, int32_t first,
                               int32_t last, void* stream) {
  return run_phases(plan, workspace, ws_bytes, first, last, stream);
}

dion_status_t dion_plan_buffer(const dion_plan* plan, int32_t idx, int32_t which, size_t* byte_offset,
                               int64_t* rows, int64_t* cols, int64_t* ld) {
  if (!plan || !byte_offset || !rows || !cols || !ld) return fail(DION_ERR_INVALID_ARG, "NULL argument");
  if (idx < 0 || idx >= plan->count) return fail(DION_ERR_INVALID_ARG, "index %d outside the plan", idx);
  const auto& d = plan->descs[idx];
  *cols = d.r;
  *ld = plan->rp[idx];
  switch (which) {
    case DION_BUF_P: *byte_offset = plan->off_P[idx]; *rows = d.m; break;
    case DION_BUF_U: *byte_offset = plan->off_U[idx]; *rows = d.m; break;
    case DION_BUF_W: *byte_offset = plan->off_W[idx]; *rows = d.n; break;
    default: return fail(DION_ERR_INVALID_ARG, "unknown buffer %d", which);
  }
  return ok();
}

dion_status_t dion_plan_get_status(dion_plan* plan, const void* workspace, size_t ws_bytes,
                                   uint32_t* per_matrix, void* stream) {
  dion_status_t st = check_ws(plan, workspace, ws_bytes);
  if (st) return st;
  if (!per_matrix) return fail(DION_ERR_INVALID_ARG, "NULL output");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned char* base = static_cast<const unsigned char*>(workspace);
  if (cudaMemcpyAsync(per_matrix, base + plan->off_status, 4 * (size_t)plan->count,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return cuda_check("status copy");
  if (cudaStreamSynchronize(s) != cudaSuccess) return cuda_check("status sync");
  return ok();
}

int32_t dion_plan_launches_per_step(const dion_plan* plan) {
  if (!plan) return -1;
  int n = 2;                                           // phase (a): V^T split + tensor-core P = M V
  if (!plan->dion_idx.empty()) n += 1 + orth_launches(plan, 2);   // phase (a): copy + orth(V) of Dion matrices
  n += orth_launches(plan, 0);                         // phase (b)
  n += 1 + (plan->any_split ? 1 : 0);                  // phase (c): W = M^T U, reduce
  n += orth_launches(plan, 1);                         // phase (d), Orth-Dion matrices
  n += plan->dion_idx.empty() ? 0 : 1;                 // phase (d), Dion matrices
  n += plan->n_split > 0 ? 1 : 0;                      // phase (d): tf32 halves left to split
  n += (int)plan->it_epi.size();                       // phase (e): tensor-core update, one launch per K pass
  return n;
}

dion_status_t dion_debug_expire_wait(int64_t limit_ns, int32_t withhold_matrix, void* stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const unsigned long long lim = limit_ns > 0 ? (unsigned long long)limit_ns : tc::kWaitNs;
  const int wm = withhold_matrix >= 0 ? withhold_matrix : -1;
  if (cudaMemcpyToSymbolAsync(tc::g_wait_limit_ns, &lim, sizeof lim, 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(tcepi::g_withhold_epi_matrix, &wm, sizeof wm, 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return cuda_check("debug hook");
  return ok();
}

dion_status_t dion_shard_stage(dion_plan* plan, void* workspace, size_t ws_bytes, int32_t stage, void* stream) {
  return run_shard_stage(plan, workspace, ws_bytes, stage, stream);
}

dion_status_t dion_plan_exchange(const dion_plan* plan, int32_t which, size_t* byte_offset, size_t* bytes) {
  if (!plan || !byte_offset || !bytes) return fail(DION_ERR_INVALID_ARG, "NULL argument");
  switch (which) {
    case DION_EXCHANGE_GRAM: *byte_offset = plan->off_gx; *bytes = plan->gx_bytes; break;
    case DION_EXCHANGE_W: *byte_offset = plan->off_wx; *bytes = plan->wx_bytes; break;
    default: return fail(DION_ERR_INVALID_ARG, "unknown exchange region %d", which);
  }
  return ok();
}

dion_status_t dion_orth_noalloc(const float* A, int64_t rows, int64_t r, int64_t lda, float* Q, int64_t ldq,
                                uint32_t* status, void* stream) {
  return orth_noalloc_impl(A, rows, r, lda, Q, ldq, status, stream);
}

}  // extern "C"
