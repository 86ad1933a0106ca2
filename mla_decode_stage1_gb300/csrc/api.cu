// api.cu -- host side of libmla_decode: argument validation, the work
// planner, workspace layout, TMA descriptor set-up and the kernel launches.
// The C declarations and their contracts are in include/mla_decode.h.

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "mla_decode.h"
#include "kernels.h"
#include "plan.h"

using mla::MergeJob;
using mla::WorkItem;
using mla::CtaHead;


namespace {

constexpr size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }


int qmode_of(int q_dtype, int kv_dtype) {
  if (q_dtype == MLA_DTYPE_BF16 && kv_dtype == MLA_DTYPE_BF16) return mla::kQBf16KvBf16;
  if (q_dtype == MLA_DTYPE_FP8_E4M3 && kv_dtype == MLA_DTYPE_FP8_E4M3) return mla::kQFp8KvFp8;
  if (q_dtype == MLA_DTYPE_BF16 && kv_dtype == MLA_DTYPE_FP8_E4M3) return mla::kQBf16KvFp8;
  if (q_dtype == MLA_DTYPE_FP8_E4M3 && kv_dtype == MLA_DTYPE_BF16) return mla::kQFp8KvBf16;
  if (q_dtype == MLA_DTYPE_BF16 && kv_dtype == MLA_DTYPE_MXFP4) return mla::kQBf16KvMx;
  return -1;
}

// Items of the balanced plan over the requests listed in `order`: their
// units (`unit` tokens each, a whole 128-token tile by default), in that
// order, cut into at most G contiguous ranges, one per CTA, appended to the
// plan.  A range costs 2 per unit plus kItemCost for every item past its
// first: an item boundary inside a CTA (an epilogue before the next item's
// first tile) costs about half a tile period by default.  The smallest
// maximum cost that G greedy ranges reach is found by bisection.
void plan_balanced(mla_plan* P, const std::vector<int32_t>& order, const std::vector<int64_t>& tiles,
                   const std::vector<int32_t>& len, const std::vector<int32_t>& page_base,
                   const std::vector<int32_t>& npages, int32_t G, int64_t kItemCost,
                   int32_t unit) {
  int64_t T = 0;
  for (const int32_t r : order) T += tiles[r];
  if (G > T) G = static_cast<int32_t>(T);
  if (G <= 0) return;
  // Greedy cut under a cost cap: each range takes tiles while its cost stays
  // within `cap` (a range always takes at least one tile).  Calls emit(k,
  // first tile, tiles taken, range index) per item and returns the ranges.
  auto cut = [&](int64_t cap, auto&& emit) {
    int32_t ranges = 0;
    size_t k = 0;
    int64_t in_req = 0;
    while (true) {
      while (k < order.size() && tiles[order[k]] - in_req == 0) { ++k; in_req = 0; }
      if (k == order.size()) break;
      int64_t cost = 0;
      bool any = false;
      while (k < order.size()) {
        const int64_t left = tiles[order[k]] - in_req;
        if (left == 0) { ++k; in_req = 0; continue; }
        const int64_t item = any ? kItemCost : 0;
        int64_t take = (cap - cost - item) / 2;
        if (take <= 0) {
          if (any) break;
          take = 1;
        }
        take = std::min(take, left);
        emit(order[k], in_req, take, ranges);
        cost += 2 * take + item;
        any = true;
        in_req += take;
        if (in_req < tiles[order[k]]) break;   // cap reached inside this request
      }
      ++ranges;
    }
    return ranges;
  };
  auto none = [](int32_t, int64_t, int64_t, int32_t) {};
  // Bisection for the smallest cap whose greedy cut needs at most G ranges.
  // Upper bound: the largest cost among the G ranges of the plain equal split
  // of the tiles.  That split meets its own largest cost with G ranges, and a
  // greedy cut under a cap needs the fewest ranges of any contiguous cut, so
  // the bound is feasible and the search spans a few units, not 2T.
  std::vector<int64_t> cum(order.size() + 1, 0);   // tiles before order[k]
  std::vector<int32_t> nz(order.size() + 1, 0);    // requests with tiles before order[k]
  for (size_t k = 0; k < order.size(); ++k) {
    cum[k + 1] = cum[k] + tiles[order[k]];
    nz[k + 1] = nz[k] + (tiles[order[k]] > 0 ? 1 : 0);
  }
  auto holder = [&](int64_t x) {                   // the request holding tile x
    return static_cast<size_t>(std::upper_bound(cum.begin(), cum.end(), x) - cum.begin()) - 1;
  };
  int64_t hi = 2;
  for (int32_t i = 0; i < G; ++i) {
    const int64_t a = T * i / G, b = T * (i + 1) / G;
    if (b <= a) continue;
    const int64_t items = nz[holder(b - 1) + 1] - nz[holder(a)];
    hi = std::max(hi, 2 * (b - a) + kItemCost * (items - 1));
  }
  int64_t lo = std::min<int64_t>((2 * T + G - 1) / G, hi);
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (cut(mid, none) <= G) hi = mid; else lo = mid + 1;
  }
  int32_t last = -1;
  const int32_t used = cut(lo, [&](int32_t b, int64_t t0, int64_t take, int32_t range) {
    if (range != last) {
      if (last >= 0) P->cta_indptr.push_back(static_cast<int32_t>(P->items.size()));
      last = range;
    }
    WorkItem w{};
    w.b = b;
    w.tok_begin = static_cast<int32_t>(t0 * unit);
    w.tok_end = static_cast<int32_t>(std::min<int64_t>((t0 + take) * unit, len[b]));
    w.slot = 0;
    w.page_base = page_base[b];
    w.npages = npages[b];
    P->items.push_back(w);
  });
  P->cta_indptr.push_back(static_cast<int32_t>(P->items.size()));
  P->num_ctas += used;
}

// Items of the fixed-split plan: request b cut into S ranges of
// ceil(units_b / S) units; one CTA per non-empty range.
void plan_fixed(mla_plan* P, const std::vector<int64_t>& tiles, const std::vector<int32_t>& len,
                const std::vector<int32_t>& page_base, const std::vector<int32_t>& npages,
                int32_t S, int32_t unit) {
  P->cta_indptr.assign(1, 0);
  for (int32_t b = 0; b < P->bs; ++b) {
    const int64_t per = (tiles[b] + S - 1) / S;
    for (int32_t s = 0; s < S && per > 0; ++s) {
      const int64_t t0 = per * s, t1 = std::min<int64_t>(per * (s + 1), tiles[b]);
      if (t1 <= t0) continue;
      WorkItem w{};
      w.b = b;
      w.tok_begin = static_cast<int32_t>(t0 * unit);
      w.tok_end = static_cast<int32_t>(std::min<int64_t>(t1 * unit, len[b]));
      w.page_base = page_base[b];
      w.npages = npages[b];
      P->items.push_back(w);
      P->cta_indptr.push_back(static_cast<int32_t>(P->items.size()));
    }
  }
  P->num_ctas = static_cast<int32_t>(P->items.size());
}

// Partial slots (consecutive per split request), direct writes and merge jobs.
void assign_slots(mla_plan* P, const std::vector<int32_t>& len) {
  std::vector<int32_t> nitems(P->bs, 0);
  for (const WorkItem& w : P->items) nitems[w.b]++;
  std::vector<int32_t> first(P->bs, -1);
  int32_t next = 0;
  for (int32_t b = 0; b < P->bs; ++b) {
    if (nitems[b] >= 2) {
      first[b] = next;
      P->jobs.push_back(MergeJob{b, next, nitems[b], 0});
      next += nitems[b];
      P->max_parts = std::max(P->max_parts, nitems[b]);
    } else if (len[b] == 0) {
      P->jobs.push_back(MergeJob{b, 0, 0, 0});
    }
  }
  std::vector<int32_t> used(P->bs, 0);
  for (WorkItem& w : P->items) w.slot = (nitems[w.b] >= 2) ? first[w.b] + used[w.b]++ : -1;
  P->num_partials = next;
}

// A process-wide unique stamp per plan.  The first value mixes the clock in,
// so that plans of two runs of a program do not share stamps either.
uint64_t next_stamp() {
  static std::atomic<uint64_t> counter{
      (static_cast<uint64_t>(
           std::chrono::steady_clock::now().time_since_epoch().count()) * 0x9E3779B97F4A7C15ull) |
      1ull};
  return counter.fetch_add(0x9E3779B97F4A7C15ull * 2ull);
}

void layout_workspace(mla_plan* P) {
  size_t off = 0;
  P->off_err = off;
  static_assert(sizeof(mla::WsHeader) == 16, "workspace header");
  off = align256(off + sizeof(mla::WsHeader));
  P->off_indptr = off;                                       // CtaHead per CTA
  off = align256(off + sizeof(CtaHead) * (P->cta_indptr.size() - 1));
  P->off_items = off;
  off = align256(off + sizeof(WorkItem) * P->items.size());
  P->off_jobs = off;
  off = align256(off + sizeof(MergeJob) * P->jobs.size());
  P->off_part_o = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(P->num_partials) * P->rows * mla::kVDim);
  P->off_part_lse = off;
  off = align256(off + sizeof(float) * static_cast<size_t>(P->num_partials) * P->rows);
  P->ws_bytes = std::max<size_t>(off, 256);
  P->table.assign(P->off_part_o, 0);
  P->stamp = next_stamp();
  mla::WsHeader hdr{};
  hdr.stamp = P->stamp;
  std::memcpy(P->table.data() + P->off_err, &hdr, sizeof(hdr));
  for (size_t c = 0; c + 1 < P->cta_indptr.size(); ++c) {
    CtaHead h{};
    h.it0 = P->cta_indptr[c];
    h.it1 = P->cta_indptr[c + 1];
    h.stamp = P->stamp;
    if (h.it0 < h.it1) h.first = P->items[h.it0];
    std::memcpy(P->table.data() + P->off_indptr + c * sizeof(CtaHead), &h, sizeof(h));
  }
  if (!P->items.empty())
    std::memcpy(P->table.data() + P->off_items, P->items.data(), sizeof(WorkItem) * P->items.size());
  if (!P->jobs.empty())
    std::memcpy(P->table.data() + P->off_jobs, P->jobs.data(), sizeof(MergeJob) * P->jobs.size());
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// KV pool as a 3-D tensor {64-byte chunk, row, chunk index}: a box of
// box_rows rows x all chunks lands in shared memory as [chunk][row][64 B]
// with the 64-byte swizzle.  Out-of-bounds rows are filled with zeros.
bool make_kv_map(CUtensorMap* map, const void* kv, int kv_dtype, int64_t rows, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const bool b16 = kv_dtype == MLA_DTYPE_BF16;
  const uint32_t esz = b16 ? 2 : 1, row_bytes = mla::kQkDim * esz;
  const cuuint64_t dims[3] = {64 / esz, static_cast<cuuint64_t>(rows), row_bytes / 64};
  const cuuint64_t strides[2] = {row_bytes, 64};
  const cuuint32_t box[3] = {64 / esz, static_cast<cuuint32_t>(box_rows), row_bytes / 64};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, b16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
             const_cast<void*>(kv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" {

// Split requests can be merged inside stage 1 when the CTAs of every
// request form one thread-block cluster: every CTA holds one item, request
// b's items are CTAs 8k .. 8k + 7 of one cluster k, and every request is
// split so (stage 2 also zero-fills empty requests, so a batch with one
// keeps it).  One query token per request, bf16 or fp8 KV.  Only eight-way
// splits use it: with 2 or 4 partials per request the narrow stage-2 merge
// (one round trip) was faster than the cluster launch and its barriers
// (0.2-0.6 us per call on GB300), with 8 the cluster merge saved 0.7-2.2 us.
constexpr int32_t kClusterMerge = 8;
static int32_t cluster_size_of(const mla_plan* P) {
  if (P->q_len != 1 || P->qmode == mla::kQBf16KvMx || P->qmode == mla::kQFp8KvFp8x2 ||
      P->qmode == mla::kQBf16KvFp8x2 ||
      P->num_ctas < 2 || static_cast<int32_t>(P->items.size()) != P->num_ctas || P->jobs.empty())
    return 0;
  for (int32_t c = 0; c < P->num_ctas; ++c)
    if (P->cta_indptr[c + 1] - P->cta_indptr[c] != 1) return 0;
  const int32_t cs = P->jobs[0].count;
  if (cs != kClusterMerge ||
      static_cast<int64_t>(P->jobs.size()) * cs != P->num_ctas)
    return 0;
  for (const MergeJob& j : P->jobs)
    if (j.count != cs) return 0;
  for (int32_t c = 0; c < P->num_ctas; ++c)
    if (P->items[c].b != P->items[(c / cs) * cs].b || P->items[c].slot < 0) return 0;
  return cs;
}

mla_status mla_decode_plan_ex(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                              int32_t batch_size, int32_t q_len, int32_t page_size,
                              mla_dtype q_dtype, mla_dtype kv_dtype,
                              const mla_plan_options* options, mla_plan** plan_out) {
  if (plan_out == nullptr) return MLA_ERR_INVALID_ARG;
  *plan_out = nullptr;
  const mla_plan_options o = options != nullptr ? *options : mla_plan_options{0, 0, 0, 0, 0};
  int32_t num_splits = o.num_splits, num_sms = o.num_sms;
  const int64_t item_cost = o.item_cost == 0 ? 1 : o.item_cost;
  const int32_t unit = o.unit_tokens == 0 ? mla::kTile : o.unit_tokens;
  if (o.item_cost < 0 || o.item_cost > 64 || o.merge < 0 || o.merge > 1 ||
      (unit != 32 && unit != 64 && unit != mla::kTile))
    return MLA_ERR_INVALID_ARG;
  if (kv_indptr_host == nullptr || batch_size < 1 || page_size < 1 || num_splits < 0 ||
      num_sms < 0 || q_len < 1 || q_len > MLA_MAX_Q_LEN ||
      static_cast<int64_t>(batch_size) * q_len > INT32_MAX / mla::kHeads)
    return MLA_ERR_INVALID_ARG;
  if (q_dtype < MLA_DTYPE_BF16 || q_dtype > MLA_DTYPE_MXFP4 || kv_dtype < MLA_DTYPE_BF16 ||
      kv_dtype > MLA_DTYPE_MXFP4)
    return MLA_ERR_INVALID_ARG;
  const int qmode = qmode_of(q_dtype, kv_dtype);
  if (qmode < 0) return MLA_ERR_UNSUPPORTED;
  if (kv_indptr_host[0] < 0) return MLA_ERR_INVALID_ARG;
  // With fp8 KV (fp8 or bf16 q) and an even q_len, query tokens run in pairs:
  // pair p of request b is "virtual request" r = b * q_len / 2 + p, whose 32
  // q rows (tokens 2p, 2p+1) share every tile (kQFp8KvFp8x2, kQBf16KvFp8x2); its first token sees
  // vis0 = n - q_len + 1 + 2p tokens, its second one more.  Otherwise query
  // token t of request b is virtual request r = b * q_len + t (its q, out
  // and lse row): it attends to the request's first n - q_len + 1 + t
  // tokens.  Either way through the request's own pages.
  const bool pairs = q_len % 2 == 0 && (qmode == mla::kQFp8KvFp8 || qmode == mla::kQBf16KvFp8);
  const int32_t qv = pairs ? q_len / 2 : q_len;    // virtual requests per request
  const int32_t nv = batch_size * qv;
  std::vector<int32_t> len(nv), page_base(nv), npages(nv), vis0(nv, 0);
  std::vector<int64_t> tiles(nv);                  // cut units of each virtual request
  int64_t total_tok = 0, total_tiles = 0, total_units = 0;
  int64_t identity_rows = 0;      // pool rows the identity table reaches
  for (int32_t b = 0; b < batch_size; ++b) {
    const int64_t np = static_cast<int64_t>(kv_indptr_host[b + 1]) - kv_indptr_host[b];
    if (np < 0) return MLA_ERR_INVALID_ARG;
    int64_t n = np * page_size;
    if (np > 0 && kv_last_page_len_host != nullptr) {
      const int32_t last = kv_last_page_len_host[b];
      if (last < 1 || last > page_size) return MLA_ERR_INVALID_ARG;
      n -= page_size - last;
    }
    if (n > INT32_MAX - mla::kTile) return MLA_ERR_INVALID_ARG;
    if (n > 0)
      identity_rows = std::max(identity_rows, static_cast<int64_t>(kv_indptr_host[b]) * page_size + n);
    for (int32_t t = 0; t < qv; ++t) {
      const int32_t r = b * qv + t;
      const int64_t first_seen = n - q_len + 1 + (pairs ? 2 * t : t);
      len[r] = static_cast<int32_t>(std::max<int64_t>(0, first_seen + (pairs ? 1 : 0)));
      vis0[r] = static_cast<int32_t>(std::max<int64_t>(0, first_seen));
      page_base[r] = kv_indptr_host[b];
      npages[r] = static_cast<int32_t>(np);
      tiles[r] = (len[r] + unit - 1) / unit;
      total_tok += len[r];
      total_tiles += (len[r] + mla::kTile - 1) / mla::kTile;
      total_units += tiles[r];
    }
  }
  if (num_sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  mla_plan* P = new (std::nothrow) mla_plan();
  if (P == nullptr) return MLA_ERR_INVALID_ARG;
  P->bs = nv;
  P->nreq = batch_size;
  P->rows = pairs ? 2 * mla::kHeads : mla::kHeads;
  P->q_len = q_len;
  P->page_size = page_size;
  P->num_splits = num_splits;
  P->q_dtype = q_dtype;
  P->kv_dtype = kv_dtype;
  P->qmode = !pairs ? qmode : qmode == mla::kQFp8KvFp8 ? mla::kQFp8KvFp8x2 : mla::kQBf16KvFp8x2;
  P->total_tokens = total_tok;
  P->identity_rows = identity_rows;
  P->total_tiles = total_tiles;
  P->unit_tokens = unit;
  P->item_cost = static_cast<int32_t>(item_cost);
  P->num_sms = num_sms;
  P->cta_indptr.assign(1, 0);
  if (num_splits == 0) {
    const int32_t G = static_cast<int32_t>(std::min<int64_t>(num_sms, total_units));
    std::vector<int32_t> order;
    if (qv == 1 || G < qv) {
      // query-token-major order: the q_len passes over a request's KV stay
      // close in time when the CTAs are too few to group them
      for (int32_t t = 0; t < qv; ++t)
        for (int32_t b = 0; b < batch_size; ++b) order.push_back(b * qv + t);
      plan_balanced(P, order, tiles, len, page_base, npages, G, item_cost, unit);
    } else {
      // one group of CTAs per query token (or pair), each balanced over
      // every request: CTA i of each group reads the same KV at about the
      // same time, so the other passes are served from L2
      for (int32_t t = 0; t < qv; ++t) {
        order.clear();
        for (int32_t b = 0; b < batch_size; ++b) order.push_back(b * qv + t);
        const int32_t Gt = static_cast<int32_t>((static_cast<int64_t>(G) * (t + 1)) / qv -
                                                (static_cast<int64_t>(G) * t) / qv);
        plan_balanced(P, order, tiles, len, page_base, npages, Gt, item_cost, unit);
      }
    }
  } else {
    plan_fixed(P, tiles, len, page_base, npages, num_splits, unit);
  }
  for (WorkItem& w : P->items) w.vis0 = vis0[w.b];
  assign_slots(P, len);
  layout_workspace(P);
  P->cluster = o.merge == 0 ? cluster_size_of(P) : 0;
  *plan_out = P;
  return MLA_OK;
}

mla_status mla_decode_plan_q(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                             int32_t batch_size, int32_t q_len, int32_t page_size,
                             mla_dtype q_dtype, mla_dtype kv_dtype, int32_t num_splits,
                             int32_t num_sms, mla_plan** plan_out) {
  const mla_plan_options o{num_splits, num_sms, 0, 0, 0};
  return mla_decode_plan_ex(kv_indptr_host, kv_last_page_len_host, batch_size, q_len, page_size,
                            q_dtype, kv_dtype, &o, plan_out);
}

mla_status mla_decode_plan(const int32_t* kv_indptr_host, const int32_t* kv_last_page_len_host,
                           int32_t batch_size, int32_t page_size, mla_dtype q_dtype,
                           mla_dtype kv_dtype, int32_t num_splits, int32_t num_sms,
                           mla_plan** plan_out) {
  return mla_decode_plan_q(kv_indptr_host, kv_last_page_len_host, batch_size, 1, page_size,
                           q_dtype, kv_dtype, num_splits, num_sms, plan_out);
}

mla_status mla_plan_workspace_size(const mla_plan* plan, size_t* bytes) {
  if (plan == nullptr || bytes == nullptr) return MLA_ERR_INVALID_ARG;
  *bytes = plan->ws_bytes;
  return MLA_OK;
}

mla_status mla_plan_get_info(const mla_plan* plan, mla_plan_info* info) {
  if (plan == nullptr || info == nullptr) return MLA_ERR_INVALID_ARG;
  info->batch_size = plan->nreq;
  info->q_len = plan->q_len;
  info->page_size = plan->page_size;
  info->num_ctas = plan->num_ctas;
  info->num_items = static_cast<int32_t>(plan->items.size());
  info->num_partials = plan->num_partials;
  info->num_merge_jobs = static_cast<int32_t>(plan->jobs.size());
  info->total_tokens = plan->total_tokens;
  info->total_tiles = plan->total_tiles;
  info->workspace_bytes = plan->ws_bytes;
  info->cluster_size = plan->cluster;
  info->unit_tokens = plan->unit_tokens;
  info->item_cost = plan->item_cost;
  return MLA_OK;
}

mla_status mla_plan_get_work(const mla_plan* plan, int32_t* cta_indptr, int32_t* items) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (cta_indptr != nullptr)
    std::memcpy(cta_indptr, plan->cta_indptr.data(), sizeof(int32_t) * plan->cta_indptr.size());
  if (items != nullptr)
    for (size_t i = 0; i < plan->items.size(); ++i) {
      items[4 * i + 0] = plan->items[i].b;
      items[4 * i + 1] = plan->items[i].tok_begin;
      items[4 * i + 2] = plan->items[i].tok_end;
      items[4 * i + 3] = plan->items[i].slot;
    }
  return MLA_OK;
}

void mla_plan_destroy(mla_plan* plan) { delete plan; }

mla_status mla_decode_run(mla_plan* plan, const void* q, const float* q_scale, const void* kv,
                          const float* kv_scale, const uint8_t* kv_e8m0,
                          int64_t kv_e8m0_row_stride, int64_t kv_pool_rows,
                          const int32_t* kv_indices, void* workspace, size_t workspace_bytes,
                          void* out, float* lse, mla_stream_t stream_) {
  if (plan == nullptr || q == nullptr || kv == nullptr || out == nullptr || workspace == nullptr)
    return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  if (kv_pool_rows < 1 || kv_pool_rows > INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (plan->q_dtype == MLA_DTYPE_FP8_E4M3 && q_scale == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->kv_dtype == MLA_DTYPE_FP8_E4M3 && kv_scale == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->kv_dtype == MLA_DTYPE_MXFP4) {
    if (kv_e8m0 == nullptr || kv_e8m0_row_stride < 18) return MLA_ERR_INVALID_ARG;
    // scale rows are read two bytes at a time
    if (kv_e8m0_row_stride % 2 != 0 || !aligned(kv_e8m0, 2)) return MLA_ERR_UNSUPPORTED;
  }
  if (workspace_bytes < plan->ws_bytes) return MLA_ERR_WORKSPACE;
  // without a page table, request b's rows follow from kv_indptr: all of them
  // must lie inside the pool
  if (kv_indices == nullptr && plan->identity_rows > kv_pool_rows) return MLA_ERR_INVALID_ARG;
  // Identity table: one TMA box of 128 rows per tile.  Page table with a
  // page size that is a multiple of 8: one box per 8-row group (a group never
  // straddles a page).  Other page sizes (bf16 / fp8 KV): every row is
  // gathered on its own (cp.async), laid out as for the identity table.
  // MXFP4 rows are loaded by the dequantising threads themselves (no tensor
  // map) and written in the 8-row-group layout, for any page size.
  const bool mx = plan->kv_dtype == MLA_DTYPE_MXFP4;
  int box_rows = mla::kTile;
  int gather = 0;
  if (kv_indices != nullptr) {
    if (kv_pool_rows % plan->page_size != 0) return MLA_ERR_INVALID_ARG;
    if (plan->page_size % 8 == 0 || mx)
      box_rows = 8;
    else
      gather = 1;
  }
  // MXFP4, and plans cut below whole tiles (a CTA's rows are then fewer
  // than 128): 8-row groups
  if (mx || plan->unit_tokens < mla::kTile) box_rows = 8;
  // bytes per row of the tile the UMMAs read (MXFP4 is dequantised to e4m3)
  const uint32_t row_bytes = mla::kQkDim * (plan->kv_dtype == MLA_DTYPE_BF16 ? 2 : 1);
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!mx && (plan->tmap_ptr != kv || plan->tmap_rows != kv_pool_rows ||
              plan->tmap_box_rows != box_rows)) {
    if (!make_kv_map(&plan->tmap, kv, plan->kv_dtype, kv_pool_rows, box_rows)) return MLA_ERR_CUDA;
    plan->tmap_ptr = kv;
    plan->tmap_rows = kv_pool_rows;
    plan->tmap_box_rows = box_rows;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (plan->uploaded_ws != workspace) {
    if (cudaMemcpyAsync(ws, plan->table.data(), plan->table.size(), cudaMemcpyHostToDevice,
                        stream) != cudaSuccess)
      return MLA_ERR_CUDA;
    plan->uploaded_ws = workspace;
  }
  float* part_o = reinterpret_cast<float*>(ws + plan->off_part_o);
  float* part_lse = reinterpret_cast<float*>(ws + plan->off_part_lse);
  int32_t* err = reinterpret_cast<int32_t*>(ws + plan->off_err);
  // cluster merge when the plan allows it and this device can hold such a
  // cluster (checked once per plan and device); otherwise stage 2 merges
  bool cluster = false;
  if (plan->cluster > 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    if (plan->cluster_dev != dev) {
      plan->cluster_fits = mla::stage1_cluster_fits(plan->qmode, plan->cluster);
      plan->cluster_dev = dev;
    }
    cluster = plan->cluster_fits;
  }
  if (plan->num_ctas > 0) {
    mla::Stage1Params p{};
    p.tmap_kv = plan->tmap;
    p.q = q;
    p.q_scale = q_scale;
    p.kv_scale = kv_scale;
    p.kv_indices = kv_indices;
    p.items = reinterpret_cast<const WorkItem*>(ws + plan->off_items);
    p.heads = reinterpret_cast<const CtaHead*>(ws + plan->off_indptr);
    p.part_o = part_o;
    p.part_lse = part_lse;
    p.out = static_cast<uint16_t*>(out);
    p.lse = lse;
    p.err = err;
    p.stamp = plan->stamp;
    p.page_size = plan->page_size;
    p.box_rows = box_rows;
    p.gather = gather;
    p.kv = static_cast<const uint8_t*>(kv);
    p.chunk_stride = static_cast<uint32_t>(box_rows) * 64u;    // [group][chunk][rows][64 B]
    p.group_stride = box_rows == 8 ? row_bytes * 8u : 512u;
    p.pool_rows = kv_pool_rows;
    p.kv_e8m0 = kv_e8m0;
    p.sc_stride = kv_e8m0_row_stride;
    p.cluster = cluster ? plan->cluster : 0;
    if (plan->ev_before != nullptr && cudaEventRecord(plan->ev_before, stream) != cudaSuccess)
      return MLA_ERR_CUDA;
    if (mla::launch_stage1(plan->qmode, p, plan->num_ctas, stream) != cudaSuccess)
      return MLA_ERR_CUDA;
    if (plan->ev_after != nullptr && cudaEventRecord(plan->ev_after, stream) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (!plan->jobs.empty() && !cluster) {
    mla::Stage2Params s{};
    s.jobs = reinterpret_cast<const MergeJob*>(ws + plan->off_jobs);
    s.err = err;
    s.stamp = plan->stamp;
    s.part_o = part_o;
    s.part_lse = part_lse;
    s.out = static_cast<uint16_t*>(out);
    s.lse = lse;
    s.num_jobs = static_cast<int32_t>(plan->jobs.size());
    s.rows = plan->rows;
    s.wide = plan->max_parts > 4 ? 1 : 0;   // the narrow merge takes up to 4 partials per round trip
    if (mla::launch_stage2(s, stream) != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

mla_status mla_decode_check(const mla_plan* plan, void* workspace, mla_stream_t stream_) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (workspace == nullptr) {
    // the array mla_decode_run_noalloc uses on the current device
    const mla_status st = mla::static_workspace(&workspace);
    if (st != MLA_OK) return st;
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int32_t word = 0;
  int32_t* dev = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + plan->off_err);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaMemcpy(&word, dev, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (word == 0) return MLA_OK;
  if (cudaMemset(dev, 0, sizeof(word)) != cudaSuccess) return MLA_ERR_CUDA;
  if (word & mla::kErrStale) {
    // the workspace held another plan's table: upload this plan's again on
    // its next run with this workspace
    if (plan->uploaded_ws == workspace) plan->uploaded_ws = nullptr;
    return MLA_ERR_WORKSPACE;
  }
  return (word & mla::kErrTimeout) ? MLA_ERR_DEVICE_TIMEOUT : MLA_ERR_INVALID_ARG;
}

mla_status mla_plan_set_stage1_events(mla_plan* plan, void* before, void* after) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  plan->ev_before = static_cast<cudaEvent_t>(before);
  plan->ev_after = static_cast<cudaEvent_t>(after);
  return MLA_OK;
}

const char* mla_status_string(mla_status status) {
  switch (status) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA";
    case MLA_ERR_DEVICE_TIMEOUT: return "MLA_ERR_DEVICE_TIMEOUT";
  }
  return "MLA_ERR_UNKNOWN";
}

}  // extern "C"
