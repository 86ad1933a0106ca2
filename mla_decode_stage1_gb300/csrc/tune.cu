// tune.cu -- runtime autotune of the decode plan: candidate plans of one
// batch shape are timed on the caller's stream with the caller's inputs, and
// the fastest is kept (and remembered for the shape).
//
// The role of the timing loops of kernelindex.com, amd-mixed-mla submission
// 600081 (the earlier version's _time_fn, _aiter_best and _best_for_shape):
// run each candidate once, time a few calls with CUDA events, keep the
// fastest and cache it per shape.  The candidates here are plan options of
// this library (balanced cuts with different item costs and cut
// granularities, and the fixed split counts of the split tables of
// submission 668813, NUM_KV_SPLITS_TABLE and MXFP4_SPLITS_TABLE).

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "mla_decode.h"
#include "plan.h"

namespace {

// Split counts of the pages' tables, keyed by (batch, kv_len).
int32_t table_splits(int32_t bs, int64_t kv_len, bool mxfp4) {
  struct Entry { int32_t bs; int64_t len; int32_t s; };
  static const Entry kFp8[] = {{4, 1024, 16},  {4, 8192, 32}, {32, 1024, 8},  {32, 8192, 8},
                               {64, 1024, 4},  {64, 8192, 8}, {256, 1024, 1}, {256, 8192, 16}};
  static const Entry kMx[] = {{32, 8192, 8}, {64, 8192, 4}, {256, 8192, 2}};
  if (mxfp4) {
    for (const Entry& e : kMx)
      if (e.bs == bs && e.len == kv_len) return e.s;
    return 0;
  }
  for (const Entry& e : kFp8)
    if (e.bs == bs && e.len == kv_len) return e.s;
  return 0;
}

// The candidates for one shape: the default balanced plan first, then
// heavier item costs, finer cut points, and fixed splits.
std::vector<mla_plan_options> candidates(int32_t bs, int64_t max_len, bool mxfp4) {
  std::vector<mla_plan_options> c = {
      {0, 0, 1, 128, 0}, {0, 0, 2, 128, 0}, {0, 0, 4, 128, 0}, {0, 0, 1, 64, 0}, {0, 0, 1, 32, 0}};
  const int32_t s = table_splits(bs, max_len, mxfp4);
  if (s > 0) c.push_back({s, 0, 0, 0, 0});
  c.push_back({1, 0, 0, 0, 0});
  return c;
}

// Shape key of the cache: batch, query tokens, page size, formats, total and
// largest request length, and whether a page table is used.
using Key = std::tuple<int32_t, int32_t, int32_t, int, int, int64_t, int64_t, bool, int>;
std::mutex g_cache_mutex;
std::map<Key, mla_plan_options> g_cache;

}  // namespace

extern "C" {

mla_status mla_autotune_select(const float* ms, int32_t num_candidates, int32_t reps,
                               int32_t* best) {
  if (ms == nullptr || best == nullptr || num_candidates < 1 || reps < 1)
    return MLA_ERR_INVALID_ARG;
  int32_t pick = -1;
  float pick_ms = 0.0f;
  std::vector<float> v(reps);
  for (int32_t c = 0; c < num_candidates; ++c) {
    bool valid = true;
    for (int32_t r = 0; r < reps; ++r) {
      v[r] = ms[static_cast<size_t>(c) * reps + r];
      if (!(v[r] >= 0.0f)) valid = false;     // negative or NaN: not run
    }
    if (!valid) continue;
    std::sort(v.begin(), v.end());
    const float med = (reps % 2) ? v[reps / 2] : 0.5f * (v[reps / 2 - 1] + v[reps / 2]);
    if (pick < 0 || med < pick_ms) {
      pick = c;
      pick_ms = med;
    }
  }
  if (pick < 0) return MLA_ERR_INVALID_ARG;
  *best = pick;
  return MLA_OK;
}

mla_status mla_decode_autotune(const int32_t* kv_indptr_host,
                               const int32_t* kv_last_page_len_host, int32_t batch_size,
                               int32_t q_len, int32_t page_size, mla_dtype q_dtype,
                               mla_dtype kv_dtype, const void* q, const float* q_scale,
                               const void* kv, const float* kv_scale, const uint8_t* kv_e8m0,
                               int64_t kv_e8m0_row_stride, int64_t kv_pool_rows,
                               const int32_t* kv_indices, void* workspace,
                               size_t workspace_bytes, void* out, float* lse, int32_t reps,
                               int32_t flags, mla_stream_t stream_, mla_tune_result* results,
                               int32_t max_results, int32_t* num_results,
                               size_t* workspace_needed, mla_plan** plan_out) {
  if (kv_indptr_host == nullptr || batch_size < 1 || reps < 1 || reps > 1000 ||
      (results == nullptr && max_results > 0) || max_results < 0)
    return MLA_ERR_INVALID_ARG;
  if (plan_out != nullptr) *plan_out = nullptr;
  if (num_results != nullptr) *num_results = 0;
  // request lengths (in tokens) for the candidate set and the cache key
  int64_t total = 0, max_len = 0;
  for (int32_t b = 0; b < batch_size; ++b) {
    int64_t n = static_cast<int64_t>(kv_indptr_host[b + 1] - kv_indptr_host[b]) * page_size;
    if (n > 0 && kv_last_page_len_host != nullptr) n -= page_size - kv_last_page_len_host[b];
    total += std::max<int64_t>(n, 0);
    max_len = std::max(max_len, n);
  }
  const bool mx = kv_dtype == MLA_DTYPE_MXFP4;
  std::vector<mla_plan_options> cand = candidates(batch_size, max_len, mx);
  // plans and the workspace the largest needs; when the default plan merges
  // inside clusters, its stage-2 form is a candidate too
  std::vector<mla_plan*> plans(cand.size(), nullptr);
  size_t need = 0;
  for (size_t i = 0; i < cand.size(); ++i) {
    const mla_status st = mla_decode_plan_ex(kv_indptr_host, kv_last_page_len_host, batch_size,
                                             q_len, page_size, q_dtype, kv_dtype, &cand[i],
                                             &plans[i]);
    if (st != MLA_OK) {
      for (mla_plan* p : plans) mla_plan_destroy(p);
      return st;
    }
    need = std::max(need, plans[i]->ws_bytes);
    if (i == 0 && plans[0]->cluster > 0) {
      mla_plan_options o = cand[0];
      o.merge = 1;
      cand.insert(cand.begin() + 1, o);
      plans.insert(plans.begin() + 1, nullptr);
    }
  }
  if (workspace_needed != nullptr) *workspace_needed = need;
  auto release = [&](int32_t keep) {
    for (size_t i = 0; i < plans.size(); ++i)
      if (static_cast<int32_t>(i) != keep) mla_plan_destroy(plans[i]);
  };
  if (workspace == nullptr) {                        // query: the size only
    release(-1);
    return MLA_OK;
  }
  if (plan_out == nullptr) {
    release(-1);
    return MLA_ERR_INVALID_ARG;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    release(-1);
    return MLA_ERR_CUDA;
  }
  const Key key{batch_size, q_len, page_size, q_dtype, kv_dtype, total, max_len,
                kv_indices != nullptr, dev};
  if ((flags & MLA_TUNE_IGNORE_CACHE) == 0) {
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    auto it = g_cache.find(key);
    if (it != g_cache.end()) {
      for (size_t i = 0; i < cand.size(); ++i) {
        const mla_plan_options& o = cand[i];
        if (o.num_splits == it->second.num_splits && o.num_sms == it->second.num_sms &&
            o.item_cost == it->second.item_cost && o.unit_tokens == it->second.unit_tokens &&
            o.merge == it->second.merge) {
          release(static_cast<int32_t>(i));
          *plan_out = plans[i];
          return MLA_OK;
        }
      }
    }
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  std::vector<cudaEvent_t> ev(2 * static_cast<size_t>(reps), nullptr);
  for (cudaEvent_t& e : ev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      for (cudaEvent_t& x : ev)
        if (x) cudaEventDestroy(x);
      release(-1);
      return MLA_ERR_CUDA;
    }
  std::vector<float> ms(cand.size() * reps, -1.0f);
  mla_status fail = MLA_OK;
  for (size_t i = 0; i < cand.size() && fail == MLA_OK; ++i) {
    mla_plan* P = plans[i];
    if (P->ws_bytes > workspace_bytes) continue;     // too large: not timed
    auto call = [&]() {
      return mla_decode_run(P, q, q_scale, kv, kv_scale, kv_e8m0, kv_e8m0_row_stride,
                            kv_pool_rows, kv_indices, workspace, workspace_bytes, out, lse,
                            stream_);
    };
    mla_status st = call();                          // uploads the table, warms the caches
    if (st != MLA_OK) {
      fail = st;
      break;
    }
    for (int32_t r = 0; r < reps && st == MLA_OK; ++r) {
      if (cudaEventRecord(ev[2 * r], stream) != cudaSuccess) st = MLA_ERR_CUDA;
      if (st == MLA_OK) st = call();
      if (st == MLA_OK && cudaEventRecord(ev[2 * r + 1], stream) != cudaSuccess) st = MLA_ERR_CUDA;
    }
    if (st != MLA_OK) {
      fail = st;
      break;
    }
    // the device error word of this candidate's runs (bounded waits, pages)
    st = mla_decode_check(P, workspace, stream_);
    if (st == MLA_ERR_DEVICE_TIMEOUT || st == MLA_ERR_CUDA || st == MLA_ERR_INVALID_ARG) {
      fail = st;
      break;
    }
    for (int32_t r = 0; r < reps; ++r) {
      float t = -1.0f;
      if (cudaEventElapsedTime(&t, ev[2 * r], ev[2 * r + 1]) != cudaSuccess) t = -1.0f;
      ms[i * reps + r] = t;
    }
  }
  for (cudaEvent_t& e : ev) cudaEventDestroy(e);
  int32_t best = -1;
  if (fail == MLA_OK && mla_autotune_select(ms.data(), static_cast<int32_t>(cand.size()), reps,
                                            &best) != MLA_OK)
    fail = MLA_ERR_WORKSPACE;                        // no candidate fitted the workspace
  if (fail != MLA_OK) {
    release(-1);
    return fail;
  }
  // report: the options and median time of each candidate
  const int32_t n = std::min<int32_t>(max_results, static_cast<int32_t>(cand.size()));
  for (int32_t i = 0; i < n; ++i) {
    results[i].options = cand[i];
    std::vector<float> v(ms.begin() + static_cast<size_t>(i) * reps,
                         ms.begin() + static_cast<size_t>(i + 1) * reps);
    std::sort(v.begin(), v.end());
    results[i].ms = v[0] < 0.0f ? -1.0f
                    : (reps % 2) ? v[reps / 2] : 0.5f * (v[reps / 2 - 1] + v[reps / 2]);
  }
  if (num_results != nullptr) *num_results = n;
  {
    std::lock_guard<std::mutex> lock(g_cache_mutex);
    g_cache[key] = cand[best];
  }
  release(best);
  // later candidates ran in the same workspace after this one: its table
  // must be copied in again on its next run
  plans[best]->uploaded_ws = nullptr;
  *plan_out = plans[best];
  return MLA_OK;
}

}  // extern "C"
