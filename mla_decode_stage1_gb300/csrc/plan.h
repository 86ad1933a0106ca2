// plan.h -- the host-side plan object behind the opaque mla_plan handle
// (internal to libmla_decode).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "kernels.h"
#include "mla_decode.h"

struct mla_plan {
  int32_t bs = 0, page_size = 0, num_splits = 0;   // bs: rows of q (requests x q_len)
  int32_t q_len = 1;                                 // query tokens per request
  int32_t nreq = 0;                                  // requests of the batch
  int32_t rows = 16;                                 // output rows per planned request (16 x tokens it holds)
  int q_dtype = 0, kv_dtype = 0, qmode = 0;
  int32_t num_ctas = 0, num_partials = 0;
  int32_t max_parts = 0;   // most partials of one request (stage 2 goes wide above 4)
  int32_t unit_tokens = mla::kTile;   // tokens between the planner's possible cut points
  int32_t item_cost = 1;              // cost of an extra item in a CTA (balanced plan)
  int32_t num_sms = 0;                // CTAs the balanced plan was cut for
  int32_t cluster = 0;                // CTAs per cluster merging a request inside stage 1 (0: stage 2)
  int64_t total_tokens = 0, total_tiles = 0;
  int64_t identity_rows = 0;   // pool rows the requests reach without a page table
  std::vector<int32_t> cta_indptr;
  std::vector<mla::WorkItem> items;
  std::vector<mla::MergeJob> jobs;
  // workspace layout (byte offsets)
  size_t off_err = 0, off_indptr = 0, off_items = 0, off_jobs = 0, off_part_o = 0,
         off_part_lse = 0, ws_bytes = 0;
  std::vector<uint8_t> table;  // image of [0, off_part_o) uploaded once per workspace
  uint64_t stamp = 0;          // unique per plan; written into the table header and CTA heads
  // per-run caches (the upload cache is reset by mla_decode_check when a
  // kernel found another plan's table in the workspace)
  mutable void* uploaded_ws = nullptr;
  CUtensorMap tmap;
  const void* tmap_ptr = nullptr;
  int64_t tmap_rows = -1;
  int32_t tmap_box_rows = -1;
  cudaEvent_t ev_before = nullptr, ev_after = nullptr;
  mutable int cluster_dev = -1;       // device whose cluster fit was checked (cluster_fits)
  mutable bool cluster_fits = false;
};

namespace mla {
// Device address of the library's own workspace array on the current device
// (noalloc.cu), looked up once per device.
mla_status static_workspace(void** out);
constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;
}  // namespace mla
