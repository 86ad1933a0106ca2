// kernels.h -- internal interface between the host API (api.cu) and the two
// CUDA kernels (stage1.cu, stage2.cu).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace mla {

constexpr int kHeads = 16;     // query heads per request, one latent KV head
constexpr int kQkDim = 576;    // 512 latent + 64 rope dims take part in QK^T
constexpr int kVDim = 512;     // V = the first 512 dims of the latent row
constexpr int kTile = 128;     // tokens per stage-1 tile (UMMA M)

// Scores are kept in the log2 domain: s2 = s * log2(e).  p = 2^(s2 - m + kPOff)
// with m the running max, allowed to lag the true max by at most kTau.
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kPOff = 4.0f;
constexpr float kTau = 4.0f;
constexpr float kPLoScale = 16.0f;    // the low part of p is stored x2^4
// (p <= 2^(kPOff+kTau) = 256, so |p - e4m3(p)| * 16 <= 256 <= 448)

// Device error word bits: one per pipeline role that gave up a wait, a page
// outside the pool, and a workspace that holds another plan's table.
enum : int32_t {
  kErrProducer = 1, kErrMma = 2, kErrSoftmax = 4, kErrQPrep = 8, kErrDrain = 16,
  kErrBadPage = 32, kErrDequant = 64, kErrStale = 128
};
constexpr int32_t kErrTimeout = kErrProducer | kErrMma | kErrSoftmax | kErrQPrep | kErrDrain |
                                kErrDequant;

// Workspace header (the first 16 bytes of every plan's workspace): the
// device error word, then the stamp of the plan whose table was uploaded
// last.  Every CTA head carries the stamp too.
struct WsHeader {
  int32_t err;
  int32_t pad;
  uint64_t stamp;
};

// One work item: a contiguous token range of one request.
struct WorkItem {
  int32_t b;          // request
  int32_t tok_begin;  // first token (multiple of kTile)
  int32_t tok_end;    // one past the last token
  int32_t slot;       // partial slot, or -1: write out/lse directly
  int32_t page_base;  // kv_indptr[b]: first page-table entry of the request
  int32_t npages;     // page-table entries of the request
  int32_t vis0;       // two query tokens per request: tokens query token 0 sees
                      // (query token t sees vis0 + t); unused with one token
  int32_t pad1;
};
static_assert(sizeof(WorkItem) == 32, "work item is two int4");

// Per-CTA head: its item range and a copy of its first item, so that one
// load gives a CTA everything its first tile needs.
struct CtaHead {
  int32_t it0, it1;   // items [it0, it1) of the work-item array
  uint64_t stamp;     // the plan's stamp
  WorkItem first;     // items[it0] (unused when it0 == it1)
};
static_assert(sizeof(CtaHead) == 48, "CTA head is three int4");

// One stage-2 job: merge `count` consecutive partials of request b (count 0:
// the request is empty, write zeros and -inf).
struct MergeJob {
  int32_t b, first, count, pad;
};

enum QMode : int {
  kQBf16KvBf16 = 0,   // kind::f16, B = q (16 rows)
  kQFp8KvFp8 = 1,     // kind::f8f6f4, B = q bytes (16 rows)
  kQBf16KvFp8 = 2,    // kind::f8f6f4, B = [q_hi ; q_lo] e4m3 (32 rows)
  kQFp8KvBf16 = 3,    // kind::f16, q decoded to bf16 (exact), B = 16 rows
  kQBf16KvMx = 4,     // MXFP4 KV dequantised in shared memory to e4m3 with a per-token
                      // power of two; then as kQBf16KvFp8
  kQFp8KvFp8x2 = 5,   // two query tokens per request, fp8 q and KV: kind::f8f6f4,
                      // B = 32 q rows (token-major), causal over the last two positions
  kQBf16KvFp8x2 = 6   // two query tokens per request, bf16 q and fp8 KV: B = [q_hi; q_lo]
                      // of the 32 q rows (64 rows), as kQBf16KvFp8 for one token
};

struct Stage1Params {
  CUtensorMap tmap_kv;          // KV pool as [chunk 64 B][row][64 B], 64-byte swizzle
                                // (bf16 / fp8; MXFP4 rows are read with plain loads)
  const void* q;                // [bs,16,576]
  const float* q_scale;         // device [1] (fp8 q) or null
  const float* kv_scale;        // device [1] (fp8 kv) or null
  const int32_t* kv_indices;    // page table or null (identity)
  const WorkItem* items;
  const CtaHead* heads;         // [num_ctas]
  float* part_o;                // [num_partials,16,512] fp32, normalised
  float* part_lse;              // [num_partials,16] log2 domain
  uint16_t* out;                // [bs,16,512] bf16 bits
  float* lse;                   // [bs,16] natural log, nullable
  int32_t* err;                 // device error word (the workspace header)
  uint64_t stamp;               // the plan's stamp; the workspace must carry the same
  int32_t page_size;
  int32_t box_rows;             // rows per TMA box: 128 (identity table) or 8 (page table)
  int32_t gather;               // 1: page size not a multiple of 8 (bf16 / fp8 KV); rows are
                                // gathered one by one with cp.async instead of TMA boxes
  int32_t cluster;              // 0: split items write partials for stage 2; cs (a divisor of
                                // 512, at most 8): the grid is in clusters of cs CTAs, one
                                // request each, whose partials are merged inside the cluster
  const uint8_t* kv;            // KV pool base (row gather, MXFP4 row loads)
  uint32_t chunk_stride;        // smem bytes between 64-byte column chunks of a tile
  uint32_t group_stride;        // smem bytes between 8-row groups of a tile
  int64_t pool_rows;
  const uint8_t* kv_e8m0;       // MXFP4 only: e8m0 scale rows (18 bytes used per row)
  int64_t sc_stride;            // bytes between scale rows (even, >= 18)
};

struct Stage2Params {
  const MergeJob* jobs;
  int32_t* err;                 // device error word (the workspace header)
  uint64_t stamp;               // the plan's stamp
  int32_t rows;                 // output rows per request: 16 heads x query tokens
  int32_t wide;                 // 1: some request has many partials (one CTA per row)
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  float* lse;
  int32_t num_jobs;
};

// Host launchers; return the cudaError_t of the launch.
cudaError_t launch_stage1(int qmode, const Stage1Params& p, int num_ctas, cudaStream_t stream);
cudaError_t launch_stage2(const Stage2Params& p, cudaStream_t stream);
int stage1_smem_bytes(int qmode);
// Whether stage 1 of `qmode` can run in clusters of `cs` CTAs on the current
// device (at least one such cluster fits).
bool stage1_cluster_fits(int qmode, int cs);

}  // namespace mla
