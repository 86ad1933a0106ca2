// stage1.cu -- split-KV stage-1 kernel of MLA decode for sm_103a.
//
// What it computes (kernelindex.com, amd-mixed-mla submission 668813, MXFP4
// qh16 stage-1 kernel; submission 695854, fp8 split stage-1 kernel): for one
// token range of one request and all 16 heads at once (all 32 q rows of two
// query tokens in the two-token mode), the scores
// s = q . k^T * (1/sqrt(576)) over 576 dims, an exp2-domain online softmax,
// and the partial output O = softmax(s) . V with V the first 512 dims of the
// same rows, plus the log-sum-exp of the range.
//
// How (GB300-first, not the pages' Triton design):
//  * one persistent CTA per SM walks a planner-built list of work items; KV
//    rows stream HBM -> shared memory as whole 128-token tiles.  One 3-D TMA
//    box moves 8 rows x all 576 dims (a page group of 4.5 KB in fp8) into a
//    [64-byte column chunk][8 rows][64 B] image with the 64-byte swizzle, so
//    a page-8 table costs 16 TMA operations per tile and an identity table 1;
//  * QK^T runs on the 5th-generation tensor cores with the tokens as M:
//    S^T[128 tok x 16 q rows] = K[128 x 576] . Q^T, accumulated in TMEM;
//  * PV reuses the very same shared-memory bytes as an MN-major operand:
//    O^T[512 x 16] += V^T[512 x 128 tok] . P^T, four M=128 blocks in TMEM;
//  * a tcgen05.mma costs the issuing thread about the same time whatever
//    its N, so QK^T and PV are issued by separate warps that run side by
//    side: warps 1 and 3 each issue half of the QK^T K-steps into their own
//    S accumulator; warps 2 and 13 issue PV for O blocks 0-1 and 2-3 (MXFP4:
//    warp 2 alone).  Warp 0 is the TMA producer; warps 4-11 do the softmax
//    and the epilogue in two groups of 8 heads (two-token mode: one group
//    per query token, 16 heads each; one thread per token / per
//    output dim, TMEM lane = thread) and convert the first item's q; warp
//    12 converts the q of later items (MXFP4: warps 12-15 dequantise the
//    packed rows in place and prepare every item's q);
//  * every mbarrier wait is bounded (see mbar_wait) and reports into the
//    device error word instead of hanging.
//
// Precision: fp8 KV is consumed as raw e4m3 bytes by kind::f8f6f4 UMMAs with
// the per-tensor scales folded into one score factor and into l.  A bf16 q
// meeting fp8 KV is split into q_hi + q_lo (two e4m3 terms with a per-request
// scale, ~bf16 precision) that share one UMMA with N = 32.  p is likewise
// split into p_hi + 2^-4 p_lo e4m3 terms, stacked as the 32 columns of one
// MN-major PV operand (one 32-byte row per token) so that one UMMA
// accumulates both parts (TMEM columns 0-15, 16-31).
// bf16 KV runs kind::f16 with bf16 q and bf16 p.

#include <cstddef>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mla {

template <int QM>
struct Layout {
  static constexpr bool kMx = (QM == kQBf16KvMx);                  // MXFP4 KV, dequantised
  static constexpr bool kKv8 =
      (QM == kQFp8KvFp8 || QM == kQBf16KvFp8 || kMx || QM == kQFp8KvFp8x2);
  static constexpr int kQL = (QM == kQFp8KvFp8x2) ? 2 : 1;         // query tokens per request
  static constexpr int kRows = kHeads * kQL;                        // q rows, token-major
  static constexpr bool kHiLo = (QM == kQBf16KvFp8 || kMx);         // q as two e4m3 terms
  static constexpr int kNq = kRows * (kHiLo ? 2 : 1);               // UMMA N of QK^T
  // Warps: producer, 2 QK^T issuers, PV issuer(s), two head groups of four
  // softmax warps (kH q rows each), then either a q warp (14 warps) or, for
  // MXFP4, 4 dequant warps that also prepare q (16 warps, register cap 128).
  static constexpr int kHeadGroups = 2;
  static constexpr int kH = kRows / kHeadGroups;                    // q rows per softmax thread
  static constexpr int kThreads = kMx ? 512 : 448;
  static constexpr int kPvIssuers = kMx ? 1 : 2;
  static constexpr int kElem = kKv8 ? 1 : 2;
  static constexpr int kRowBytes = kQkDim * kElem;                  // 576 | 1152
  static constexpr int kChunks = kRowBytes / 64;                    // 64-byte column chunks
  static constexpr int kVChunks = kVDim * kElem / 64;               // chunks holding V
  static constexpr int kTileBytes = kTile * kRowBytes;              // 72 KB | 144 KB
  static constexpr int kKSteps = kRowBytes / 32;                    // QK^T steps of 32 bytes
  static constexpr int kQAtoms = kKv8 ? 5 : 9;                      // 128-byte K atoms of q
  static constexpr int kQAtomBytes = kNq * 128;
  static constexpr int kQBytes = kQAtoms * kQAtomBytes;
  static constexpr int kPRow = 2 * kRows;                           // P bytes per token
  static constexpr int kPBytes = kTile * kPRow;
  static constexpr int kRawRowBytes = kQkDim / 2;                   // packed MXFP4 row
  static constexpr bool kQ8 = (QM == kQFp8KvFp8 || QM == kQFp8KvBf16 || QM == kQFp8KvFp8x2);
  static constexpr int kQSrcBytes = kRows * kQkDim * (kQ8 ? 1 : 2);  // one request's q
  static constexpr uint32_t kOCols = kRows * (kKv8 ? 2 : 1);       // TMEM columns per O block
  // TMEM: S^T at 0 (2 buffers x 2 K-halves x 32 columns), O^T from 128
  static constexpr uint32_t kTmemCols = 128 + 4 * kOCols <= 256 ? 256 : 512;
  static constexpr int kMiscBytes = 2560;
  static constexpr int kScRowBytes = kMx ? kTile * 24 : 0;         // e8m0 row of each dequant thread
  static constexpr int kMaxSmem = 232448;
  static constexpr int kNumTiles =
      (kMaxSmem - 1024 - 2 * kQBytes - 2 * kPBytes - kMiscBytes - kScRowBytes - kQSrcBytes) /
      kTileBytes;
  static constexpr int kQOff = kNumTiles * kTileBytes;
  static constexpr int kPOff = kQOff + 2 * kQBytes;
  static constexpr int kMiscOff = kPOff + 2 * kPBytes;
  static constexpr int kScRowOff = kMiscOff + kMiscBytes;
  static constexpr int kQStageOff = kScRowOff + kScRowBytes;         // raw q of the next item
  static constexpr int kSmemBytes = kQStageOff + kQSrcBytes + 1024;
  static_assert(kNumTiles >= 1 && kNumTiles <= 4, "tile ring");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory over budget");
  static_assert(kTileBytes % 1024 == 0 && kQBytes % 1024 == 0, "operand alignment");
  static_assert(kNq <= 32, "S^T columns per K-half");
};

// Misc region: barriers, reduction scratch, q scales, TMEM address.
struct Misc {
  uint64_t full[4], empty[4];
  uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2], q_full[2], q_empty[2], drain[4];
  alignas(16) float red[2][4][32];   // per-warp partial max / sum of every q row
  float qscale[2][2];
  uint32_t tmem_base;
  int32_t abort_sm;                  // set by a softmax thread whose bounded wait gave up
  uint64_t q_stage;                  // raw q of the next item landed in the staging buffer
  uint64_t q_stage_free;             // the softmax warps converted the first item's q
  float qred[8];                     // per-warp |q| maxima (q prepared by a warp group)
  // MXFP4 only
  uint64_t deq[4];                   // tile slot dequantised (128 dequant threads)
  uint64_t deq_a[4];                 // its dims 0-319 dequantised (first QK^T K-half)
  uint64_t upper_free[4];            // PV no longer reads the slot's upper box halves
  int32_t abort_dq;                  // set by a dequant thread whose bounded wait gave up
  int32_t stale;                     // the workspace holds another plan's table
  float uexp[2][128];                // per-token power of two u_t = r_t - 127 of a slot
  uint2 e2m1_tab[16];                // e4m3 tables for 2^k, k = index - 14 (k <= -14: all 0)
};
static_assert(sizeof(Misc) <= 2560, "misc region");
static_assert(offsetof(Misc, red) % 16 == 0, "reduction scratch is read as float4");

// TMEM columns: S^T as 2 buffers x 2 K-halves x 32 columns [0,128) (the two
// QK^T issuers each accumulate half of the 576 dims), then O^T: four 128-dim
// blocks of kOCols columns (fp8 KV: the q rows of p_hi, then of p_lo).
constexpr uint32_t kColS = 0, kColO = 128;

// Byte offset of (row, byte x) inside a 128-byte-wide K-major operand with
// the 128-byte swizzle (8-row / 1024-byte atoms, 16-byte chunks XOR row%8).
__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t x) {
  return (row >> 3) * 1024u + (row & 7u) * 128u + ((((x >> 4) ^ row) & 7u) << 4) + (x & 15u);
}

// Walks the tiles of this CTA's items in order (items hold whole 128-token
// tiles except for a ragged last one).
struct TileCursor {
  const WorkItem* items;
  int it, it1, k;        // item index, end, item ordinal within the CTA
  int j, ntile;          // tile within the item
  uint32_t t;            // tile ordinal within the CTA
  WorkItem w;
  // `first` is a copy of items_[it0] (the CTA head), so starting costs no load
  __device__ __forceinline__ void init(const WorkItem* items_, int it0, int it1_,
                                       const WorkItem& first) {
    items = items_;
    it = it0;
    it1 = it1_;
    k = 0;
    j = 0;
    t = 0;
    if (it < it1) {
      w = first;
      ntile = (w.tok_end - w.tok_begin + kTile - 1) / kTile;
    } else {
      ntile = 0;
    }
  }
  __device__ __forceinline__ void load() {
    if (it < it1) {
      w = items[it];
      ntile = (w.tok_end - w.tok_begin + kTile - 1) / kTile;
    } else {
      ntile = 0;
    }
  }
  __device__ __forceinline__ bool done() const { return it >= it1; }
  __device__ __forceinline__ void advance() {
    ++t;
    if (++j == ntile) {
      ++it;
      ++k;
      j = 0;
      load();
    }
  }
  __device__ __forceinline__ int t0() const { return w.tok_begin + j * kTile; }
  __device__ __forceinline__ int nvalid() const { return min(kTile, w.tok_end - t0()); }
};

// What lane `lane` needs to issue its TMA box of one tile.  The page-table
// entry is loaded when the tile is looked ahead at and only checked (and
// turned into a row) when the box is issued, so the load overlaps the wait.
struct BoxFetch {
  int nbox;    // boxes of the tile (lanes [0, nbox) issue one each)
  int raw;     // page id as loaded (page table), or the row (identity table)
  int off;     // row offset inside the page
};

__device__ __forceinline__ BoxFetch box_fetch(const Stage1Params& p, const TileCursor& c,
                                              int lane) {
  BoxFetch f{0, 0, 0};
  if (c.done()) return f;
  f.nbox = (c.nvalid() + p.box_rows - 1) / p.box_rows;
  if (lane >= f.nbox) return f;
  const int pos = c.t0() + lane * p.box_rows;
  if (p.kv_indices == nullptr) {
    f.raw = c.w.page_base * p.page_size + pos;
  } else {
    f.raw = ld_nc_early(p.kv_indices + c.w.page_base + pos / p.page_size);
    f.off = pos % p.page_size;
  }
  return f;
}

__device__ __forceinline__ int box_row(const Stage1Params& p, const BoxFetch& f, int lane) {
  if (lane >= f.nbox) return 0;
  if (p.kv_indices == nullptr) return f.raw;
  int page = f.raw;
  if (page < 0 || static_cast<int64_t>(page + 1) * p.page_size > p.pool_rows) {
    atomicOr(p.err, kErrBadPage);
    page = 0;
  }
  return page * p.page_size + f.off;
}

// ---------------------------------------------------------------- producer
// One warp: lane i owns TMA box i of every tile.  Page-table entries are
// fetched two tiles ahead of the tile being issued.
template <int QM>
__device__ void run_producer(const Stage1Params& p, Misc* ms, uint32_t ring, int it0, int it1,
                             const WorkItem& first, int lane) {
  using L = Layout<QM>;
  const uint64_t pol = l2_policy_evict_first();
  const uint32_t box_bytes = static_cast<uint32_t>(p.box_rows) * L::kRowBytes;
  TileCursor cur, ahead;
  cur.init(p.items, it0, it1, first);
  ahead = cur;
  BoxFetch f0 = box_fetch(p, ahead, lane);
  ahead.advance();
  BoxFetch f1 = box_fetch(p, ahead, lane);
  ahead.advance();
  bool ok = true;
  uint32_t t = 0;
  while (!cur.done() && ok) {
    if (!L::kMx && p.gather) {
      // Page size not a multiple of 8: lane l copies rows l, l+32, l+64,
      // l+96 of the tile, each through its own page-table entry, in 16-byte
      // pieces into the identity-table layout ([chunk][128 rows][64 B], the
      // 64-byte swizzle), then arrives on the tile's barrier once its copies
      // have landed (32 arrivals per tile).  (Lanes on consecutive pieces of
      // one row, with the pool rows staged in shared memory, measured 2x
      // slower; a row's chunks are 8 KB apart there, so its pieces share
      // banks.)
      const uint32_t s = t % L::kNumTiles, ph = (t / L::kNumTiles) & 1u;
      const uint32_t full = smem_u32(&ms->full[s]);
      const int t0 = cur.t0(), nvalid = cur.nvalid();
      int32_t page[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {       // loaded before the waits, used after
        const int r = lane + 32 * j;
        page[j] = r < nvalid ? ld_nc_early(p.kv_indices + cur.w.page_base + (t0 + r) / p.page_size)
                             : 0;
      }
      // (the slot's previous tile must have landed before these arrivals)
      if (t >= static_cast<uint32_t>(L::kNumTiles)) {
        ok = __all_sync(0xffffffffu, mbar_wait(full, ph ^ 1u, p.err, kErrProducer));
        if (!ok) break;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->empty[s]), ph ^ 1u, p.err, kErrProducer));
      if (!ok) break;
      const uint32_t tile = ring + s * L::kTileBytes;
      const uint32_t cs = p.chunk_stride, gs = p.group_stride;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = lane + 32 * j;
        if (r >= nvalid) continue;
        int pg = page[j];
        if (pg < 0 || static_cast<int64_t>(pg + 1) * p.page_size > p.pool_rows) {
          atomicOr(p.err, kErrBadPage);
          pg = 0;
        }
        const int64_t grow = static_cast<int64_t>(pg) * p.page_size + (t0 + r) % p.page_size;
        const uint8_t* src = p.kv + grow * L::kRowBytes;
        const uint32_t dst = tile + (r >> 3) * gs + (r & 7) * 64u;
        const uint32_t swz = ((r & 7) >> 1) & 3u;
#pragma unroll 3
        for (int c = 0; c < L::kChunks; ++c)
#pragma unroll
          for (int q = 0; q < 4; ++q)
            cp_async_16(dst + c * cs + ((q ^ swz) << 4), src + c * 64 + q * 16);
      }
      cp_async_arrive(full);
      cur.advance();
      ++t;
      continue;
    }
    const BoxFetch f = f0;
    f0 = f1;
    f1 = box_fetch(p, ahead, lane);
    ahead.advance();
    const uint32_t s = t % L::kNumTiles, ph = (t / L::kNumTiles) & 1u;
    const uint32_t full = smem_u32(&ms->full[s]);
    const uint32_t raw_bytes = p.box_rows * L::kRawRowBytes;
    // Before waiting for the slot to be free: resolve the rows and arm the
    // slot's next full phase with the bytes to come.  That arrive must fall
    // in the next phase, so the slot's previous tile must have landed first
    // (it has, in the steady state); the armed phase cannot complete before
    // the copies, which are only issued once the slot is free.
    // Every lane waits: a lone lane-0 wait followed by a broadcast cost
    // about 1500 cycles of reconvergence per tile on GB300.
    const int row = box_row(p, f, lane);
    if (t >= static_cast<uint32_t>(L::kNumTiles)) {
      ok = __all_sync(0xffffffffu, mbar_wait(full, ph ^ 1u, p.err, kErrProducer));
      if (!ok) break;
    }
    if (lane == 0)
      mbar_arrive_expect_tx(full, static_cast<uint32_t>(f.nbox) * (L::kMx ? raw_bytes : box_bytes));
    // (MXFP4: the packed rows land in the upper box halves, free once PV has
    // read O blocks 2-3; the dequantisation waits for the whole slot)
    ok = __all_sync(0xffffffffu, mbar_wait(L::kMx ? smem_u32(&ms->upper_free[s]) : smem_u32(&ms->empty[s]),
                                           ph ^ 1u, p.err, kErrProducer));
    if (!ok) break;
    if constexpr (L::kMx) {
      // packed rows of box i into the upper half of box i's e4m3 region
      // (the e8m0 scale rows are read by the dequantising threads)
      if (lane < f.nbox)
        tma_load_3d(ring + s * L::kTileBytes + lane * box_bytes + raw_bytes, &p.tmap_kv, full, 0,
                    row, 0, pol);
    } else {
      if (lane < f.nbox)
        tma_load_3d(ring + s * L::kTileBytes + lane * box_bytes, &p.tmap_kv, full, 0, row, 0, pol);
    }
    cur.advance();
    ++t;
  }
  // Drain: wait (bounded) until the last copies issued into each tile landed.
  if (lane == 0) {
    const uint32_t n = t < static_cast<uint32_t>(L::kNumTiles) ? t : L::kNumTiles;
    for (uint32_t i = 0; i < n; ++i) {
      const uint32_t tt = t - 1 - i;
      if (!mbar_wait(smem_u32(&ms->full[tt % L::kNumTiles]), (tt / L::kNumTiles) & 1u, p.err,
                     kErrDrain))
        break;
    }
  }
}

// ---------------------------------------------------------- UMMA issuers
// QK^T issuer: S^T[sb] = K_tile . Q^T over kKSteps steps of 32 bytes.  The K
// tile is K-major with the 64-byte swizzle: column chunk j at j*cs, 8-row
// groups at gs.
template <int QM>
__device__ void run_qk(const Stage1Params& p, Misc* ms, uint32_t ring, uint32_t qbase,
                       uint32_t tmem, int it0, int it1, const WorkItem& first, int half,
                       int lane) {
  using L = Layout<QM>;
  constexpr uint32_t idesc = L::kKv8 ? make_idesc(0, 0, false, false, 128, L::kNq)
                                     : make_idesc(1, 1, false, false, 128, 16);
  const uint32_t cs = p.chunk_stride, gs = p.group_stride;
  TileCursor qc;
  qc.init(p.items, it0, it1, first);
  int q_ready = -1;
  while (!qc.done()) {
    const uint32_t t = qc.t, sb = t & 1u, s = t % L::kNumTiles;
    // the whole warp waits (converged); lane 0 issues
    if (q_ready != qc.k) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->q_full[qc.k & 1]), (qc.k >> 1) & 1,
                                             p.err, kErrMma)))
        break;
      q_ready = qc.k;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->s_empty[sb]), ((t >> 1) & 1u) ^ 1u,
                                           p.err, kErrMma)))
      break;
    // the tile is ready once it landed (MXFP4: once the dims of this K-half
    // were dequantised)
    const uint32_t ready = !L::kMx ? smem_u32(&ms->full[s])
                           : half == 0 ? smem_u32(&ms->deq_a[s]) : smem_u32(&ms->deq[s]);
    if (!__all_sync(0xffffffffu, mbar_wait(ready, (t / L::kNumTiles) & 1u, p.err, kErrMma)))
      break;
    tc_fence_after();
    if (p.gather) fence_proxy_async_smem();   // rows copied by cp.async (generic proxy)
    const uint32_t tile = ring + s * L::kTileBytes;
    const uint32_t qaddr = qbase + (qc.k & 1) * L::kQBytes;
    const uint32_t d = tmem + kColS + 64 * sb + 32 * half;
    const int k0 = half * (L::kKSteps / 2), k1 = k0 + L::kKSteps / 2;
    if (lane == 0) {
    // descriptors built once per tile; a K step only moves the start address
    const uint64_t a0 = smem_desc(tile, 16, gs, kSwizzle64B);
    const uint64_t b0 = smem_desc(qaddr, 16, 1024, kSwizzle128B);
#pragma unroll 3
    for (int kk = k0; kk < k1; ++kk) {
      const uint64_t a = a0 + (((kk >> 1) * cs + (kk & 1) * 32) >> 4);
      const uint64_t b = b0 + (((kk >> 2) * L::kQAtomBytes + (kk & 3) * 32) >> 4);
      if constexpr (L::kKv8)
        umma_f8f6f4(d, a, b, idesc, kk != k0);
      else
        umma_f16(d, a, b, idesc, kk != k0);
    }
    tc_commit(smem_u32(&ms->s_full[sb]));
    if (qc.j == qc.ntile - 1) tc_commit(smem_u32(&ms->q_empty[qc.k & 1]));
    }
    __syncwarp();
    qc.advance();
  }
  if (lane == 0) tc_commit(smem_u32(&ms->drain[half]));
  mbar_wait(smem_u32(&ms->drain[half]), 0, p.err, kErrDrain);
}

// PV issuer: O^T[128 dims of block c] (+)= V^T . P^T.  V^T is the tile read
// MN-major: 64-dim atoms at cs (LBO), 8-token groups at gs (SBO).  Issuer
// `half` owns O blocks 2*half, 2*half+1 (two issuers) or all four (one).
template <int QM>
__device__ void run_pv(const Stage1Params& p, Misc* ms, uint32_t ring, uint32_t pbase,
                       uint32_t tmem, int it0, int it1, const WorkItem& first, int half,
                       int lane) {
  using L = Layout<QM>;
  constexpr int kBlocks = 4 / L::kPvIssuers;
  const uint32_t cs = p.chunk_stride, gs = p.group_stride;
  TileCursor pc;
  pc.init(p.items, it0, it1, first);
  while (!pc.done()) {
    const uint32_t t = pc.t, pb = t & 1u, s = t % L::kNumTiles;
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->p_full[pb]), (t >> 1) & 1u, p.err,
                                           kErrMma)))
      break;
    tc_fence_after();
    if (p.gather) fence_proxy_async_smem();   // V rows copied by cp.async (generic proxy)
    const uint32_t tile = ring + s * L::kTileBytes;
    const uint32_t pa = pbase + pb * L::kPBytes;
    const bool first = pc.j == 0;
    if (lane == 0) {
    for (int i = 0; i < kBlocks; ++i) {
      // MXFP4 (one issuer): O blocks 2-3 first.  Their V chunks 4-7 and the
      // rope chunk 8 are the upper half of every 8-row box, where the next
      // packed rows land, so the producer may refill the slot as soon as
      // they are read; blocks 0-1 follow.
      const int c = L::kMx ? (i + 2) & 3 : kBlocks * half + i;
      const uint32_t d = tmem + kColO + L::kOCols * c;
      // B = P^T, MN-major: one kPRow-byte row per token (fp8: the q rows of
      // p_hi then of p_lo; bf16: the q rows), 8-token groups of 8 rows, with
      // the swizzle of the row width (32 or 64 bytes).
      constexpr uint32_t kPGroup = 8 * L::kPRow;
      const uint64_t b0 =
          smem_desc(pa, kPGroup, kPGroup, L::kPRow == 64 ? kSwizzle64B : kSwizzle32B);
      if constexpr (L::kKv8) {
        constexpr uint32_t idesc = make_idesc(0, 0, true, true, 128, L::kOCols);
        const uint64_t a0 = smem_desc(tile + (2 * c) * cs, cs, gs, kSwizzle64B);  // 2 chunks
        for (int kk = 0; kk < 4; ++kk) {                          // 32 tokens = 4 groups
          const uint64_t a = a0 + ((kk * 4 * gs) >> 4);
          const uint64_t b = b0 + ((kk * 4 * kPGroup) >> 4);
          umma_f8f6f4(d, a, b, idesc, (first && kk == 0) ? 0u : 1u);
        }
      } else {
        constexpr uint32_t idesc = make_idesc(1, 1, true, true, 128, L::kOCols);
        const uint64_t a0 = smem_desc(tile + (4 * c) * cs, cs, gs, kSwizzle64B);  // 4 chunks
        for (int kk = 0; kk < 8; ++kk) {                          // 16 tokens = 2 groups
          const uint64_t a = a0 + ((kk * 2 * gs) >> 4);
          const uint64_t b = b0 + ((kk * 2 * kPGroup) >> 4);
          umma_f16(d, a, b, idesc, (first && kk == 0) ? 0u : 1u);
        }
      }
      if (L::kMx && i == 1) tc_commit(smem_u32(&ms->upper_free[s]));
    }
    tc_commit(smem_u32(&ms->pv_done[pb]));
    tc_commit(smem_u32(&ms->empty[s]));      // QK^T of this tile completed before P existed
    }
    __syncwarp();
    pc.advance();
  }
  if (lane == 0) tc_commit(smem_u32(&ms->drain[2 + half]));
  mbar_wait(smem_u32(&ms->drain[2 + half]), 0, p.err, kErrDrain);
}

// ------------------------------------------------------ MXFP4 dequantise
// e4m3 bytes of m * 2^k for the eight e2m1 magnitudes m = {0, .5, 1, 1.5, 2,
// 3, 4, 6} (byte c of {lo, hi} = code c).  k <= 0; 2^k below 2^-126 flushes
// the block to zero (it is then below 2^-126 of the row's largest block).
// A block uses one of 15 tables (k = 0 .. -14; from k = -14 down every entry
// rounds to 0, below half the smallest e4m3 subnormal); the dequant warps
// build them once per CTA.
__device__ __forceinline__ void e2m1_e4m3_table(int k, uint32_t& lo, uint32_t& hi) {
  const float f = k >= -126 ? __int_as_float((k + 127) << 23) : 0.0f;
  const uint32_t a = __nv_cvt_float2_to_fp8x2(make_float2(0.0f, 0.5f * f), __NV_SATFINITE, __NV_E4M3);
  const uint32_t b = __nv_cvt_float2_to_fp8x2(make_float2(1.0f * f, 1.5f * f), __NV_SATFINITE, __NV_E4M3);
  const uint32_t c = __nv_cvt_float2_to_fp8x2(make_float2(2.0f * f, 3.0f * f), __NV_SATFINITE, __NV_E4M3);
  const uint32_t d = __nv_cvt_float2_to_fp8x2(make_float2(4.0f * f, 6.0f * f), __NV_SATFINITE, __NV_E4M3);
  lo = a | (b << 16);
  hi = c | (d << 16);
}

// Eight packed e2m1 codes (nibble n = element n) -> eight e4m3 bytes: the
// magnitude through the table (byte permute with the sign bits cleared), the
// sign from bit 3 of each nibble.  That bit is the msb of byte n/2 of w << 4
// (n even) or of w (n odd), so a byte permute that replicates msbs turns it
// into a 0x00 / 0xFF mask per output byte.
__device__ __forceinline__ uint2 e2m1x8_to_e4m3(uint32_t w, uint32_t lo, uint32_t hi) {
  const uint32_t sel = w & 0x77777777u;
  const uint32_t m0 = prmt(lo, hi, sel), m1 = prmt(lo, hi, sel >> 16);
  const uint32_t w4 = w << 4;
  const uint32_t s0 = prmt(w4, w, 0xD9C8u), s1 = prmt(w4, w, 0xFBEAu);
  return make_uint2(m0 | (s0 & 0x80808080u), m1 | (s1 & 0x80808080u));
}

// ------------------------------------------------------- MXFP4 scale rows
// The dequantising thread of token `tq` reads that token's 18 e8m0 bytes
// from global memory itself (no TMA box: the pages' scale rows are 18 bytes,
// which no tensor map can stride over).  The row is found as the producer
// finds it: through the page table, a page outside the pool replaced by page
// 0.  The loads of a tile are issued one tile ahead and its page-table entry
// two tiles ahead, so neither waits on the path.

// Raw page-table entry of token tq of the cursor's tile (0 for the identity
// table or a token past the tile's end).
__device__ __forceinline__ int32_t scale_page(const Stage1Params& p, const TileCursor& c, int tq) {
  if (c.done() || tq >= c.nvalid() || p.kv_indices == nullptr) return 0;
  return ld_nc_early(p.kv_indices + c.w.page_base + (c.t0() + tq) / p.page_size);
}

// Issues the nine 2-byte loads of the token's scale row (zeros past the
// tile's end); `page` is scale_page() of the same tile and token.
__device__ __forceinline__ void scale_load(const Stage1Params& p, const TileCursor& c, int tq,
                                           int32_t page, uint16_t (&h)[9]) {
  if (c.done() || tq >= c.nvalid()) {
#pragma unroll
    for (int i = 0; i < 9; ++i) h[i] = 0;
    return;
  }
  const int pos = c.t0() + tq;
  int64_t row;
  if (p.kv_indices == nullptr) {
    row = static_cast<int64_t>(c.w.page_base) * p.page_size + pos;
    if (row >= p.pool_rows) row = 0;   // (the host rejects such plans; never reached)
  } else {
    if (page < 0 || static_cast<int64_t>(page + 1) * p.page_size > p.pool_rows) {
      atomicOr(p.err, kErrBadPage);
      page = 0;
    }
    row = static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
  }
  const uint16_t* src = reinterpret_cast<const uint16_t*>(p.kv_e8m0 + row * p.sc_stride);
#pragma unroll
  for (int i = 0; i < 9; ++i) h[i] = ld_nc_u16_early(src + i);
}

// ----------------------------------------------------- q staging helpers
// One bulk copy brings q of request `bb` (all its q rows) into the staging buffer.
template <int QM>
__device__ __forceinline__ void q_fetch(const Stage1Params& p, Misc* ms, uint8_t* stage, int bb) {
  using L = Layout<QM>;
  const uint32_t bar = smem_u32(&ms->q_stage);
  mbar_arrive_expect_tx(bar, L::kQSrcBytes);
  bulk_load(smem_u32(stage), static_cast<const uint8_t*>(p.q) + static_cast<int64_t>(bb) * L::kQSrcBytes,
            L::kQSrcBytes, bar);
}

// Eight bf16 q values (vector `vid` of the [16 heads][576] q) -> their e4m3
// q_hi = rn(q / s_hi) and q_lo = rn(16 (q - q_hi s_hi) / s_hi) bytes, stored
// as rows h and 16 + h of the K-major, 128-byte-swizzled q operand.
__device__ __forceinline__ void q_split_store(const uint4 v, int vid, float s_hi, float inv_hi,
                                              uint8_t* dst, int atom_bytes) {
  const int h = vid / 72, d0 = (vid % 72) * 8;
  const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&v);
  uint32_t hw[2], lw[2];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(h2[e]);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(f.x * inv_hi, f.y * inv_hi), __NV_SATFINITE, __NV_E4M3);
    const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
    const float rx = (f.x - hf.x * s_hi) * inv_hi * 16.0f;
    const float ry = (f.y - hf.y * s_hi) * inv_hi * 16.0f;
    const __nv_fp8x2_storage_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(rx, ry), __NV_SATFINITE, __NV_E4M3);
    const int wd = e >> 1, sh = (e & 1) * 16;
    if ((e & 1) == 0) { hw[wd] = 0; lw[wd] = 0; }
    hw[wd] |= static_cast<uint32_t>(hi) << sh;
    lw[wd] |= static_cast<uint32_t>(lo) << sh;
  }
  const int atom = d0 >> 7, x = d0 & 127;
  uint8_t* base = dst + atom * atom_bytes;
  *reinterpret_cast<uint2*>(base + sw128(h, x)) = make_uint2(hw[0], hw[1]);
  *reinterpret_cast<uint2*>(base + sw128(16 + h, x)) = make_uint2(lw[0], lw[1]);
}

// Writes q of one request from the staging buffer into q buffer `dst` (the
// UMMA B operand) with n threads (this is thread i, n a multiple of 32) and
// returns the two score factors.  A bf16 q meeting fp8 or MXFP4 KV is split
// into two e4m3 terms with one scale for the request, which needs |q|max
// over all n threads: warp shuffles, then (n > 32) ms->qred and named
// barrier `bar`.  The caller fences and publishes the buffer.
template <int QM>
__device__ __forceinline__ void q_convert(const Stage1Params& p, Misc* ms, const uint8_t* stage,
                                          uint8_t* dst, int i, int n, int bar, float& c_hi,
                                          float& c_lo) {
  using L = Layout<QM>;
  constexpr float kSmScale = 1.0f / 24.0f;          // 1/sqrt(576)
  c_lo = 0.f;
  if constexpr (QM == kQBf16KvFp8 || QM == kQBf16KvMx) {
    constexpr int kV = L::kQSrcBytes / 16;           // 16-byte vectors of 8 bf16
    const uint4* src = reinterpret_cast<const uint4*>(stage);
    float amax = 0.f;
    for (int v = i; v < kV; v += n) {
      const uint4 x = src[v];
      const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h2[e]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (n > 32) {
      if ((i & 31) == 0) ms->qred[i >> 5] = amax;
      named_bar_sync(bar, n);
      amax = 0.f;
      for (int w = 0; w < n / 32; ++w) amax = fmaxf(amax, ms->qred[w]);
    }
    amax = fmaxf(amax, 1e-30f);
    const float s_hi = amax / 448.0f, inv_hi = 448.0f / amax;
    for (int v = i; v < kV; v += n) q_split_store(src[v], v, s_hi, inv_hi, dst, L::kQAtomBytes);
    const float kvs = (QM == kQBf16KvMx) ? 1.0f : __ldg(p.kv_scale);
    c_hi = s_hi * kvs * kSmScale * kLog2e;
    c_lo = c_hi * (1.0f / 16.0f);
  } else if constexpr (QM == kQFp8KvFp8 || QM == kQFp8KvFp8x2) {
    const uint4* src = reinterpret_cast<const uint4*>(stage);
    for (int v = i; v < L::kRows * 36; v += n) {     // 36 vectors of 16 e4m3 per q row
      const int h = v / 36, d0 = (v % 36) * 16;
      *reinterpret_cast<uint4*>(dst + (d0 >> 7) * L::kQAtomBytes + sw128(h, d0 & 127)) = src[v];
    }
    c_hi = __ldg(p.q_scale) * __ldg(p.kv_scale) * kSmScale * kLog2e;
  } else {
    // bf16 operand for kind::f16; fp8 q is decoded exactly to bf16 first.
    for (int v = i; v < kHeads * 72; v += n) {       // 72 vectors of 8 values per head
      const int h = v / 72, d0 = (v % 72) * 8;
      uint4 x;
      if constexpr (QM == kQBf16KvBf16) {
        x = reinterpret_cast<const uint4*>(stage)[v];
      } else {
        const uint2 raw = reinterpret_cast<const uint2*>(stage)[v];
        uint32_t wv[4];
        const uint32_t rr[2] = {raw.x, raw.y};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_fp8x2_storage_t pr =
              static_cast<__nv_fp8x2_storage_t>((rr[e >> 1] >> ((e & 1) * 16)) & 0xFFFFu);
          const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3)));
          const __nv_bfloat162 bb = __float22bfloat162_rn(f);
          wv[e] = *reinterpret_cast<const uint32_t*>(&bb);
        }
        x = make_uint4(wv[0], wv[1], wv[2], wv[3]);
      }
      const int atom = d0 >> 6, xb = (d0 & 63) * 2;
      *reinterpret_cast<uint4*>(dst + atom * L::kQAtomBytes + sw128(h, xb)) = x;
    }
    c_hi = (QM == kQFp8KvBf16 ? __ldg(p.q_scale) : 1.0f) * kSmScale * kLog2e;
  }
}

// MXFP4 variant: the four dequant warps (128 threads, named barrier 3)
// prepare q of item `it` (ordinal k) into q buffer k & 1, then start the copy
// of the next item's q.  Returns false once the group gave up.
template <int QM>
__device__ bool qprep_group(const Stage1Params& p, Misc* ms, uint8_t* qgen, uint8_t* stage, int it,
                            int k, int it1, int t) {
  using L = Layout<QM>;
  volatile int32_t* abort = &ms->abort_dq;
  const uint32_t qb = k & 1;
  if (!mbar_wait(smem_u32(&ms->q_empty[qb]), ((k >> 1) & 1) ^ 1, p.err, kErrQPrep)) *abort = 1;
  if (!mbar_wait(smem_u32(&ms->q_stage), k & 1, p.err, kErrQPrep)) *abort = 1;
  named_bar_sync(3, 128);
  if (*abort) return false;
  float c_hi, c_lo;
  q_convert<QM>(p, ms, stage, qgen + qb * L::kQBytes, t, 128, 3, c_hi, c_lo);
  fence_proxy_async_smem();
  named_bar_sync(3, 128);                           // staging buffer and qred free again
  if (t == 0) {
    if (it + 1 < it1) q_fetch<QM>(p, ms, stage, p.items[it + 1].b);
    ms->qscale[qb][0] = c_hi;
    ms->qscale[qb][1] = c_lo;
    mbar_arrive(smem_u32(&ms->q_full[qb]));
  }
  return true;
}

// Four warps turn the packed MXFP4 rows of a tile slot into the e4m3 tile the
// UMMAs read (thread t = token t).  With r_t the largest e8m0 exponent of the
// token, block b becomes e2m1 * 2^(E_b - r_t): exact in e4m3 while
// E_b - r_t >= -8.  The remaining factor 2^(r_t - 127) of the token is left
// to the softmax (u_t = r_t - 127 in shared memory).
//
// In place, without holding a row in registers: 8-row box i of the slot owns
// bytes [i*4608, (i+1)*4608) of e4m3 rows ([chunk c][8 rows][64 B], chunk c =
// dims 64c..64c+63) and its packed rows land chunk-major in the upper half,
// [chunk c][8 rows][32 B] at 2304 + 256c.  Packed chunk c therefore lies in
// e4m3 chunk floor(4.5 + c/2) >= c, so writing e4m3 chunk c only overwrites
// packed chunks the box's 8 threads (one quarter of a warp) have already
// read: a warp barrier between the reads and the writes of each chunk is
// enough.
//
// The same threads prepare q: item 0's before the first tile, item k+1's
// right after the first tile of item k (its q buffer is free by then: QK^T
// of item k-1 has been issued on tiles this group already dequantised).
template <int QM>
__device__ void run_dequant(const Stage1Params& p, Misc* ms, uint8_t* ring_gen, uint8_t* qgen,
                            uint8_t* stage, int it0, int it1, const WorkItem& first, int t) {
  using L = Layout<QM>;
  static_assert(L::kRowBytes * 8 == 4608 && L::kRawRowBytes * 8 == 2304, "box layout");
  volatile int32_t* abort = &ms->abort_dq;
  if (it0 >= it1) return;
  if (t == 0) q_fetch<QM>(p, ms, stage, first.b);
  if (t < 15) {
    uint32_t lo, hi;
    e2m1_e4m3_table(t - 14, lo, hi);
    ms->e2m1_tab[t] = make_uint2(lo, hi);
  }
  // (qprep_group and every tile begin with a group barrier, so the tables
  // are visible before their first use)
  if (!qprep_group<QM>(p, ms, qgen, stage, it0, 0, it1, t)) return;
  // this thread's row: box t/8, row t%8 (8-row boxes)
  const uint32_t box_off = (t >> 3) * 4608u, r8 = t & 7u;
  const uint32_t swz = (r8 >> 1) & 3u;                 // 64-byte swizzle of this row
  // this thread's copy of its token's scale row (nine 2-byte block pairs)
  uint16_t* sc = reinterpret_cast<uint16_t*>(ring_gen + L::kScRowOff + t * 24);
  TileCursor c, a1, a2;                                // this tile, the next, the one after
  c.init(p.items, it0, it1, first);
  a1 = c;
  a1.advance();
  a2 = a1;
  a2.advance();
  uint16_t h[9];
  scale_load(p, c, t, scale_page(p, c, t), h);
  int32_t page1 = scale_page(p, a1, t);
  while (!c.done()) {
    const uint32_t tt = c.t, s = tt % L::kNumTiles;
    // this tile's scale bytes into shared memory, then the next tile's loads
    int r = 0;
    {
      uint32_t ew[5];
#pragma unroll
      for (int i = 0; i < 4; ++i) ew[i] = h[2 * i] | (static_cast<uint32_t>(h[2 * i + 1]) << 16);
      ew[4] = h[8];
      *reinterpret_cast<uint2*>(sc) = make_uint2(ew[0], ew[1]);
      *reinterpret_cast<uint2*>(sc + 4) = make_uint2(ew[2], ew[3]);
      *reinterpret_cast<uint32_t*>(sc + 8) = ew[4];
#pragma unroll
      for (int b = 0; b < 18; ++b)
        r = max(r, static_cast<int>((ew[b >> 2] >> ((b & 3) * 8)) & 0xFFu));
    }
    scale_load(p, a1, t, page1, h);
    page1 = scale_page(p, a2, t);
    if (!mbar_wait(smem_u32(&ms->full[s]), (tt / L::kNumTiles) & 1u, p.err, kErrDequant)) *abort = 1;
    // e4m3 rows are written over the whole slot: PV of its previous tile
    // must have finished (the packed rows only needed the upper halves)
    if (!mbar_wait(smem_u32(&ms->empty[s]), ((tt / L::kNumTiles) & 1u) ^ 1u, p.err, kErrDequant))
      *abort = 1;
    named_bar_sync(3, 128);
    if (*abort) return;
    uint8_t* box = ring_gen + s * L::kTileBytes + box_off;
    const uint8_t* raw = box + 2304u + r8 * 32u;
    ms->uexp[s][t] = static_cast<float>(r - 127);
    uint8_t* row = box + r8 * 64u;
    // packed chunk ch+1 and its two scale bytes are read while chunk ch is
    // converted (reading early is always safe; only writes must wait)
    uint4 na = reinterpret_cast<const uint4*>(raw)[0];
    uint4 nb = reinterpret_cast<const uint4*>(raw)[1];
    uint32_t neb = sc[0];
    auto chunk = [&](int ch, bool sync) {
      const uint4 a = na, b = nb;
      const uint32_t eb = neb;                          // e8m0 of blocks 2ch, 2ch+1
      if (ch < 8) {
        na = reinterpret_cast<const uint4*>(raw + (ch + 1) * 256)[0];
        nb = reinterpret_cast<const uint4*>(raw + (ch + 1) * 256)[1];
        neb = sc[ch + 1];
      }
      if (sync) __syncwarp();                           // the box read the packed chunks
      const uint2 t0 = ms->e2m1_tab[max(static_cast<int>(eb & 0xFFu) - r, -14) + 14];
      const uint2 t1 = ms->e2m1_tab[max(static_cast<int>(eb >> 8) - r, -14) + 14];
      const uint32_t lo0 = t0.x, hi0 = t0.y, lo1 = t1.x, hi1 = t1.y;
      const uint2 o0 = e2m1x8_to_e4m3(a.x, lo0, hi0), o1 = e2m1x8_to_e4m3(a.y, lo0, hi0);
      const uint2 o2 = e2m1x8_to_e4m3(a.z, lo0, hi0), o3 = e2m1x8_to_e4m3(a.w, lo0, hi0);
      const uint2 o4 = e2m1x8_to_e4m3(b.x, lo1, hi1), o5 = e2m1x8_to_e4m3(b.y, lo1, hi1);
      const uint2 o6 = e2m1x8_to_e4m3(b.z, lo1, hi1), o7 = e2m1x8_to_e4m3(b.w, lo1, hi1);
      uint8_t* dst = row + ch * 512;
      *reinterpret_cast<uint4*>(dst + ((0u ^ swz) << 4)) = make_uint4(o0.x, o0.y, o1.x, o1.y);
      *reinterpret_cast<uint4*>(dst + ((1u ^ swz) << 4)) = make_uint4(o2.x, o2.y, o3.x, o3.y);
      *reinterpret_cast<uint4*>(dst + ((2u ^ swz) << 4)) = make_uint4(o4.x, o4.y, o5.x, o5.y);
      *reinterpret_cast<uint4*>(dst + ((3u ^ swz) << 4)) = make_uint4(o6.x, o6.y, o7.x, o7.y);
    };
    // e4m3 chunks 0-3 lie below every packed chunk: no barrier.  From chunk
    // 4 on, e4m3 chunk ch overwrites packed chunks 2ch-9 and 2ch-8, which
    // the box's threads read (one chunk ahead) in earlier iterations: a warp
    // barrier before each write orders those reads first.
#pragma unroll 1
    for (int ch = 0; ch < 4; ++ch) chunk(ch, false);
#pragma unroll 1
    for (int ch = 4; ch < 9; ++ch) {
      chunk(ch, true);
      if (ch == 4) {
        // dims 0-319 done: the first QK^T K-half (dims 0-287) may start
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&ms->deq_a[s]));
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(smem_u32(&ms->deq[s]));
    const bool first = c.j == 0;
    const int it = c.it, k = c.k;
    c.advance();
    a1 = a2;
    a2.advance();
    if (first && it + 1 < it1 && !qprep_group<QM>(p, ms, qgen, stage, it + 1, k + 1, it1, t)) return;
  }
}

// Softmax threads share named barriers, so a thread must never leave alone:
// a wait that gives up raises the group's abort flag and the thread carries
// on to the next named barrier, after which the whole group leaves.
__device__ __forceinline__ void wait_or_flag(uint32_t bar, uint32_t parity, int32_t* err,
                                             int32_t code, volatile int32_t* flag) {
  if (!mbar_wait(bar, parity, err, code)) *flag = 1;
}

// -------------------------------------------------------------- q prepare
// One bulk copy per request brings q into the staging buffer.  The first
// item's q gates the first QK^T, so the softmax warps (idle until then)
// convert it together; this warp converts the q of every later item into the
// free q buffer, off the critical path, and starts the next copy as soon as
// the staging buffer is free.
template <int QM>
__device__ void run_qprep(const Stage1Params& p, Misc* ms, uint8_t* qgen, uint8_t* stage, int it0,
                          int it1, const WorkItem& first, int lane) {
  using L = Layout<QM>;
  const uint32_t stage_bar = smem_u32(&ms->q_stage);
  if (it0 >= it1) return;
  if (lane == 0) q_fetch<QM>(p, ms, stage, first.b);
  if (it0 + 1 >= it1) return;
  // the softmax warps are done with the first item's staged q
  if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->q_stage_free), 0, p.err, kErrQPrep))) return;
  if (lane == 0) q_fetch<QM>(p, ms, stage, p.items[it0 + 1].b);
  int k = 1;
  for (int it = it0 + 1; it < it1; ++it, ++k) {
    const uint32_t qb = k & 1;
    if (!__all_sync(0xffffffffu,
                    mbar_wait(smem_u32(&ms->q_empty[qb]), ((k >> 1) & 1) ^ 1, p.err, kErrQPrep)))
      return;
    if (!__all_sync(0xffffffffu, mbar_wait(stage_bar, k & 1, p.err, kErrQPrep))) return;
    float c_hi, c_lo;
    q_convert<QM>(p, ms, stage, qgen + qb * L::kQBytes, lane, 32, 0, c_hi, c_lo);
    fence_proxy_async_smem();
    __syncwarp();                                     // every lane is done with the stage
    if (lane == 0) {
      if (it + 1 < it1) q_fetch<QM>(p, ms, stage, p.items[it + 1].b);
      ms->qscale[qb][0] = c_hi;
      ms->qscale[qb][1] = c_lo;
      mbar_arrive(smem_u32(&ms->q_full[qb]));
    }
  }
}

// ------------------------------------------------------ softmax / epilogue
// Reduce kH per-thread values (q rows h0..h0+kH-1) over the 128 threads of a
// head group (op = max or sum).  A transpose-reduce over the lane bits
// 16, 8, ... leaves one head per group of lanes after log2(kH) shuffle
// stages; the four warp results meet in shared memory behind the group's
// named barrier `bar`.
template <bool kMax, int kH>
__device__ __forceinline__ void reduce_heads(const float (&v)[kH], float (&out)[kH],
                                             float (*red)[32], int h0, int qw, int lane, int bar) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  constexpr int kStages = kH == 16 ? 4 : 3;
  float buf[kH];
#pragma unroll
  for (int i = 0; i < kH; ++i) buf[i] = v[i];
  int h = 0;
#pragma unroll
  for (int st = 0; st < kStages; ++st) {
    const int half = kH >> (st + 1), off = 16 >> st;
    const bool up = lane & off;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? buf[i] : buf[i + half], keep = up ? buf[i + half] : buf[i];
      buf[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
    if (up) h += half;
  }
#pragma unroll
  for (int off = 16 >> kStages; off >= 1; off >>= 1)
    buf[0] = op(buf[0], __shfl_xor_sync(0xffffffffu, buf[0], off));
  if ((lane & ((32 >> kStages) - 1)) == 0) red[qw][h0 + h] = buf[0];
  named_bar_sync(bar, 128);
#pragma unroll
  for (int i = 0; i < kH; ++i)
    out[i] = op(op(red[0][h0 + i], red[1][h0 + i]), op(red[2][h0 + i], red[3][h0 + i]));
}

// Softmax warps: kHeadGroups groups of four warps (one per TMEM lane
// quadrant); thread tq of a group owns token tq of every tile (its TMEM lane)
// and q rows h0..h0+kH-1 (one query token: 8 of its heads, or with two query
// tokens all 16 heads of token hg).  Per tile: S from TMEM, the running max,
// the lazy rescale of O, p = exp2(s - m + 4) into l and into the P operand.
// After an item's last tile, the epilogue normalises O and writes it out.
template <int QM>
__device__ void run_softmax(const Stage1Params& p, Misc* ms, uint8_t* ring_gen, uint8_t* pgen,
                            uint8_t* qgen, uint8_t* stage, uint32_t tmem, int it0, int it1,
                            const WorkItem& first, int tid) {
  using L = Layout<QM>;
  constexpr int kHG = L::kHeadGroups, kH = L::kH;
  volatile int32_t* abort = &ms->abort_sm;
  const int hg = tid >> 7, tq = tid & 127;
  const int h0 = kH * hg, bar = 1 + hg;
  const int qw = tq >> 5, lane = tq & 31;
  const uint32_t tl = tmem + (static_cast<uint32_t>(qw * 32) << 16);   // this warp's lanes
  uint32_t g = 0;
  const uint32_t cs = p.chunk_stride, gs = p.group_stride;
  if constexpr (!L::kMx) {
    if (it0 < it1) {
      // The first item's q gates the first QK^T: all softmax threads convert
      // it (into q buffer 0) while they would otherwise wait for S.
      constexpr int kN = 128 * kHG;
      wait_or_flag(smem_u32(&ms->q_stage), 0, p.err, kErrSoftmax, abort);
      named_bar_sync(6, kN);
      if (*abort) return;
      float c_hi, c_lo;
      q_convert<QM>(p, ms, stage, qgen, tid, kN, 6, c_hi, c_lo);
      fence_proxy_async_smem();
      named_bar_sync(6, kN);
      if (tid == 0) {
        ms->qscale[0][0] = c_hi;
        ms->qscale[0][1] = c_lo;
        mbar_arrive(smem_u32(&ms->q_full[0]));
        mbar_arrive(smem_u32(&ms->q_stage_free));
      }
    }
  }
  int k = 0;
  float m[kH], l[kH];
  for (int it = it0; it < it1; ++it, ++k) {
    const WorkItem w = it == it0 ? first : p.items[it];
    const uint32_t qb = k & 1;
    wait_or_flag(smem_u32(&ms->q_full[qb]), (k >> 1) & 1, p.err, kErrSoftmax, abort);
    const float c_hi = ms->qscale[qb][0], c_lo = ms->qscale[qb][1];
    named_bar_sync(bar, 128);
    if (*abort) return;
    if (tq == 0) mbar_arrive(smem_u32(&ms->q_empty[qb]));
    const int ntile = (w.tok_end - w.tok_begin + kTile - 1) / kTile;
    for (int j = 0; j < ntile; ++j, ++g) {
      const uint32_t sb = g & 1u;
      wait_or_flag(smem_u32(&ms->s_full[sb]), (g >> 1) & 1u, p.err, kErrSoftmax, abort);
      tc_fence_after();
      float s[kH];
      {
        // S^T columns of buffer sb: two K-halves of 32 columns; q split in two
        // terms puts the rows of q_hi first, then those of q_lo
        const uint32_t sc = tl + kColS + 64 * sb + h0;
        float a0[kH], a1[kH];
        tmem_ld(sc, a0);
        tmem_ld(sc + 32, a1);
        if constexpr (L::kHiLo) {
          float b0[kH], b1[kH];
          tmem_ld(sc + L::kRows, b0);
          tmem_ld(sc + 32 + L::kRows, b1);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kH; ++h) s[h] = (a0[h] + a1[h]) * c_hi + (b0[h] + b1[h]) * c_lo;
        } else {
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < kH; ++h) s[h] = (a0[h] + a1[h]) * c_hi;
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&ms->s_empty[sb]));
      const int nvalid = min(kTile, w.tok_end - (w.tok_begin + j * kTile));
      const bool valid = tq < nvalid;
      // two query tokens: query token hg sees the request's first vis0 + hg
      // tokens (causal over the last two positions)
      bool vis = valid;
      if constexpr (L::kQL > 1) vis = valid && w.tok_begin + j * kTile + tq < w.vis0 + hg;
      // MXFP4: the token's scores carry its factor 2^u; the running max and
      // P use s + u (the factor of its V row), l uses s: P' = p 2^u.
      float gl = 1.0f;                                   // 2^-u, turns P' back into p
      if constexpr (L::kMx) {
        const int u = static_cast<int>(ms->uexp[g % L::kNumTiles][tq]);
        const float f = u >= -126 ? __int_as_float((u + 127) << 23) : 0.0f;
        gl = (valid && u <= 126) ? __int_as_float((127 - u) << 23) : 0.0f;
#pragma unroll
        for (int h = 0; h < kH; ++h) s[h] = s[h] * f + static_cast<float>(u);
      }
#pragma unroll
      for (int h = 0; h < kH; ++h) s[h] = vis ? s[h] : -INFINITY;
      // The running max only moves when some score of the tile exceeds it by
      // more than kTau (always on an item's first tile).  One barrier vote
      // settles that; only then is the tile max reduced over the group.
      bool over = j == 0;
#pragma unroll
      for (int h = 0; h < kH; ++h) over |= s[h] > m[h] + kTau;
      over = named_bar_any(4 + hg, 128, over);
      if (*abort) return;
      bool resc = false;
      float alpha[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) alpha[h] = 1.0f;
      if (over) {
        float mt[kH];
        reduce_heads<true, kH>(s, mt, ms->red[g & 1u], h0, qw, lane, bar);
        if (*abort) return;
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          if (j == 0) {
            m[h] = mt[h];
            l[h] = 0.0f;
          } else if (mt[h] > m[h] + kTau) {
            alpha[h] = ex2(m[h] - mt[h]);
            m[h] = mt[h];
            resc = true;
          }
        }
      }
      if (resc) {
        // The running max moved by more than kTau: scale this group's O
        // columns (both parts) once the previous tile's PV has landed.
        const uint32_t gp = g - 1;
        wait_or_flag(smem_u32(&ms->pv_done[gp & 1u]), (gp >> 1) & 1u, p.err, kErrSoftmax, abort);
        tc_fence_after();
        const int nparts = L::kKv8 ? 2 : 1;
        for (int part = 0; part < nparts; ++part) {
          for (int c = 0; c < 4; ++c) {
            const uint32_t col = kColO + L::kOCols * c + L::kRows * part + h0;
            float o[kH];
            tmem_ld(tl + col, o);
            tmem_wait_ld();
#pragma unroll
            for (int h = 0; h < kH; ++h) o[h] *= alpha[h];
            tmem_st(tl + col, o);
          }
        }
        tmem_wait_st();
#pragma unroll
        for (int h = 0; h < kH; ++h) l[h] *= alpha[h];
      }
      float pv[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) {
        pv[h] = vis ? ex2(s[h] - m[h] + kPOff) : 0.0f;
        l[h] += L::kMx ? pv[h] * gl : pv[h];
      }
      // P buffer (g & 1) is free once PV of tile g-2 completed.
      if (g >= 2)
        wait_or_flag(smem_u32(&ms->pv_done[sb]), ((g >> 1) - 1) & 1u, p.err, kErrSoftmax, abort);
      // This token's row of P^T.  32-byte rows: two 16-byte halves swapped
      // on every other group of 4 tokens (32-byte swizzle: bit 4 ^= bit 7).
      // 64-byte rows (two query tokens): 16-byte chunk c at c ^ ((tq >> 1) & 3)
      // (64-byte swizzle), 8-token groups of 512 bytes.
      uint8_t* prow = pgen + sb * L::kPBytes + tq * L::kPRow;
      const uint32_t flip = ((tq >> 2) & 1u) << 4;
      const uint32_t sw64 = (tq >> 1) & 3u;
      if constexpr (L::kKv8) {
        // fp8: p_hi of the q rows, then p_lo of the q rows (one byte each)
        uint32_t hw[kH / 4], lw[kH / 4];
#pragma unroll
        for (int h = 0; h < kH; h += 2) {
          const __nv_fp8x2_storage_t hi =
              __nv_cvt_float2_to_fp8x2(make_float2(pv[h], pv[h + 1]), __NV_SATFINITE, __NV_E4M3);
          const float2 hf = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
          const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2((pv[h] - hf.x) * kPLoScale, (pv[h + 1] - hf.y) * kPLoScale),
              __NV_SATFINITE, __NV_E4M3);
          const int wd = h >> 2, sh = (h & 2) * 8;
          if ((h & 2) == 0) { hw[wd] = 0; lw[wd] = 0; }
          hw[wd] |= static_cast<uint32_t>(hi) << sh;
          lw[wd] |= static_cast<uint32_t>(lo) << sh;
        }
        if constexpr (L::kPRow == 64) {
          // [p_hi token 0 | p_hi token 1 | p_lo token 0 | p_lo token 1]
          *reinterpret_cast<uint4*>(prow + ((static_cast<uint32_t>(hg) ^ sw64) << 4)) =
              make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(prow + (((2u + hg) ^ sw64) << 4)) =
              make_uint4(lw[0], lw[1], lw[2], lw[3]);
        } else {
          *reinterpret_cast<uint2*>(prow + ((8u * hg) ^ flip)) = make_uint2(hw[0], hw[1]);
          *reinterpret_cast<uint2*>(prow + ((16u + 8u * hg) ^ flip)) = make_uint2(lw[0], lw[1]);
        }
      } else {
        // bf16: the 16 heads, 2 bytes each
        uint32_t bw[kH / 2];
#pragma unroll
        for (int h = 0; h < kH; h += 2) {
          const __nv_bfloat162 v = __floats2bfloat162_rn(pv[h], pv[h + 1]);
          bw[h >> 1] = *reinterpret_cast<const uint32_t*>(&v);
        }
        static_assert(L::kPRow == 32, "bf16 P rows: one query token");
        *reinterpret_cast<uint4*>(prow + ((16u * hg) ^ flip)) = make_uint4(bw[0], bw[1], bw[2], bw[3]);
      }
      if (nvalid < kTile) {
        // Tail tile: rows past the range may hold anything (stale tiles,
        // unused page slots); zero their V bytes so that 0 * V stays 0.
        const uint32_t s2 = g % L::kNumTiles;
        wait_or_flag(L::kMx ? smem_u32(&ms->deq[s2]) : smem_u32(&ms->full[s2]),
                     (g / L::kNumTiles) & 1u, p.err, kErrSoftmax, abort);
        if (!valid) {
          uint8_t* row = ring_gen + s2 * L::kTileBytes + (tq >> 3) * gs + (tq & 7) * 64;
          constexpr int kZc = L::kVChunks / kHG;       // chunks zeroed by each group
          for (int c = hg * kZc; c < (hg + 1) * kZc; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<uint4*>(row + c * cs)[i] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&ms->p_full[sb]));
    }
    // ------------------------------------------------------------ epilogue
    const uint32_t gl = g - 1;
    wait_or_flag(smem_u32(&ms->pv_done[gl & 1u]), (gl >> 1) & 1u, p.err, kErrSoftmax, abort);
    tc_fence_after();
    float lt[kH];
    reduce_heads<false, kH>(l, lt, ms->red[g & 1u], h0, qw, lane, bar);
    if (*abort) return;
    // fp8 V entered the UMMAs as raw e4m3: its per-tensor scale is applied here.
    const float vscale = (L::kKv8 && !L::kMx) ? __ldg(p.kv_scale) : 1.0f;
    float inv[kH];
#pragma unroll
    for (int h = 0; h < kH; ++h) inv[h] = vscale / lt[h];
    if constexpr (L::kQL > 1) {
      // a query token may see none of the item's tokens (l = 0): O = 0
#pragma unroll
      for (int h = 0; h < kH; ++h) inv[h] = lt[h] > 0.0f ? inv[h] : 0.0f;
    }
    const int slot = w.slot;
    // rows of this group's q rows in the partial slot or in out (request b's
    // rows are b * kRows .. : [query token][head])
    const int64_t row0 = (slot >= 0 ? static_cast<int64_t>(slot) : static_cast<int64_t>(w.b)) *
                             L::kRows + h0;
    auto store_block = [&](int c, float (&o)[kH]) {
      const int d = c * 128 + tq;
      if (slot >= 0) {
        float* po = p.part_o + row0 * kVDim + d;
#pragma unroll
        for (int h = 0; h < kH; ++h) po[h * kVDim] = o[h];
      } else {
        uint16_t* po = p.out + row0 * kVDim + d;
#pragma unroll
        for (int h = 0; h < kH; ++h) {
          const __nv_bfloat16 v = __float2bfloat16_rn(o[h]);
          po[h * kVDim] = *reinterpret_cast<const uint16_t*>(&v);
        }
      }
    };
    if constexpr (kH <= 8) {
      // O^T of this thread's dim in all four blocks: every TMEM load is
      // issued before one wait
      float oh[4][kH], ol[4][kH];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tmem_ld(tl + kColO + L::kOCols * c + h0, oh[c]);
        if constexpr (L::kKv8) tmem_ld(tl + kColO + L::kOCols * c + L::kRows + h0, ol[c]);
      }
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int h = 0; h < kH; ++h)
          oh[c][h] = L::kKv8 ? (oh[c][h] + ol[c][h] * (1.0f / kPLoScale)) * inv[h] : oh[c][h] * inv[h];
        store_block(c, oh[c]);
      }
    } else {
      // 16 rows per thread: one block at a time (registers)
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float oh[kH], ol[kH];
        tmem_ld(tl + kColO + L::kOCols * c + h0, oh);
        if constexpr (L::kKv8) tmem_ld(tl + kColO + L::kOCols * c + L::kRows + h0, ol);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < kH; ++h)
          oh[h] = L::kKv8 ? (oh[h] + ol[h] * (1.0f / kPLoScale)) * inv[h] : oh[h] * inv[h];
        store_block(c, oh);
      }
    }
    tc_fence_before();
    if (tq < kH) {
      float mh = 0.f, lh = 1.f;
#pragma unroll
      for (int h = 0; h < kH; ++h)
        if (h == tq) { mh = m[h]; lh = lt[h]; }
      float lse2 = mh + __log2f(lh) - kPOff;
      if constexpr (L::kQL > 1) lse2 = lh > 0.0f ? lse2 : -INFINITY;
      if (slot >= 0)
        p.part_lse[row0 + tq] = lse2;
      else if (p.lse != nullptr)
        p.lse[row0 + tq] = lse2 * kLn2;
    }
  }
}

// -------------------------------------------------------------------- kernel
template <int QM>
__global__ void __launch_bounds__(Layout<QM>::kThreads, 1) mla_stage1_kernel(const __grid_constant__ Stage1Params p) {
  using L = Layout<QM>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t ring = smem_u32(smem);
  Misc* ms = reinterpret_cast<Misc*>(smem + L::kMiscOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const CtaHead& head = p.heads[blockIdx.x];
  const int it0 = head.it0, it1 = head.it1;
  const WorkItem first = head.first;

  if (threadIdx.x == 0) {
    // The workspace must hold this plan's table: its stamp in the header and
    // in this CTA's head.  Otherwise (another plan's table was uploaded at
    // this address since) nothing is read from the table and nothing is
    // written; mla_decode_check reports it.
    const uint64_t hs = reinterpret_cast<const WsHeader*>(p.err)->stamp;
    ms->stale = (hs != p.stamp || head.stamp != p.stamp) ? 1 : 0;
    for (int i = 0; i < L::kNumTiles; ++i) {
      mbar_init(smem_u32(&ms->full[i]), p.gather ? 32 : 1);   // gather: one per producer lane
      mbar_init(smem_u32(&ms->empty[i]), L::kPvIssuers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&ms->s_full[i]), 2);        // both QK^T issuers
      mbar_init(smem_u32(&ms->s_empty[i]), 128 * L::kHeadGroups);
      mbar_init(smem_u32(&ms->p_full[i]), 128 * L::kHeadGroups);
      mbar_init(smem_u32(&ms->pv_done[i]), L::kPvIssuers);
      mbar_init(smem_u32(&ms->q_full[i]), 1);
      mbar_init(smem_u32(&ms->q_empty[i]), 2 + L::kHeadGroups);  // QK^T issuers + softmax groups
    }
    for (int i = 0; i < 4; ++i) mbar_init(smem_u32(&ms->drain[i]), 1);
    for (int i = 0; i < L::kNumTiles; ++i) {
      mbar_init(smem_u32(&ms->deq[i]), 128);
      mbar_init(smem_u32(&ms->deq_a[i]), 128);
      mbar_init(smem_u32(&ms->upper_free[i]), 1);
    }
    mbar_init(smem_u32(&ms->q_stage), 1);
    mbar_init(smem_u32(&ms->q_stage_free), 1);
    ms->abort_dq = 0;
    ms->abort_sm = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&p.tmap_kv);
  if (warp == 1) {
    tmem_alloc(smem_u32(&ms->tmem_base), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;

  if (ms->stale) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrStale);
  } else if (warp == 0) {
    run_producer<QM>(p, ms, ring, it0, it1, first, lane);
  } else if (warp == 1 || warp == 3) {
    run_qk<QM>(p, ms, ring, ring + L::kQOff, tmem, it0, it1, first, warp == 3 ? 1 : 0, lane);
  } else if (warp == 2 || (!L::kMx && warp == 13)) {
    run_pv<QM>(p, ms, ring, ring + L::kPOff, tmem, it0, it1, first, warp == 13 ? 1 : 0, lane);
  } else if (warp < 4 + 4 * L::kHeadGroups) {
    run_softmax<QM>(p, ms, smem, smem + L::kPOff, smem + L::kQOff, smem + L::kQStageOff, tmem, it0,
                    it1, first, threadIdx.x - 128);
  } else if constexpr (L::kMx) {
    run_dequant<QM>(p, ms, smem, smem + L::kQOff, smem + L::kQStageOff, it0, it1, first,
                    threadIdx.x - 384);
  } else {
    run_qprep<QM>(p, ms, smem + L::kQOff, smem + L::kQStageOff, it0, it1, first, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

int stage1_smem_bytes(int qmode) {
  switch (qmode) {
    case kQBf16KvBf16: return Layout<kQBf16KvBf16>::kSmemBytes;
    case kQFp8KvFp8: return Layout<kQFp8KvFp8>::kSmemBytes;
    case kQBf16KvFp8: return Layout<kQBf16KvFp8>::kSmemBytes;
    case kQFp8KvBf16: return Layout<kQFp8KvBf16>::kSmemBytes;
    case kQBf16KvMx: return Layout<kQBf16KvMx>::kSmemBytes;
    case kQFp8KvFp8x2: return Layout<kQFp8KvFp8x2>::kSmemBytes;
  }
  return -1;
}

template <int QM>
static cudaError_t launch_t(const Stage1Params& p, int num_ctas, cudaStream_t stream) {
  const int smem = Layout<QM>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(mla_stage1_kernel<QM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mla_stage1_kernel<QM><<<num_ctas, Layout<QM>::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_stage1(int qmode, const Stage1Params& p, int num_ctas, cudaStream_t stream) {
  switch (qmode) {
    case kQBf16KvBf16: return launch_t<kQBf16KvBf16>(p, num_ctas, stream);
    case kQFp8KvFp8: return launch_t<kQFp8KvFp8>(p, num_ctas, stream);
    case kQBf16KvFp8: return launch_t<kQBf16KvFp8>(p, num_ctas, stream);
    case kQFp8KvBf16: return launch_t<kQFp8KvBf16>(p, num_ctas, stream);
    case kQBf16KvMx: return launch_t<kQBf16KvMx>(p, num_ctas, stream);
    case kQFp8KvFp8x2: return launch_t<kQFp8KvFp8x2>(p, num_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mla
