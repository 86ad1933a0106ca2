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
//    S accumulator; warps 2 and 13 (MXFP4: 2 and 0) issue PV for O blocks
//    0-1 and 2-3.  Warp 0 is the TMA producer (bf16 / fp8); warps 4-11 do
//    the softmax and the epilogue in two groups of 8 heads (two-token mode:
//    one group per query token, 16 heads each; one thread per token / per
//    output dim, TMEM lane = thread) and convert the first item's q; warp
//    12 converts the q of later items; warp 14 prefetches each tile's rows
//    into L2 a slot hold ahead (page tables, and the one-slot bf16 ring),
//    so that the producer's boxes read from L2;
//  * MXFP4: warps 12-19 load the packed rows from global memory straight
//    into registers (any page size), dequantise them into the e4m3 tile slot
//    and prepare every item's q; the warpgroups then run with their own
//    register limits (setmaxnreg);
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
  static constexpr bool kKv8 = (QM == kQFp8KvFp8 || QM == kQBf16KvFp8 || kMx ||
                                QM == kQFp8KvFp8x2 || QM == kQBf16KvFp8x2);
  static constexpr int kQL =                                         // query tokens per request
      (QM == kQFp8KvFp8x2 || QM == kQBf16KvFp8x2) ? 2 : 1;
  static constexpr int kRows = kHeads * kQL;                        // q rows, token-major
  static constexpr bool kHiLo =                                      // q as two e4m3 terms
      (QM == kQBf16KvFp8 || kMx || QM == kQBf16KvFp8x2);
  static constexpr int kNq = kRows * (kHiLo ? 2 : 1);               // UMMA N of QK^T
  // Warps: producer (MXFP4: a PV issuer), 2 QK^T issuers, PV issuers, two
  // head groups of four softmax warps (kH q rows each), then either a q warp,
  // a PV issuer and an L2 prefetcher (15 warps) or, for MXFP4, 8 dequant
  // warps that also load the packed rows and prepare q (20 warps).
  static constexpr int kHeadGroups = 2;
  static constexpr int kH = kRows / kHeadGroups;                    // q rows per softmax thread
  static constexpr int kThreads = kMx ? 640 : 480;
  // MXFP4 register plan per warpgroup (setmaxnreg after the launch): the
  // producer and UMMA issuers need few, the softmax warps many
  static constexpr int kRegsLaunch = 96;
  static constexpr int kRegsIssue = 56, kRegsSoftmax = 104, kRegsDequant = 104;
  static constexpr int kRegsPlanned = 128 * kRegsIssue + 256 * kRegsSoftmax + 256 * kRegsDequant;
  static_assert(!kMx || (kThreads == 640 && kRegsPlanned <= kThreads * kRegsLaunch &&
                         kRegsIssue <= kRegsLaunch),
                "the warpgroups' register limits exceed the launch's pool");
  static constexpr int kPvIssuers = 2;
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
  // q staging buffer (raw q of the next item); MXFP4 and bf16 q in pairs
  // convert q from global memory into their one q buffer (so that two KV
  // tiles fit)
  static constexpr bool kQGlobal = kMx || QM == kQBf16KvFp8x2;
  static constexpr int kQStageBytes = kQGlobal ? 0 : kQSrcBytes;
  static constexpr int kQBufs = kQGlobal ? 1 : 2;
  static constexpr uint32_t kOCols = kRows * (kKv8 ? 2 : 1);       // TMEM columns per O block
  // TMEM: S^T at 0 (2 buffers x 2 K-halves x kSC columns), then O^T: four
  // 128-dim blocks of kOCols columns (fp8 KV: the q rows of p_hi, then of p_lo)
  static constexpr uint32_t kSC = kNq > 32 ? kNq : 32;              // columns per S K-half
  static constexpr uint32_t kColO = 4 * kSC;
  static constexpr uint32_t kTmemCols = kColO + 4 * kOCols <= 256 ? 256 : 512;
  static constexpr int kMiscBytes = 2560;
  static constexpr int kMaxSmem = 232448;
  static constexpr int kNumTiles =
      kMx ? 2
          : (kMaxSmem - 1024 - kQBufs * kQBytes - 2 * kPBytes - kMiscBytes - kQStageBytes) /
                kTileBytes;
  static constexpr int kQOff = kNumTiles * kTileBytes;
  static constexpr int kPOff = kQOff + kQBufs * kQBytes;
  static constexpr int kMiscOff = kPOff + 2 * kPBytes;
  static constexpr int kQStageOff = kMiscOff + kMiscBytes;        // raw q of the next item
  static constexpr int kSmemBytes = kQStageOff + kQStageBytes + 1024;
  static_assert(kNumTiles >= 1 && kNumTiles <= 4, "tile ring");
  static_assert(kSmemBytes <= kMaxSmem, "shared memory over budget");
  static_assert(kTileBytes % 1024 == 0 && kQBytes % 1024 == 0, "operand alignment");
  static_assert(kNq <= 64 && kTmemCols >= kColO + 4 * kOCols, "TMEM columns");
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
  uint64_t deq_a[4];                 // tile slot chunks 0-4 (dims 0-319) dequantised: the
                                     // first QK^T K-half (dims 0-287) may start
  uint64_t deq_b[4];                 // chunks 5-8 dequantised (the slot is complete)
  int32_t stale;                     // the workspace holds another plan's table
  uint32_t landed;                   // tiles the first QK^T issuer has seen land (bf16 / fp8)
  int16_t uexp[2][128];              // per-token power of two u_t = r_t - 127 of a slot
  uint2 e2m1_tab[16];                // e4m3 tables for 2^k, k = index - 14 (k <= -14: all 0)
};
static_assert(sizeof(Misc) <= 2560, "misc region");
static_assert(offsetof(Misc, red) % 16 == 0, "reduction scratch is read as float4");

// TMEM columns: S^T from 0 as 2 buffers x 2 K-halves (the two QK^T issuers
// each accumulate half of the 576 dims) x Layout::kSC columns, then O^T from
// Layout::kColO.
constexpr uint32_t kColS = 0;

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
    if (p.gather) {
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
    if (lane == 0) mbar_arrive_expect_tx(full, static_cast<uint32_t>(f.nbox) * box_bytes);
    ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->empty[s]), ph ^ 1u, p.err, kErrProducer));
    if (!ok) break;
    if (lane < f.nbox)
      tma_load_3d(ring + s * L::kTileBytes + lane * box_bytes, &p.tmap_kv, full, 0, row, 0, pol);
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
// L2 prefetcher (one warp): the rows of tile t are prefetched into L2 once
// tile t - kNumTiles has landed, i.e. about one slot hold before the
// producer's boxes for tile t go out into the slot that tile frees, so that
// those boxes read from L2.  Plain prefetch instructions, not bulk
// prefetches: the TMA unit spends about 60 cycles on each box of a tile
// already, and a bulk prefetch would add as many again.  It runs where the
// landing sits on the critical path: page tables (16 boxes per tile) and the
// one-slot bf16 ring.  Two cases were slower with it on GB300 and skip it:
// an identity table with two slots (one 128-row box per tile), and bf16 q in
// pairs (whose softmax warps read the next item's q from global memory).  A
// hint only: its waits give up quietly, the roles on the data path report a
// stalled tile.
template <int QM>
__device__ void run_prefetch(const Stage1Params& p, Misc* ms, int it0, int it1,
                             const WorkItem& first, int lane) {
  using L = Layout<QM>;
  if (QM == kQBf16KvFp8x2 || p.gather || (p.box_rows != 8 && L::kNumTiles > 1)) return;
  TileCursor c;
  c.init(p.items, it0, it1, first);
  BoxFetch f = box_fetch(p, c, lane);
  uint32_t t = 0;
  while (!c.done()) {
    TileCursor n = c;
    n.advance();
    const BoxFetch fn = box_fetch(p, n, lane);    // in flight during the wait
    // (the first kNumTiles tiles go out at once: a prefetch would only
    // compete with their boxes)
    if (t < static_cast<uint32_t>(L::kNumTiles)) {
      f = fn;
      c = n;
      ++t;
      continue;
    }
    {
      // Tile t - kNumTiles has landed once the first QK^T issuer has seen it
      // land.  A count, not the slot's mbarrier: this warp may fall two
      // phases behind a slot, and a parity wait would then wait for a phase
      // that never comes.
      const volatile uint32_t* landed = &ms->landed;
      const uint32_t need = t - L::kNumTiles + 1;
      if (*landed < need) {
        const uint64_t t0 = globaltimer_ns();
        while (*landed < need) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) return;
          __nanosleep(128);
        }
      }
    }
    // lane l: box l's rows (8-row groups), or a share of the one 128-row box
    int64_t r0 = 0, nrows = 0;
    if (p.box_rows == 8) {
      if (lane < f.nbox) { r0 = box_row(p, f, lane); nrows = 8; }
    } else if (f.nbox > 0) {
      r0 = __shfl_sync(0xffffffffu, box_row(p, f, lane), 0);
      nrows = kTile;
    }
    nrows = min(nrows, static_cast<int64_t>(p.pool_rows) - r0);   // inside the pool
    const uint8_t* a = p.kv + r0 * L::kRowBytes;
    const int lines = static_cast<int>(nrows * L::kRowBytes / 128);
    const int first_line = p.box_rows == 8 ? 0 : lane;
    const int step = p.box_rows == 8 ? 1 : 32;
    for (int i = first_line; i < lines; i += step) prefetch_l2_last(a + i * 128);
    f = fn;
    c = n;
    ++t;
  }
}

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
    const int qb = qc.k % L::kQBufs;
    if (q_ready != qc.k) {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->q_full[qb]), (qc.k / L::kQBufs) & 1,
                                             p.err, kErrMma)))
        break;
      q_ready = qc.k;
    }
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&ms->s_empty[sb]), ((t >> 1) & 1u) ^ 1u,
                                           p.err, kErrMma)))
      break;
    // the tile is ready once it landed (MXFP4: once the chunks holding this
    // K-half were dequantised: 0-4 for dims 0-287, all for dims 288-575)
    const uint32_t ready = !L::kMx ? smem_u32(&ms->full[s])
                           : half == 0 ? smem_u32(&ms->deq_a[s]) : smem_u32(&ms->deq_b[s]);
    if (!__all_sync(0xffffffffu, mbar_wait(ready, (t / L::kNumTiles) & 1u, p.err, kErrMma)))
      break;
    if (half == 0 && lane == 0) *reinterpret_cast<volatile uint32_t*>(&ms->landed) = t + 1;
    tc_fence_after();
    if (p.gather) fence_proxy_async_smem();   // rows copied by cp.async (generic proxy)
    const uint32_t tile = ring + s * L::kTileBytes;
    const uint32_t qaddr = qbase + qb * L::kQBytes;
    const uint32_t d = tmem + kColS + 2 * L::kSC * sb + L::kSC * half;
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
    if (qc.j == qc.ntile - 1) tc_commit(smem_u32(&ms->q_empty[qb]));
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
      const int c = kBlocks * half + i;
      const uint32_t d = tmem + L::kColO + L::kOCols * c;
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

// The same table computed instead of loaded, for k in [-5, 0]: there every
// product m 2^k of a nonzero magnitude is a normal e4m3 number, whose code
// is that of m (0x30, 0x38, 0x3C, 0x40, 0x44, 0x48, 0x4C for .5 .. 6) with
// k added to the exponent field (bits 3-6), so each nonzero byte moves by
// 8k.  Below k = -5 the smallest magnitudes turn subnormal: the shared
// table built by e2m1_e4m3_table() serves those blocks.
__device__ __forceinline__ void e2m1_e4m3_table_normal(int k, uint32_t& lo, uint32_t& hi) {
  lo = 0x3C383000u + static_cast<uint32_t>(k) * 0x08080800u;
  hi = 0x4C484440u + static_cast<uint32_t>(k) * 0x08080808u;
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
// The dequantising threads of token `tq` read that token's 18 e8m0 bytes
// from global memory themselves (no TMA box: the pages' scale rows are 18 bytes,
// which no tensor map can stride over).  The row is found as the producer
// finds it: through the page table, a page outside the pool replaced by page
// 0.  The loads of a tile are issued one tile ahead and its page-table entry
// two tiles ahead, so neither waits on the path.

// A light cursor over the same tiles as TileCursor, for looking ahead: only
// what locating a token's pool row needs (ntile == 0 once past the end).
struct TileAhead {
  int it, j, ntile, tok_begin, tok_end, page_base;
  __device__ __forceinline__ void from(const TileCursor& c) {
    it = c.it;
    j = c.j;
    ntile = c.ntile;
    tok_begin = c.w.tok_begin;
    tok_end = c.w.tok_end;
    page_base = c.w.page_base;
  }
  __device__ __forceinline__ void advance(const WorkItem* items, int it1) {
    if (ntile == 0 || ++j < ntile) return;
    j = 0;
    ntile = 0;
    if (++it < it1) {
      const WorkItem& w = items[it];
      tok_begin = w.tok_begin;
      tok_end = w.tok_end;
      page_base = w.page_base;
      ntile = (tok_end - tok_begin + kTile - 1) / kTile;
    }
  }
  __device__ __forceinline__ int t0() const { return tok_begin + j * kTile; }
  __device__ __forceinline__ int nvalid() const { return min(kTile, tok_end - t0()); }
};

// Raw page-table entry of token tq of a look-ahead tile (0 for the identity
// table or a token past the tile's end).
__device__ __forceinline__ int32_t scale_page(const Stage1Params& p, const TileAhead& c, int tq) {
  if (c.ntile == 0 || tq >= c.nvalid() || p.kv_indices == nullptr) return 0;
  return ld_nc_early(p.kv_indices + c.page_base + (c.t0() + tq) / p.page_size);
}

// Pool row of token tq of a look-ahead tile, or -1 past the tile's end.
// `page` is scale_page() of the same tile and token: a page outside the pool
// reads page 0 and is reported.
__device__ __forceinline__ int64_t pool_row(const Stage1Params& p, const TileAhead& c, int tq,
                                            int32_t page) {
  if (c.ntile == 0 || tq >= c.nvalid()) return -1;
  const int pos = c.t0() + tq;
  if (p.kv_indices == nullptr) {
    const int64_t row = static_cast<int64_t>(c.page_base) * p.page_size + pos;
    return row < p.pool_rows ? row : 0;   // (the host rejects such plans; never reached)
  }
  if (page < 0 || static_cast<int64_t>(page + 1) * p.page_size > p.pool_rows) {
    atomicOr(p.err, kErrBadPage);
    page = 0;
  }
  return static_cast<int64_t>(page) * p.page_size + pos % p.page_size;
}

// Issues the nine 1-byte loads of bytes hb, hb + 2, .. hb + 16 of scale row
// `row` (the blocks of one dequant half; zeros for row -1).
__device__ __forceinline__ void scale_load(const Stage1Params& p, int64_t row, int hb,
                                           uint32_t (&e)[9]) {
  if (row < 0) {
#pragma unroll
    for (int i = 0; i < 9; ++i) e[i] = 0;
    return;
  }
  const uint8_t* src = p.kv_e8m0 + row * p.sc_stride + hb;
#pragma unroll
  for (int i = 0; i < 9; ++i) e[i] = ld_nc_u8_early(src + 2 * i);
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

// Eight bf16 q values (vector `vid` of the [rows][576] q) -> their e4m3
// q_hi = rn(q / s_hi) and q_lo = rn(16 (q - q_hi s_hi) / s_hi) bytes, stored
// as rows h and rows + h of the K-major, 128-byte-swizzled q operand.
__device__ __forceinline__ void q_split_store(const uint4 v, int vid, float s_hi, float inv_hi,
                                              uint8_t* dst, int atom_bytes, int rows) {
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
  *reinterpret_cast<uint2*>(base + sw128(rows + h, x)) = make_uint2(lw[0], lw[1]);
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
  if constexpr (QM == kQBf16KvFp8 || QM == kQBf16KvMx || QM == kQBf16KvFp8x2) {
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
    for (int v = i; v < kV; v += n)
      q_split_store(src[v], v, s_hi, inv_hi, dst, L::kQAtomBytes, L::kRows);
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

// MXFP4: the eight dequant warps (256 threads, named barrier 3) prepare q of
// every item straight from global memory into the single q buffer.  All the
// request's bf16 values are held in registers while |q|max over the request
// is reduced, then split into two e4m3 terms (q_split_store).
template <int QM>
__device__ __forceinline__ void q_convert_mx(const Stage1Params& p, Misc* ms, int b, uint8_t* dst,
                                             int i, float& c_hi, float& c_lo) {
  using L = Layout<QM>;
  constexpr float kSmScale = 1.0f / 24.0f;                       // 1/sqrt(576)
  constexpr int kN = 256, kV = kHeads * kQkDim / 8;              // 1152 vectors of 8 bf16
  constexpr int kPer = (kV + kN - 1) / kN;
  const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.q) +
                                                    static_cast<int64_t>(b) * kHeads * kQkDim * 2);
  // two passes over the request's q (the second from L1/L2): |q|max, then the
  // split, so that no vector stays live across the reduction
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int v = i + kN * u;
    if (v >= kV) break;
    const uint4 x = __ldg(src + v);
    const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&x);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h2[e]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((i & 31) == 0) ms->qred[i >> 5] = amax;
  named_bar_sync(3, kN);
  amax = 0.f;
#pragma unroll
  for (int w = 0; w < kN / 32; ++w) amax = fmaxf(amax, ms->qred[w]);
  amax = fmaxf(amax, 1e-30f);
  const float s_hi = amax / 448.0f, inv_hi = 448.0f / amax;
#pragma unroll 1
  for (int u = 0; u < kPer; ++u) {
    const int v = i + kN * u;
    if (v < kV) q_split_store(__ldg(src + v), v, s_hi, inv_hi, dst, L::kQAtomBytes, L::kRows);
  }
  c_hi = s_hi * kSmScale * kLog2e;
  c_lo = c_hi * (1.0f / 16.0f);
}

// q of item k (request b) into the q buffer, once QK^T of item k-1 and its
// softmax released the buffer.  `failed` carries this thread's failed waits;
// the group's barrier ORs them, so that all 256 threads leave together
// (returns false) or carry on together.
template <int QM>
__device__ bool qprep_mx(const Stage1Params& p, Misc* ms, uint8_t* qgen, int b, int k, int d,
                         bool& failed) {
  if (k > 0 && !failed && !mbar_wait(smem_u32(&ms->q_empty[0]), (k - 1) & 1, p.err, kErrQPrep))
    failed = true;
  if (named_bar_any(3, 256, failed)) return false;
  float c_hi, c_lo;
  q_convert_mx<QM>(p, ms, b, qgen, d, c_hi, c_lo);
  fence_proxy_async_smem();
  named_bar_sync(3, 256);                           // every thread wrote its part; qred free
  if (d == 0) {
    ms->qscale[0][0] = c_hi;
    ms->qscale[0][1] = c_lo;
    mbar_arrive(smem_u32(&ms->q_full[0]));
  }
  return true;
}

// Chunks [j0, j1) of one dequant thread: block 2j + h of its token (packed
// in x[j], e8m0 byte in eb[j]) into e4m3 chunk j of its row at dst,
// pieces pc0 / pc1; zeros for a row past the tile's end.  As soon as block j
// is converted, x[j] is reloaded with the same block of the next tile's row
// (from `next`, unless null), so each load has one tile period to arrive.
// Returns whether anything was written (the caller then fences the writes
// for the UMMAs).
template <int kN>
__device__ __forceinline__ bool half_of_tile(bool ok, bool live, bool fast, uint4 (&x)[kN],
                                             const uint32_t (&eb)[kN], int r, const uint2* tab,
                                             uint8_t* dst, uint32_t pc0, uint32_t pc1, int j0,
                                             int j1, const uint8_t* next) {
  if (!ok) return false;
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    if (j < j0 || j >= j1) continue;
    uint4 o0 = make_uint4(0, 0, 0, 0), o1 = make_uint4(0, 0, 0, 0);
    if (live) {
      const int k = static_cast<int>(eb[j]) - r;
      uint32_t lo, hi;
      if (fast) {
        e2m1_e4m3_table_normal(k, lo, hi);
      } else {
        const uint2 tb = tab[max(k, -14) + 14];
        lo = tb.x;
        hi = tb.y;
      }
      const uint2 e0 = e2m1x8_to_e4m3(x[j].x, lo, hi), e1 = e2m1x8_to_e4m3(x[j].y, lo, hi);
      const uint2 e2 = e2m1x8_to_e4m3(x[j].z, lo, hi), e3 = e2m1x8_to_e4m3(x[j].w, lo, hi);
      o0 = make_uint4(e0.x, e0.y, e1.x, e1.y);
      o1 = make_uint4(e2.x, e2.y, e3.x, e3.y);
    }
    if (next != nullptr) x[j] = ld_nc_na_v4(next + 32 * j);
    *reinterpret_cast<uint4*>(dst + j * 512 + pc0) = o0;
    *reinterpret_cast<uint4*>(dst + j * 512 + pc1) = o1;
  }
  return true;
}

// Eight warps turn the packed MXFP4 rows of a tile into the e4m3 tile slot
// the UMMAs read.  Dequant warp wi owns rows 16 wi .. 16 wi + 15 of every
// tile: lane l works on row 16 wi + 4 (l >> 3) + (l & 3) and, with
// h = (l >> 2) & 1, on every other scale block of it (the even blocks 0, 2,
// .. 16 for h = 0, the odd ones for h = 1).  Block 2j + h is the h-th
// 32-byte half of e4m3 chunk j, so a thread's nine blocks go to the same two
// swizzled 16-byte pieces of chunks 0-8: every address is a fixed offset
// from the thread's row, and in each group of eight lanes (four rows, both
// halves) the swizzled e4m3 writes hit eight different bank groups.
//
// The packed blocks go from global memory straight into registers: block j
// of the next tile is loaded as soon as block j of this tile is converted,
// so every load has a tile period to arrive and nothing lands in shared
// memory first.  (An L2 prefetch of the rows two tiles ahead made the
// kernel slower.)  Chunks 0-4 (dims 0-319, which hold the first QK^T
// K-half) are published before chunks 5-8.
//
// With r_t the token's largest e8m0 exponent, block b becomes
// e2m1 * 2^(E_b - r_t): exact in e4m3 while E_b - r_t >= -8.  The remaining
// factor 2^(r_t - 127) of the token is left to the softmax (u_t in shared
// memory).  The e4m3 magnitudes of a block are computed for
// E_b - r_t >= -5 (every block of the token within five binades of its
// largest, the common case) and looked up otherwise.  Rows past the tile's
// end are written as zeros, so that 0 * V stays 0 in PV.
//
// The same threads prepare q: item 0's before the first tile, item k's
// right after dequantising item k's first tile (QK^T of item k waits for it).
template <int QM>
__device__ void run_dequant_mx(const Stage1Params& p, Misc* ms, uint8_t* ring_gen, uint8_t* qgen,
                               int it0, int it1, const WorkItem& first, int d) {
  using L = Layout<QM>;
  static_assert(L::kRowBytes * 8 == 4608 && L::kRawRowBytes == 288, "row layout");
  if (it0 >= it1) return;
  const int lane = d & 31, wi = d >> 5;
  const int row = 16 * wi + 4 * (lane >> 3) + (lane & 3), h = (lane >> 2) & 1;
  bool failed = false;                                 // a bounded wait of this thread gave up
  TileCursor c;                                        // this tile
  TileAhead a0, a1, a2;                                // it, the next, the one after
  c.init(p.items, it0, it1, first);
  a0.from(c);
  a1 = a0;
  a1.advance(p.items, it1);
  a2 = a1;
  a2.advance(p.items, it1);
  // the first tile's packed blocks and scale bytes
  uint4 x[9];
  uint32_t ec[9], en[9];                               // scale bytes: this tile, the next
  {
    const int64_t r0 = pool_row(p, a0, row, scale_page(p, a0, row));
    if (r0 >= 0) {
      const uint8_t* src = p.kv + r0 * L::kRawRowBytes + 16 * h;
#pragma unroll
      for (int j = 0; j < 9; ++j) x[j] = ld_nc_na_v4(src + 32 * j);
    }
    scale_load(p, r0, h, ec);
  }
  int32_t pg1 = scale_page(p, a1, row);                // raw page entry of this row, next tile
  if (d < 15) {
    uint32_t lo, hi;
    e2m1_e4m3_table(d - 14, lo, hi);
    ms->e2m1_tab[d] = make_uint2(lo, hi);
  }
  // (qprep_mx and every tile begin with a group barrier, so the tables are
  // visible before their first use)
  if (!qprep_mx<QM>(p, ms, qgen, first.b, 0, d, failed)) return;
  // this row in the e4m3 tile: 8-row group at 4608, 64-byte chunk j at
  // 512 j, row at 64; this thread's two 16-byte pieces under the 64-byte
  // swizzle
  const uint32_t row_off = (row >> 3) * 4608u + (row & 7) * 64u;
  const uint32_t swz = ((row & 7) >> 1) & 3u;
  const uint32_t pc0 = ((2u * h) ^ swz) << 4, pc1 = ((2u * h + 1u) ^ swz) << 4;
  // No group barrier per tile: once a bounded wait of a thread gave up
  // (`failed`), that thread skips every later wait and all work, so it runs
  // through its remaining tiles at once; the group decides to leave together
  // at the barrier of the next q preparation (or the loop ends).
  while (!c.done()) {
    const uint32_t tt = c.t, s = tt % L::kNumTiles;
    const int nvalid = c.nvalid();
    // this tile's scale bytes: r = max over all 18 (this thread's nine and
    // those of lane ^ 4, the other half of the token), and the smallest of
    // this thread's nine
    int r = 0, emin = 255;
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      r = max(r, static_cast<int>(ec[j]));
      emin = min(emin, static_cast<int>(ec[j]));
    }
    r = max(r, __shfl_xor_sync(0xffffffffu, r, 4));
    // the next tile's row: its scale bytes now, its packed blocks while this
    // tile's are converted
    const int64_t rn = pool_row(p, a1, row, pg1);
    scale_load(p, rn, h, en);
    const uint8_t* next = rn >= 0 ? p.kv + rn * L::kRawRowBytes + 16 * h : nullptr;
    pg1 = scale_page(p, a2, row);
    const bool live = row < nvalid;
    const bool fast = emin - r >= -5;                  // all nine blocks on the computed path
    // the slot is overwritten whole: PV of its previous tile must be done
    const bool ok = !failed && mbar_wait(smem_u32(&ms->empty[s]),
                                         ((tt / L::kNumTiles) & 1u) ^ 1u, p.err, kErrDequant);
    if (!ok) failed = true;
    uint8_t* dst = ring_gen + s * L::kTileBytes + row_off;
    // the token's factor for the softmax (read once S of the tile exists)
    if (h == 0 && ok) ms->uexp[s][row] = static_cast<int16_t>(live ? r - 127 : 0);
    if (half_of_tile(ok, live, fast, x, ec, r, ms->e2m1_tab, dst, pc0, pc1, 0, 5, next)) {
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(smem_u32(&ms->deq_a[s]));   // chunks 0-4
    if (half_of_tile(ok, live, fast, x, ec, r, ms->e2m1_tab, dst, pc0, pc1, 5, 9, next)) {
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(smem_u32(&ms->deq_b[s]));   // chunks 5-8
#pragma unroll
    for (int j = 0; j < 9; ++j) ec[j] = en[j];
    const bool item_start = c.j == 0;
    const int k = c.k, b = c.w.b;
    c.advance();
    a1 = a2;
    a2.advance(p.items, it1);
    if (item_start && k > 0 && !qprep_mx<QM>(p, ms, qgen, b, k, d, failed)) return;
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
  // bf16 q in pairs: the softmax warps convert every item's q from global
  // memory into the one q buffer (run_softmax); nothing to do here
  if constexpr (L::kQGlobal) return;
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
      // (bf16 q in pairs: straight from global memory, no staging buffer)
      constexpr int kN = 128 * kHG;
      const uint8_t* src = stage;
      if constexpr (L::kQGlobal) {
        src = static_cast<const uint8_t*>(p.q) + static_cast<int64_t>(first.b) * L::kQSrcBytes;
      } else {
        wait_or_flag(smem_u32(&ms->q_stage), 0, p.err, kErrSoftmax, abort);
      }
      named_bar_sync(6, kN);
      if (*abort) return;
      float c_hi, c_lo;
      q_convert<QM>(p, ms, src, qgen, tid, kN, 6, c_hi, c_lo);
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
    const uint32_t qb = k % L::kQBufs;
    wait_or_flag(smem_u32(&ms->q_full[qb]), (k / L::kQBufs) & 1, p.err, kErrSoftmax, abort);
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
        // S^T columns of buffer sb: two K-halves of kSC columns; q split in two
        // terms puts the rows of q_hi first, then those of q_lo
        const uint32_t sc = tl + kColS + 2 * L::kSC * sb + h0;
        float a0[kH], a1[kH];
        tmem_ld(sc, a0);
        tmem_ld(sc + L::kSC, a1);
        if constexpr (L::kHiLo) {
          float b0[kH], b1[kH];
          tmem_ld(sc + L::kRows, b0);
          tmem_ld(sc + L::kSC + L::kRows, b1);
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
        const int u = ms->uexp[g % L::kNumTiles][tq];
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
            const uint32_t col = L::kColO + L::kOCols * c + L::kRows * part + h0;
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
      if (!L::kMx && nvalid < kTile) {
        // Tail tile: rows past the range may hold anything (stale tiles,
        // unused page slots); zero their V bytes so that 0 * V stays 0.
        // (The MXFP4 dequantisation writes those rows as zeros itself.)
        const uint32_t s2 = g % L::kNumTiles;
        wait_or_flag(smem_u32(&ms->full[s2]), (g / L::kNumTiles) & 1u, p.err, kErrSoftmax, abort);
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
    if constexpr (L::kQGlobal && !L::kMx) {
      // bf16 q in pairs (one q buffer): QK^T of this item's last tile is
      // done, so its q buffer is free; convert the next item's q into it
      // before the epilogue, with all softmax threads
      if (it + 1 < it1) {
        constexpr int kN = 128 * kHG;
        wait_or_flag(smem_u32(&ms->q_empty[0]), static_cast<uint32_t>(k) & 1u, p.err,
                     kErrSoftmax, abort);
        const uint8_t* src =
            static_cast<const uint8_t*>(p.q) + static_cast<int64_t>(p.items[it + 1].b) * L::kQSrcBytes;
        named_bar_sync(6, kN);
        if (*abort) return;
        float c_hi2, c_lo2;
        q_convert<QM>(p, ms, src, qgen, tid, kN, 6, c_hi2, c_lo2);
        fence_proxy_async_smem();
        named_bar_sync(6, kN);
        if (tid == 0) {
          ms->qscale[0][0] = c_hi2;
          ms->qscale[0][1] = c_lo2;
          mbar_arrive(smem_u32(&ms->q_full[0]));
        }
      }
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
    // cluster merge: the CTA's partial stays in its own shared memory (its
    // tile ring, idle once the item's last PV is done) as [row][512] fp32
    // plus the rows' log2 LSE; the cluster's CTAs read it after a barrier.
    // (Another CTA's ring may still be in use: nothing is written there.)
    const bool to_cluster = p.cluster > 0 && slot >= 0;
    float* xo = reinterpret_cast<float*>(ring_gen);
    // rows of this group's q rows in the partial slot or in out (request b's
    // rows are b * kRows .. : [query token][head])
    const int64_t row0 = (slot >= 0 ? static_cast<int64_t>(slot) : static_cast<int64_t>(w.b)) *
                             L::kRows + h0;
    auto store_block = [&](int c, float (&o)[kH]) {
      const int d = c * 128 + tq;
      if (to_cluster) {
#pragma unroll
        for (int h = 0; h < kH; ++h) xo[(h0 + h) * kVDim + d] = o[h];
      } else if (slot >= 0) {
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
        tmem_ld(tl + L::kColO + L::kOCols * c + h0, oh[c]);
        if constexpr (L::kKv8) tmem_ld(tl + L::kColO + L::kOCols * c + L::kRows + h0, ol[c]);
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
        tmem_ld(tl + L::kColO + L::kOCols * c + h0, oh);
        if constexpr (L::kKv8) tmem_ld(tl + L::kColO + L::kOCols * c + L::kRows + h0, ol);
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
      if (to_cluster)
        xo[L::kRows * kVDim + h0 + tq] = lse2;
      else if (slot >= 0)
        p.part_lse[row0 + tq] = lse2;
      else if (p.lse != nullptr)
        p.lse[row0 + tq] = lse2 * kLn2;
    }
  }
}

// ------------------------------------------------------------ cluster merge
// The CTAs of a cluster hold the cs partials of one request (request b) in
// their shared memory: [16 rows][512] fp32 and the rows' log2 LSE after it
// (the epilogue above).  CTA `rank` merges dims [rank 512/cs, (rank+1) 512/cs)
// of every row, reading all cs partials through distributed shared memory:
// M = max_s lse_s, w_s = 2^(lse_s - M), o = sum_s w_s o_s / sum_s w_s, as the
// stage-2 merge does (the merge of the split-KV kernels of submission 668813,
// _mla_mxfp4_stage2_log2).  Rank 0 writes the rows' natural-log LSE.
template <int QM>
__device__ void cluster_merge(const Stage1Params& p, const uint8_t* smem, int b) {
  using L = Layout<QM>;
  static_assert(L::kRows == kHeads, "cluster merge: one query token per request");
  const int cs = p.cluster;
  const uint32_t rank = cluster_ctarank();
  const int span = kVDim / cs, vec = span / 4;                 // dims / float4s of this CTA
  const uint32_t xo = smem_u32(smem), xl = xo + kHeads * kVDim * 4;
  for (int v = threadIdx.x; v < kHeads * vec; v += L::kThreads) {
    const int h = v / vec, d = static_cast<int>(rank) * span + 4 * (v % vec);
    // every load of the cs partials is issued before the first use
    float ls[8];
    float4 o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j < cs) {
        ls[j] = ld_dsmem_f32(dsmem_addr(xl + 4u * h, j));
        o[j] = ld_dsmem_v4(dsmem_addr(xo + 4u * (h * kVDim + d), j));
      } else {
        ls[j] = -INFINITY;
        o[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int j = 0; j < 8; ++j) M = fmaxf(M, ls[j]);
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    float W = 0.0f;
    if (M != -INFINITY) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float w = ex2(ls[j] - M);          // 0 for an empty or absent partial
        W += w;
        acc.x += w > 0.0f ? w * o[j].x : 0.0f;
        acc.y += w > 0.0f ? w * o[j].y : 0.0f;
        acc.z += w > 0.0f ? w * o[j].z : 0.0f;
        acc.w += w > 0.0f ? w * o[j].w : 0.0f;
      }
    }
    const float inv = W > 0.0f ? 1.0f / W : 0.0f;
    const __nv_bfloat162 x = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    const __nv_bfloat162 y = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 o2;
    o2.x = *reinterpret_cast<const uint32_t*>(&x);
    o2.y = *reinterpret_cast<const uint32_t*>(&y);
    *reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(b) * kHeads + h) * kVDim + d) = o2;
    if (d == 0 && p.lse != nullptr)
      p.lse[static_cast<int64_t>(b) * kHeads + h] = W > 0.0f ? (M + __log2f(W)) * kLn2 : -INFINITY;
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
  // bf16 / fp8: the CTA's item range and first item are loaded at once, so
  // that the loads overlap the set-up below (MXFP4 reads them after its
  // register limits are set, see below)
  int it0 = 0, it1 = 0;
  WorkItem first{};
  if constexpr (!L::kMx) {
    it0 = head.it0;
    it1 = head.it1;
    first = head.first;
  }

  if (threadIdx.x == 0) {
    // The workspace must hold this plan's table: its stamp in the header and
    // in this CTA's head.  Otherwise (another plan's table was uploaded at
    // this address since) nothing is read from the table and nothing is
    // written; mla_decode_check reports it.  The two stamps are loaded first
    // and compared after the barrier set-up, which hides their latency.
    const uint64_t hs = ld_nc_early_u64(&reinterpret_cast<const WsHeader*>(p.err)->stamp);
    const uint64_t cs = ld_nc_early_u64(&head.stamp);
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
    if constexpr (L::kMx) {
      for (int i = 0; i < L::kNumTiles; ++i) {
        mbar_init(smem_u32(&ms->deq_a[i]), 8);       // one arrival per dequant warp
        mbar_init(smem_u32(&ms->deq_b[i]), 8);
      }
    }
    mbar_init(smem_u32(&ms->q_stage), 1);
    mbar_init(smem_u32(&ms->q_stage_free), 1);
    ms->abort_sm = 0;
    ms->landed = 0;
    fence_mbar_init();
    ms->stale = (hs != p.stamp || cs != p.stamp) ? 1 : 0;
  }
  if (!L::kMx && warp == 0 && lane == 0) prefetch_tensormap(&p.tmap_kv);
  if (warp == 1) {
    tmem_alloc(smem_u32(&ms->tmem_base), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;

  // MXFP4: the CTA's item range and first item are read by every role after
  // its warpgroup set its register limit, so that nothing is live across it.
  auto head_items = [&](int& i0, int& i1, WorkItem& f) {
    i0 = head.it0;
    i1 = head.it1;
    f = head.first;
  };
  if (ms->stale) {
    if (threadIdx.x == 0) atomicOr(p.err, kErrStale);
  } else if constexpr (L::kMx) {
    // One branch per warpgroup, each opening with its register limit (every
    // warp of the group executes the same setmaxnreg), so that the limit
    // governs the role code it dominates: 0 = UMMA issuers, 1-2 = softmax,
    // 3-4 = dequantisation (with the loads of the packed rows).
    const int wg = warp >> 2;
    if (wg == 0) {
      regs_lower<L::kRegsIssue>();
      head_items(it0, it1, first);
      if (warp == 0 || warp == 2)
        run_pv<QM>(p, ms, ring, ring + L::kPOff, tmem, it0, it1, first, warp == 0 ? 1 : 0, lane);
      else
        run_qk<QM>(p, ms, ring, ring + L::kQOff, tmem, it0, it1, first, warp == 3 ? 1 : 0, lane);
    } else if (wg <= 2) {
      if constexpr (L::kRegsSoftmax < L::kRegsLaunch) regs_lower<L::kRegsSoftmax>();
      if constexpr (L::kRegsSoftmax > L::kRegsLaunch) regs_raise<L::kRegsSoftmax>();
      head_items(it0, it1, first);
      run_softmax<QM>(p, ms, smem, smem + L::kPOff, smem + L::kQOff, smem + L::kQStageOff, tmem,
                      it0, it1, first, threadIdx.x - 128);
    } else {
      if constexpr (L::kRegsDequant < L::kRegsLaunch) regs_lower<L::kRegsDequant>();
      if constexpr (L::kRegsDequant > L::kRegsLaunch) regs_raise<L::kRegsDequant>();
      head_items(it0, it1, first);
      run_dequant_mx<QM>(p, ms, smem, smem + L::kQOff, it0, it1, first,
                         threadIdx.x - 384);
    }
  } else {
    if (warp == 0) {
      run_producer<QM>(p, ms, ring, it0, it1, first, lane);
    } else if (warp == 1 || warp == 3) {
      run_qk<QM>(p, ms, ring, ring + L::kQOff, tmem, it0, it1, first, warp == 3 ? 1 : 0, lane);
    } else if (warp == 2 || warp == 13) {
      run_pv<QM>(p, ms, ring, ring + L::kPOff, tmem, it0, it1, first, warp == 13 ? 1 : 0, lane);
    } else if (warp < 4 + 4 * L::kHeadGroups) {
      run_softmax<QM>(p, ms, smem, smem + L::kPOff, smem + L::kQOff, smem + L::kQStageOff, tmem,
                      it0, it1, first, threadIdx.x - 128);
    } else if (warp == 12) {
      run_qprep<QM>(p, ms, smem + L::kQOff, smem + L::kQStageOff, it0, it1, first, lane);
    } else {
      run_prefetch<QM>(p, ms, it0, it1, first, lane);
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (!L::kMx && L::kRows == kHeads) {
    // cluster merge: every thread of every CTA of the cluster reaches both
    // barriers (each role's loop ends, its waits being bounded).  The first
    // publishes the partials; the second keeps each CTA's partial alive until
    // the others have read it (their loads have returned: the merge used the
    // values), and needs no release ordering of the merge's global stores
    if (p.cluster > 0) {
      cluster_sync();
      // (the CTA head is read again here, so that nothing stays live
      // across the roles for the merge)
      if (!ms->stale && head.it0 < head.it1) cluster_merge<QM>(p, smem, head.first.b);
      cluster_sync_relaxed();
    }
  }
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
    case kQBf16KvFp8x2: return Layout<kQBf16KvFp8x2>::kSmemBytes;
  }
  return -1;
}

template <int QM>
static cudaError_t launch_t(const Stage1Params& p, int num_ctas, cudaStream_t stream) {
  using L = Layout<QM>;
  const int smem = L::kSmemBytes;
  if constexpr (L::kMx) {
    // the warpgroups' register limits must fit the pool the launch provides
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, mla_stage1_kernel<QM>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs * L::kThreads < L::kRegsPlanned) return cudaErrorInvalidConfiguration;
  }
  cudaError_t e = cudaFuncSetAttribute(mla_stage1_kernel<QM>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.cluster > 0) {
    if (L::kMx || L::kRows != kHeads || num_ctas % p.cluster != 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas);
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(p.cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mla_stage1_kernel<QM>, p);
  }
  mla_stage1_kernel<QM><<<num_ctas, Layout<QM>::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

template <int QM>
static bool cluster_fits_t(int cs) {
  using L = Layout<QM>;
  if (L::kMx || L::kRows != kHeads) return false;
  if (cudaFuncSetAttribute(mla_stage1_kernel<QM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::kSmemBytes) != cudaSuccess)
    return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cs);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_stage1_kernel<QM>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return n > 0;
}

bool stage1_cluster_fits(int qmode, int cs) {
  switch (qmode) {
    case kQBf16KvBf16: return cluster_fits_t<kQBf16KvBf16>(cs);
    case kQFp8KvFp8: return cluster_fits_t<kQFp8KvFp8>(cs);
    case kQBf16KvFp8: return cluster_fits_t<kQBf16KvFp8>(cs);
    case kQFp8KvBf16: return cluster_fits_t<kQFp8KvBf16>(cs);
  }
  return false;
}

cudaError_t launch_stage1(int qmode, const Stage1Params& p, int num_ctas, cudaStream_t stream) {
  switch (qmode) {
    case kQBf16KvBf16: return launch_t<kQBf16KvBf16>(p, num_ctas, stream);
    case kQFp8KvFp8: return launch_t<kQFp8KvFp8>(p, num_ctas, stream);
    case kQBf16KvFp8: return launch_t<kQBf16KvFp8>(p, num_ctas, stream);
    case kQFp8KvBf16: return launch_t<kQFp8KvBf16>(p, num_ctas, stream);
    case kQBf16KvMx: return launch_t<kQBf16KvMx>(p, num_ctas, stream);
    case kQFp8KvFp8x2: return launch_t<kQFp8KvFp8x2>(p, num_ctas, stream);
    case kQBf16KvFp8x2: return launch_t<kQBf16KvFp8x2>(p, num_ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace mla
