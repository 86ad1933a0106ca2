// stage2.cu -- log-sum-exp merge of split partials (stage 2).
//
// The merge algebra of the log2-domain stage-2 kernel of kernelindex.com,
// amd-mixed-mla submission 668813 (and the natural-log reduce kernels of
// submissions 695854 and 600081): for one (request, head) with partials
// (o_s, lse_s), M = max_s lse_s, w_s = 2^(lse_s - M),
// out = sum_s w_s o_s / sum_s w_s (cast to bf16), lse = (M + log2 sum w) ln 2.
// Partials with lse = -inf carry no weight; a request with no partials is
// empty and gets out = 0, lse = -inf.
//
// One warp per (request, output row: head, or query token x head); a lane
// owns 16 of the 512 dims as four
// float4 columns, so every partial row is read as coalesced 512-byte lines.
// Up to four partials are loaded together with their lse values, so that a
// request split in at most four takes one round trip to memory.

#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace mla {

// Whether the workspace holds this plan's table.  Lane 0 reads the header
// stamp and the warp takes its answer, so that the whole warp leaves or stays.
__device__ __forceinline__ bool table_is_ours(const Stage2Params& p, int lane) {
  uint64_t hs = 0;
  if (lane == 0) hs = reinterpret_cast<const WsHeader*>(p.err)->stamp;
  hs = __shfl_sync(0xffffffffu, hs, 0);
  if (hs == p.stamp) return true;
  if (lane == 0) atomicOr(p.err, kErrStale);
  return false;
}

__global__ void __launch_bounds__(256) mla_stage2_kernel(const Stage2Params p) {
  const int gw = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const int job = gw / p.rows, h = gw % p.rows;   // h: output row of the request
  if (job >= p.num_jobs) return;
  // The job table is plan data (not written by stage 1): read it first,
  // together with the stamp of the table the workspace holds.  A table of
  // another plan is not used: nothing is written (mla_decode_check reports it).
  const MergeJob J = p.jobs[job];
  if (!table_is_ours(p, lane)) return;
  uint16_t* out = p.out + (static_cast<int64_t>(J.b) * p.rows + h) * kVDim;
  // Launched as a programmatic dependent of stage 1: wait here until stage 1
  // has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
  float M = -INFINITY, wsum = 0.0f;
  // Adds partials [s0, s0 + n) (n <= 4) with weights 2^(lse - M); a partial
  // whose weight is 0 adds exactly nothing (a select, not a branch, so that
  // no load waits on the weight).
  auto add = [&](int s0, int n, const float (&ls)[4], const float4 (&v)[4][4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float w = (u < n) ? ex2(ls[u] - M) : 0.0f;
      wsum += w;
      const bool live = w > 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[4 * i + 0] += live ? w * v[u][i].x : 0.0f;
        acc[4 * i + 1] += live ? w * v[u][i].y : 0.0f;
        acc[4 * i + 2] += live ? w * v[u][i].z : 0.0f;
        acc[4 * i + 3] += live ? w * v[u][i].w : 0.0f;
      }
    }
  };
  // Loads of up to four partials (lse and this lane's 16 dims) in flight together.
  auto load = [&](int s0, int n, float (&ls)[4], float4 (&v)[4][4]) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int64_t row = static_cast<int64_t>(J.first + s0 + (u < n ? u : 0)) * p.rows + h;
      ls[u] = p.part_lse[row];
      const float4* src = reinterpret_cast<const float4*>(p.part_o + row * kVDim);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[u][i] = src[lane + 32 * i];
    }
  };
  if (J.count == 0) {
    // empty request: no partial to read (out = 0, lse = -inf below)
  } else if (J.count <= 4) {
    // the common case: one round trip for every lse and every row
    float ls[4];
    float4 v[4][4];
    load(0, J.count, ls, v);
#pragma unroll
    for (int u = 0; u < 4; ++u) M = u < J.count ? fmaxf(M, ls[u]) : M;
    if (M != -INFINITY) add(0, J.count, ls, v);
  } else {
    for (int s = lane; s < J.count; s += 32)
      M = fmaxf(M, p.part_lse[static_cast<int64_t>(J.first + s) * p.rows + h]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (M != -INFINITY) {
      for (int s = 0; s < J.count; s += 4) {
        float ls[4];
        float4 v[4][4];
        const int n = min(4, J.count - s);
        load(s, n, ls, v);
        add(s, n, ls, v);
      }
    }
  }
  const float inv = wsum > 0.0f ? 1.0f / wsum : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(acc[4 * i + 0] * inv, acc[4 * i + 1] * inv);
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
    uint2 v;
    v.x = *reinterpret_cast<const uint32_t*>(&a);
    v.y = *reinterpret_cast<const uint32_t*>(&b);
    reinterpret_cast<uint2*>(out)[lane + 32 * i] = v;
  }
  if (lane == 0 && p.lse != nullptr)
    p.lse[static_cast<int64_t>(J.b) * p.rows + h] =
        wsum > 0.0f ? (M + __log2f(wsum)) * kLn2 : -INFINITY;
}

// Wide merge, for plans where a request has many partials (one long request
// spread over every SM): one CTA of 8 warps per (request, output row, quarter
// of the 512 dims), so that a lane owns one float4 of every partial row and a
// warp keeps 16 partials in flight per round trip to memory.  The 256
// threads find M = max_s lse_s together; warp w adds partials w, w + 8, ...
// with weights 2^(lse_s - M); the eight partial sums meet in shared memory.
constexpr int kWideSplit = 4;                 // CTAs per output row (128 dims each)
constexpr int kWideBatch = 16;                // partials per warp per round trip

__global__ void __launch_bounds__(256) mla_stage2_wide_kernel(const Stage2Params p) {
  __shared__ float red_m[8], red_w[8];
  __shared__ float4 red_acc[8][32];
  __shared__ int ours;
  const int quarter = blockIdx.x % kWideSplit, rowid = blockIdx.x / kWideSplit;
  const int job = rowid / p.rows, h = rowid % p.rows;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (job >= p.num_jobs) return;
  const MergeJob J = p.jobs[job];
  if (warp == 0) {
    const bool ok = table_is_ours(p, lane);
    if (lane == 0) ours = ok ? 1 : 0;
  }
  __syncthreads();
  if (!ours) return;                      // the whole CTA leaves together
  const int col = quarter * 32 + lane;        // this lane's float4 column (dims 4 col ..)
  uint16_t* out = p.out + (static_cast<int64_t>(J.b) * p.rows + h) * kVDim;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float M = -INFINITY;
  for (int s = tid; s < J.count; s += 256)
    M = fmaxf(M, p.part_lse[static_cast<int64_t>(J.first + s) * p.rows + h]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) red_m[warp] = M;
  __syncthreads();
  M = red_m[0];
#pragma unroll
  for (int w = 1; w < 8; ++w) M = fmaxf(M, red_m[w]);
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float wsum = 0.0f;
  if (M != -INFINITY) {
    for (int s0 = warp; s0 < J.count; s0 += 8 * kWideBatch) {
      float ls[kWideBatch];
      float4 v[kWideBatch];
#pragma unroll
      for (int u = 0; u < kWideBatch; ++u) {
        const int s = s0 + 8 * u;
        const int64_t row = static_cast<int64_t>(J.first + (s < J.count ? s : s0)) * p.rows + h;
        ls[u] = s < J.count ? p.part_lse[row] : -INFINITY;
        v[u] = reinterpret_cast<const float4*>(p.part_o + row * kVDim)[col];
      }
#pragma unroll
      for (int u = 0; u < kWideBatch; ++u) {
        const float w = ex2(ls[u] - M);         // 0 for a missing or empty partial
        wsum += w;
        const bool live = w > 0.0f;
        acc.x += live ? w * v[u].x : 0.0f;
        acc.y += live ? w * v[u].y : 0.0f;
        acc.z += live ? w * v[u].z : 0.0f;
        acc.w += live ? w * v[u].w : 0.0f;
      }
    }
  }
  if (lane == 0) red_w[warp] = wsum;           // every lane added the same weights
  red_acc[warp][lane] = acc;
  __syncthreads();
  if (tid < 32) {
    float4 a = red_acc[0][tid];
    float W = red_w[0];
#pragma unroll
    for (int w = 1; w < 8; ++w) {
      const float4 b = red_acc[w][tid];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
      W += red_w[w];
    }
    const float inv = W > 0.0f ? 1.0f / W : 0.0f;
    const __nv_bfloat162 x = __floats2bfloat162_rn(a.x * inv, a.y * inv);
    const __nv_bfloat162 y = __floats2bfloat162_rn(a.z * inv, a.w * inv);
    uint2 o2;
    o2.x = *reinterpret_cast<const uint32_t*>(&x);
    o2.y = *reinterpret_cast<const uint32_t*>(&y);
    reinterpret_cast<uint2*>(out)[quarter * 32 + tid] = o2;
    if (quarter == 0 && tid == 0 && p.lse != nullptr)
      p.lse[static_cast<int64_t>(J.b) * p.rows + h] = W > 0.0f ? (M + __log2f(W)) * kLn2 : -INFINITY;
  }
}

cudaError_t launch_stage2(const Stage2Params& p, cudaStream_t stream) {
  if (p.num_jobs <= 0) return cudaSuccess;
  const int warps = p.num_jobs * p.rows;
  const bool wide = p.wide != 0;
  // Programmatic dependent launch: the merge grid is scheduled while stage 1
  // drains, instead of after a full launch gap.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(wide ? warps * kWideSplit : (warps + 7) / 8);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return wide ? cudaLaunchKernelEx(&cfg, mla_stage2_wide_kernel, p)
              : cudaLaunchKernelEx(&cfg, mla_stage2_kernel, p);
}

}  // namespace mla
