// noalloc.cu -- mla_decode_run_noalloc: the decode call for callers that
// cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc for the workspace: code that
// runs inside a framework whose allocator they must not bypass, plug-ins and
// C clients loaded into a process that owns all device memory, or code paths
// that must not allocate at all once started.  For them the library carries
// its own workspace: a fixed array in device global memory that every GPU
// which loads the library holds until the process exits.  The caller still
// passes the inputs and the outputs.
//
// This entry point changes nothing in the regular path: it resolves the
// array's device address and hands it to mla_decode_run as the workspace.

#include <cuda_runtime.h>

#include <mutex>

#include "mla_decode.h"
#include "plan.h"

namespace mla {
namespace {

// kStaticWorkspaceBytes (16 MiB), the largest workspace a plan may need to
// use this entry point, covers the work table and split partials of balanced
// plans for batches of a few hundred requests (bs=256 x 8192 tokens needs
// about 9.5 MB).

// The workspace.  In host code `g_static_workspace` names a host-side stand-in,
// not the device array: only the address from cudaGetSymbolAddress below may
// be handed to a kernel.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_device_ptr[kMaxDevices] = {};

}  // namespace

// Device address of the array on the current device; looked up once per
// device (with that device current) and cached.
mla_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_device_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || ptr == nullptr)
      return MLA_ERR_CUDA;
    g_device_ptr[dev] = ptr;
  }
  *out = g_device_ptr[dev];
  return MLA_OK;
}

}  // namespace mla

extern "C" mla_status mla_decode_run_noalloc(mla_plan* plan, const void* q, const float* q_scale,
                                             const void* kv, const float* kv_scale,
                                             const uint8_t* kv_e8m0, int64_t kv_e8m0_row_stride,
                                             int64_t kv_pool_rows, const int32_t* kv_indices,
                                             void* out, float* lse, mla_stream_t stream) {
  if (plan == nullptr) return MLA_ERR_INVALID_ARG;
  if (plan->ws_bytes > mla::kStaticWorkspaceBytes) return MLA_ERR_WORKSPACE;
  void* ws = nullptr;
  const mla_status st = mla::static_workspace(&ws);
  if (st != MLA_OK) return st;
  // Every call shares the array and it keeps what the last call left there:
  // copy this plan's work table in again (that also zeroes the error word),
  // whatever plan used the array before.
  plan->uploaded_ws = nullptr;
  return mla_decode_run(plan, q, q_scale, kv, kv_scale, kv_e8m0, kv_e8m0_row_stride, kv_pool_rows,
                        kv_indices, ws, mla::kStaticWorkspaceBytes, out, lse, stream);
}
