// selftest.cu -- exercises the bounded-wait path of the pipeline on the GPU.
//
// One warp waits on an mbarrier that nothing arrives on, with the helper
// every pipeline wait of the decode kernel uses (mbar_wait_for), but with a
// short limit.  The wait gives up, records its error bit in the caller's
// device error word and the kernel returns: the context stays usable, and
// mla_decode_check reports the timeout exactly as for a decode call.

#include "mla_decode.h"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace mla {

__global__ void __launch_bounds__(32, 1) bounded_wait_kernel(int32_t* err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  // phase 0 never completes: no thread arrives
  mbar_wait_for(smem_u32(&bar), 0, err, kErrProducer, limit_ns);
}

}  // namespace mla

extern "C" mla_status mla_selftest_bounded_wait(const mla_plan* plan, void* workspace,
                                                size_t workspace_bytes, uint32_t limit_us,
                                                mla_stream_t stream) {
  if (plan == nullptr || workspace == nullptr || limit_us == 0 || limit_us > 1000000)
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->ws_bytes) return MLA_ERR_WORKSPACE;
  int32_t* err = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + plan->off_err);
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The word starts clear, whatever the workspace held before: the check
  // that follows must see this wait's bit alone.
  if (cudaMemsetAsync(err, 0, sizeof(int32_t), st) != cudaSuccess) return MLA_ERR_CUDA;
  mla::bounded_wait_kernel<<<1, 32, 0, st>>>(err, static_cast<uint64_t>(limit_us) * 1000u);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
