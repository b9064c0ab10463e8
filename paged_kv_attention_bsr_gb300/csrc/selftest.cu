// selftest.cu -- exercises the kernels' failure detection without a fault.
//
// Every wait in the library's kernels is bounded: when a phase does not
// complete in time, the waiting warp records a code in the workspace error
// word and its kernel returns, so the context stays usable and
// attn_workspace_status reports ATTN_ERR_TIMEOUT. This kernel runs that same
// wait on an mbarrier that no thread ever arrives on.
#include "internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

__global__ void wait_selftest_kernel(int32_t* error_word, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  // phase 0 never completes: the wait ends by its limit (or at once if the
  // word already holds another code)
  mbar_wait_limit(smem_u32(&bar), 0, error_word, ERR_WAIT_SELFTEST, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* error_word, uint64_t limit_ns, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(error_word, limit_ns);
  return cudaGetLastError();
}

}  // namespace attn
