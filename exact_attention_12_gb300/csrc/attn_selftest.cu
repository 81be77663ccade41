// attn_selftest_timeout: exercises the kernels' failure path on purpose.
//
// Every wait in the attention kernels is bounded; when one gives up, the
// kernel records ATTN_ERR_TIMEOUT and the wait site in the workspace status
// words and returns, and attn_check reports it.  This kernel runs exactly
// that path: it waits on an mbarrier that nothing ever arrives at, with a
// short limit, so the wait must give up.  Nothing faults, traps or hangs.
#include "attn.h"
#include "attn_kernels.cuh"
#include "sm103.cuh"

namespace {

constexpr int kSiteSelfTest = 99;

__global__ void __launch_bounds__(32) wait_forever_bounded(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    sm103::mbar_init(&bar, 1);
    sm103::fence_mbar_init();
  }
  __syncthreads();
  const sm103::WaitCtx wc{&abort_flag, status, limit_ns};
  // phase 0 of `bar` never completes: no thread arrives on it
  sm103::mbar_wait(&bar, 0, wc, kSiteSelfTest);
}

}  // namespace

extern "C" attn_status attn_selftest_timeout(void* ws, uint64_t limit_ns, void* stream) {
  if (ws == nullptr)
    return static_cast<attn_status>(attn::record_error(ATTN_ERR_WORKSPACE, "workspace is NULL"));
  if (limit_ns < 1000000ull) limit_ns = 1000000ull;          // 1 ms
  if (limit_ns > 2000000000ull) limit_ns = 2000000000ull;    // 2 s
  wait_forever_bounded<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int*>(ws),
                                                                         limit_ns);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess)
    return static_cast<attn_status>(attn::record_error(ATTN_ERR_CUDA, cudaGetErrorString(e)));
  return ATTN_OK;
}
