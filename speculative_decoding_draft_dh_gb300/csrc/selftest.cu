// Self-test of the bounded waits used by the pipelined kernels (no counterpart on the pages).
//
// k_wait_probe runs the same two waits the production kernels use, on conditions that are never
// met, with a short limit:
//   mode 0: an mbarrier that nothing arrives at (as a TMA or MMA completion that never comes);
//   mode 1: a grid barrier expecting one more block than the grid has.
// Each must give up after limit_us, raise DH_ERR_TIMEOUT in the workspace status word and return,
// leaving the CUDA context usable.  Nothing faults, traps or hangs.
#include "grid_sync.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

__global__ void k_wait_probe(int mode, unsigned long long limit_ns, int* status, GridBar* bar) {
  __shared__ uint64_t mbar;
  __shared__ volatile int s_fail;
  if (threadIdx.x == 0) {
    s_fail = 0;
    sm100::mbar_init(&mbar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (mode == 0) {
    if (threadIdx.x == 0 && !sm100::mbar_wait(&mbar, 0, limit_ns)) atomicOr(status, 1 << DH_ERR_TIMEOUT);
  } else {
    if (!grid_sync(bar, gridDim.x + 1, limit_ns, status, &s_fail) && blockIdx.x == 0 && threadIdx.x == 0) {
      // the barrier never filled: undo this launch's arrivals so the counter is clean again
      atomicExch(&bar->count, 0u);
    }
  }
}

}  // namespace
}  // namespace dh

using namespace dh;

extern "C" int dh_selftest_wait_timeout(int mode, int limit_us, void* workspace, size_t ws_bytes, void* stream) {
  if ((mode != 0 && mode != 1) || limit_us <= 0 || limit_us > 1000000) return DH_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < WS_HEADER) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  const int blocks = mode == 0 ? 1 : 2;  // two co-resident blocks, barrier expects three
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(32);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_wait_probe, mode, (unsigned long long)limit_us * 1000ull,
                                     reinterpret_cast<int*>(ws), reinterpret_cast<GridBar*>(ws + WS_BARRIER_OFFSET));
  if (note_error(e, "cudaLaunchKernelEx(k_wait_probe)") != cudaSuccess) return DH_ERR_CUDA;
  return DH_OK;
}
