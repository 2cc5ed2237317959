// Self-test of the bounded waits used by the pipelined kernels (no counterpart on the pages).
//
// k_wait_probe runs the wait the production kernels use for TMA, bulk-copy and MMA completions (an
// mbarrier phase wait with a time limit) on an mbarrier that nothing arrives at, with a short limit.
// It must give up after limit_us, raise DH_ERR_TIMEOUT in the workspace status word and return,
// leaving the CUDA context usable.  Nothing faults, traps or hangs.
#include "dh_internal.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

__global__ void k_wait_probe(unsigned long long limit_ns, int* status) {
  __shared__ uint64_t mbar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&mbar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !sm100::mbar_wait(&mbar, 0, limit_ns)) atomicOr(status, 1 << DH_ERR_TIMEOUT);
}

}  // namespace
}  // namespace dh

using namespace dh;

extern "C" int dh_selftest_wait_timeout(int mode, int limit_us, void* workspace, size_t ws_bytes, void* stream) {
  if (mode != 0 || limit_us <= 0 || limit_us > 1000000) return DH_ERR_INVALID_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || ws_bytes < WS_HEADER) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  k_wait_probe<<<1, 32, 0, c.stream>>>((unsigned long long)limit_us * 1000ull, static_cast<int*>(workspace));
  if (note_error(cudaGetLastError(), "k_wait_probe launch") != cudaSuccess) return DH_ERR_CUDA;
  return DH_OK;
}
