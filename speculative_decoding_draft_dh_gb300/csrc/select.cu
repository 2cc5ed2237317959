// Stage 1c: exact top-K per row from the group records, one block per row (see select.cuh).
#include "select.cuh"

namespace dh {
namespace {

// MINB blocks per SM: 1 for up to 1.5 rows per SM (all registers for one block), 2 beyond (64
// registers a thread, so two latency-bound blocks share each SM: 512 rows on 152 SMs select in
// 48 instead of 61 µs, 300 rows in 24 instead of 29 µs; at 200 rows the single wave of slower
// blocks loses to 1.3 waves of faster ones).  With two blocks per SM the rescoring kernel is
// released only as the blocks finish, so that its blocks, launched early, do not take the SM slots
// later waves need.
template <typename T, int MINB>
__global__ void __launch_bounds__(sel::SEL_THREADS, MINB) k_select(const GroupRec* __restrict__ recs,
                                                               const T* __restrict__ t, unsigned long long* acc,
                                                               const T* __restrict__ V, int r, int vocab, int K,
                                                               int32_t* __restrict__ idx_out,
                                                               float* __restrict__ score_out,
                                                               uint32_t* __restrict__ tickets) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  // the rescoring kernel that follows counts the row's candidates with a ticket that starts at zero
  // (where the caller's workspace keeps other calls' data, it may hold anything before)
  if (tickets && threadIdx.x == 0) tickets[blockIdx.x] = 0u;
  // the rescoring kernel may launch now (it stages h, then waits for this grid's candidates)
  if (MINB == 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the records come from the previous kernel
  const int row = blockIdx.x;
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  sel::select_row<T>(smem_raw, recs + (size_t)row * n_groups, t ? t + (size_t)row * r : nullptr,
                     acc ? acc + (size_t)row * r : nullptr, (int)gridDim.x * r, V, r, vocab, K,
                     idx_out + (size_t)row * K, score_out + (size_t)row * K);
  if (MINB != 1) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T>
cudaError_t run(const Ctx& c, const GroupRec* recs, const void* t, unsigned long long* acc, const void* V, int B,
                int r, int vocab, int K, int32_t* idx_out, float* score_out, uint32_t* tickets) {
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const size_t smem = sel::select_smem_bytes(n_groups);
  const bool waves = 2 * B > 3 * c.num_sms;
  static unsigned long long smem_done1 = 0, smem_done2 = 0;
  const bool first2 = waves && c.device < 64 && !((smem_done2 >> c.device) & 1ull);
  cudaError_t e = waves ? allow_max_smem(k_select<T, 2>, c.device, &smem_done2)
                        : allow_max_smem(k_select<T, 1>, c.device, &smem_done1);
  if (e != cudaSuccess) return e;
  if (first2) {  // two blocks' shared memory on one SM
    e = cudaFuncSetAttribute(k_select<T, 2>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return note_error(e, "cudaFuncSetAttribute(PreferredSharedMemoryCarveout)");
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(sel::SEL_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("select", c.stream);
  e = waves ? cudaLaunchKernelEx(&cfg, k_select<T, 2>, recs, static_cast<const T*>(t), acc, static_cast<const T*>(V), r,
                                 vocab, K, idx_out, score_out, tickets)
            : cudaLaunchKernelEx(&cfg, k_select<T, 1>, recs, static_cast<const T*>(t), acc, static_cast<const T*>(V), r,
                                 vocab, K, idx_out, score_out, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const Ctx& c, const GroupRec* recs, const void* t, unsigned long long* acc,
                          const void* V, int B, int r, int vocab, int K, int dtype, int32_t* idx_out,
                          float* score_out, uint32_t* tickets) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, recs, t, acc, V, B, r, vocab, K, idx_out, score_out, tickets);
  return run<float>(c, recs, t, acc, V, B, r, vocab, K, idx_out, score_out, tickets);
}

}  // namespace dh
