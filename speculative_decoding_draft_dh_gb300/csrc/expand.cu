// Expanding frontier nodes of the draft tree: each node's children are its w candidates of highest
// exact probability, with path probabilities carried from the parent.
//
// EAGLE-4 summary page, section "Why a draft tree needs a cost model": products of draft
// probabilities approximate a branch's benefit A in accepted tokens, and a branch is worth
// computing when A over its latency cost C passes a threshold (the page's formula is lost; the
// caller supplies min_benefit = threshold x C, looked up in its latency table for the batch and
// width).  AlphaSignal page, section "Runtime-sized speculation": a top-k of 1 drafts a chain,
// larger k a tree.
//
// k_expand: one block per node.  Every candidate's rank is counted against the others in the order
// (probability desc, token asc, position asc), with a NaN probability below every number; P threads
// share a candidate (interleaved over the others) and add their counts with shuffles.  Candidate
// of rank c < w becomes child c: its token, and its path probability parent x p rounded once to
// fp32.  n_keep counts the children whose path probability is strictly above min_benefit, which
// is always a prefix.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int EX_THREADS = 256;

__global__ void __launch_bounds__(EX_THREADS) k_expand(const float* __restrict__ probs, const int32_t* __restrict__ idx,
                                                     const float* __restrict__ parent_prob, int K, int w,
                                                     float min_benefit, int32_t* __restrict__ child_token,
                                                     float* __restrict__ child_prob, int32_t* __restrict__ n_keep) {
  __shared__ uint32_t sk[DH_MAX_K];
  __shared__ int32_t st[DH_MAX_K];
  __shared__ float sp[DH_MAX_K];
  __shared__ int s_keep;
  const int b = blockIdx.x;
  // the next kernel may launch now (its own wait orders it after this grid); the expansion
  // follows the rescoring kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int k = threadIdx.x; k < K; k += EX_THREADS) {
    const float p = probs[(size_t)b * K + k];
    sp[k] = p;
    sk[k] = isnan(p) ? 0u : fkey(p);
    st[k] = idx[(size_t)b * K + k];
  }
  if (threadIdx.x == 0) s_keep = 0;
  __syncthreads();
  const float par = parent_prob ? parent_prob[b] : 1.0f;
  int P = 1;
  while (P < 32 && K * (2 * P) <= EX_THREADS) P <<= 1;
  for (int base = 0; base < K * P; base += EX_THREADS) {
    const int t = base + (int)threadIdx.x;
    const int i = t / P, h = t % P;
    int rank = 0;
    if (i < K) {
      const uint32_t ki = sk[i];
      const int32_t ti = st[i];
      // thread h counts over j = h, h + P, ...: the P threads of a candidate read consecutive words
      for (int j = h; j < K; j += P) {
        const uint32_t kj = sk[j];
        const int32_t tj = st[j];
        rank += (kj > ki || (kj == ki && (tj < ti || (tj == ti && j < i)))) ? 1 : 0;
      }
    }
    for (int o = 1; o < P; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
    if (i < K && h == 0 && rank < w) {
      const float a = __fmul_rn(par, sp[i]);
      child_token[(size_t)b * w + rank] = st[i];
      child_prob[(size_t)b * w + rank] = a;
      if (a > min_benefit) atomicAdd(&s_keep, 1);
    }
  }
  __syncthreads();
  if (n_keep && threadIdx.x == 0) n_keep[b] = s_keep;
}

}  // namespace

cudaError_t launch_expand(const Ctx& c, const float* probs, const int32_t* idx, const float* parent_prob, int B,
                          int K, int w, float min_benefit, int32_t* child_token, float* child_prob,
                          int32_t* n_keep) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(EX_THREADS);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("expand", c.stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_expand, probs, idx, parent_prob, K, w, min_benefit, child_token,
                                     child_prob, n_keep);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dh
