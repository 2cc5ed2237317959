// Sizing the next draft level: how many of the frontier's candidate children to draft and verify
// next, at the current load.
//
// EAGLE-4 summary page, section "Why a draft tree needs a cost model": products of draft
// probabilities estimate a branch's benefit A in accepted tokens; latency tables indexed by batch
// and verification width price another level; each round decides whether to deepen the tree and how
// wide to go, by comparing benefit with cost against a threshold (the page's formula is lost: the
// per-branch reading is that the j-th best child is kept while A_j > theta x (cost[j+1] - cost[j]),
// its benefit per unit of the latency it adds).  AlphaSignal page, section "Runtime-sized
// speculation": depth and branching are chosen for the active batch size.
//
// k_size_level: one block per request.  The request's valid children (slot k < n_valid of frontier
// node f) are ranked by counting in the order (A desc, f asc, slot asc), with a NaN probability
// below every number; P threads share a child and add their counts with shuffles.  The child of
// rank j compares its A with theta x (cost[j+1] - cost[j]) of the batch's cost row, each operation
// rounded once in fp32 (no fused multiply-add), and the first rank that fails (or the width limit)
// gives the width.  The kept children are written in rank order: parent slot, token, A.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int SZ_THREADS = 256;

struct SizeParams {
  const float* child_prob;
  const int32_t* child_token;
  const int32_t* n_valid;
  const float* cost;
  const int32_t* bin_batch;
  int F, Wc, n_bins, wmax, batch;
  float theta;
  int32_t* width;
  int32_t* sel_parent;
  int32_t* sel_token;
  float* sel_prob;
};

__global__ void __launch_bounds__(SZ_THREADS) k_size_level(SizeParams p) {
  extern __shared__ uint32_t sz_smem[];
  const int n_all = p.F * p.Wc;
  uint32_t* key = sz_smem;  // fkey(A) (0 for NaN); 0xFFFFFFFF marks an invalid child
  int32_t* by_rank = reinterpret_cast<int32_t*>(sz_smem + n_all);  // the child at each rank < wmax
  __shared__ int s_width, s_bin;
  const int r = blockIdx.x;
  const size_t base = (size_t)r * n_all;
  // the next kernel may launch now (its own wait orders it after this grid); the children come
  // from the expansion kernel (programmatic dependent launch)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    int bin = p.n_bins - 1;
    for (int i = 0; i < p.n_bins; ++i)
      if (p.batch <= p.bin_batch[i]) { bin = i; break; }
    s_bin = bin;
    s_width = p.wmax;
  }
  for (int c = threadIdx.x; c < n_all; c += SZ_THREADS) {
    const int f = c / p.Wc, k = c % p.Wc;
    const int nv = p.n_valid ? min(max(p.n_valid[(size_t)r * p.F + f], 0), p.Wc) : p.Wc;
    const float a = p.child_prob[base + c];
    key[c] = k < nv ? (isnan(a) ? 0u : fkey(a)) : 0xFFFFFFFFu;  // 0xFFFFFFFF marks an invalid child
  }
  for (int j = threadIdx.x; j < p.wmax; j += SZ_THREADS) by_rank[j] = -1;
  __syncthreads();
  // rank by counting over the valid children: larger key first, then the lower index c (which
  // orders by parent, then slot)
  int P = 1;
  while (P < 32 && n_all * (2 * P) <= SZ_THREADS) P <<= 1;
  for (int b0 = 0; b0 < n_all * P; b0 += SZ_THREADS) {
    const int t = b0 + (int)threadIdx.x;
    const int i = t / P, h = t % P;
    int rank = 0;
    const uint32_t ki = i < n_all ? key[i] : 0xFFFFFFFFu;
    if (i < n_all && ki != 0xFFFFFFFFu) {
      for (int j = h; j < n_all; j += P) {
        const uint32_t kj = key[j];
        rank += (kj != 0xFFFFFFFFu && (kj > ki || (kj == ki && j < i))) ? 1 : 0;
      }
    }
    for (int o = 1; o < P; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
    if (i < n_all && h == 0 && ki != 0xFFFFFFFFu && rank < p.wmax) by_rank[rank] = i;
  }
  __syncthreads();
  // the rule, rank by rank: keep while A > theta x (cost[j+1] - cost[j])
  const float* crow = p.cost + (size_t)s_bin * (p.wmax + 1);
  for (int j = threadIdx.x; j < p.wmax; j += SZ_THREADS) {
    const int c = by_rank[j];
    bool keep = false;
    if (c >= 0) {
      const float thr = __fmul_rn(p.theta, __fsub_rn(crow[j + 1], crow[j]));
      keep = p.child_prob[base + c] > thr;
    }
    if (!keep) atomicMin(&s_width, j);
  }
  __syncthreads();
  const int w = s_width;
  if (threadIdx.x == 0) p.width[r] = w;
  for (int j = threadIdx.x; j < p.wmax; j += SZ_THREADS) {
    const size_t o = (size_t)r * p.wmax + j;
    const int c = j < w ? by_rank[j] : -1;
    p.sel_parent[o] = c >= 0 ? c / p.Wc : -1;
    p.sel_token[o] = c >= 0 ? p.child_token[base + c] : -1;
    p.sel_prob[o] = c >= 0 ? p.child_prob[base + c] : 0.f;
  }
}

}  // namespace

size_t size_level_smem(int F, int Wc, int wmax) { return ((size_t)F * Wc + (size_t)wmax) * 4; }

cudaError_t launch_size_level(const Ctx& c, const float* child_prob, const int32_t* child_token,
                              const int32_t* n_valid, int R, int F, int Wc, const float* cost,
                              const int32_t* bin_batch, int n_bins, int wmax, int batch, float theta,
                              int32_t* width, int32_t* sel_parent, int32_t* sel_token, float* sel_prob) {
  SizeParams p;
  p.child_prob = child_prob;
  p.child_token = child_token;
  p.n_valid = n_valid;
  p.cost = cost;
  p.bin_batch = bin_batch;
  p.F = F;
  p.Wc = Wc;
  p.n_bins = n_bins;
  p.wmax = wmax;
  p.batch = batch;
  p.theta = theta;
  p.width = width;
  p.sel_parent = sel_parent;
  p.sel_token = sel_token;
  p.sel_prob = sel_prob;
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_size_level, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)R);
  cfg.blockDim = dim3(SZ_THREADS);
  cfg.dynamicSmemBytes = size_level_smem(F, Wc, wmax);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("size_level", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_size_level, p);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace dh
