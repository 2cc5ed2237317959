// Greedy draft-tree acceptance.
//
// daily.dev "EAGLE-4 speeds up LLM inference with an adaptive speculative decoding drafter",
// section "How it works": the target checks every drafted token in one forward pass; drafted
// tokens are kept while they match, and the first mismatch is replaced by the target's own token.
// EAGLE-4 summary page, section "Distribution preservation has algorithmic and implementation
// conditions": greedy decoding follows the target's choices.  AlphaSignal "EAGLE-4 Triples Qwen3
// Inference Speed by Adapting to Serving Load", section "Runtime-sized speculation": top-k = 1
// drafts a chain, larger k a tree.
//
// k_tree_argmax: one block per (request, node) row scans the vocabulary with 16-byte loads, keeps
// a running (max, id) per thread and reduces a packed 64-bit key (order-preserving score bits, then
// the complement of the id) so that ties resolve to the lowest id exactly.  This scan is all of the
// step's memory traffic.
// k_tree_walk: one block per request; thread n checks its edge, pointer jumping gives every node
// "all edges to the root accepted" and its depth, a block max picks the deepest accepted node
// (lowest index on ties) and thread 0 writes the path.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int ARGMAX_THREADS = 256;

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

// Each thread scans its 16-byte vectors in increasing id order keeping (best value, its id).  Per
// vector it takes the max with an fmax tree and only searches for the id when that max beats the
// running best (strictly: an equal value later in the row has a larger id), which happens a few
// times per thread.  The block then reduces (value, id) with ties to the lower id.  NaN ranks below
// every number: fmaxf drops NaN operands, a vector of NaN only (max NaN) is skipped, and a thread
// that saw no number keeps its first id with key 0, below the key of any number, so a row holding
// only NaN gives its lowest id, 0.
template <typename T>
__global__ void __launch_bounds__(ARGMAX_THREADS) k_tree_argmax(const T* __restrict__ logits, int vocab,
                                                                int32_t* __restrict__ am) {
  constexpr int PER = Elem<T>::PER16;
  constexpr int BATCH = 8;  // 16-byte loads per thread in flight
  __shared__ unsigned long long red[ARGMAX_THREADS / 32];
  const size_t row = blockIdx.x;
  const T* p = logits + row * (size_t)vocab;
  float best = -INFINITY;
  int best_id = -1;
  for (int c0 = threadIdx.x * PER; c0 < vocab; c0 += ARGMAX_THREADS * PER * BATCH) {
    uint4 u[BATCH];
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int c = c0 + q * ARGMAX_THREADS * PER;
      if (c < vocab) u[q] = ld_nc_v4(p + c);
    }
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int c = c0 + q * ARGMAX_THREADS * PER;
      if (c < vocab) {
        float x[PER];
        Elem<T>::unpack(u[q], x);
        float m = x[0];
#pragma unroll
        for (int e = 1; e < PER; ++e) m = fmaxf(m, x[e]);
        if (m > best || (best_id < 0 && m == m)) {
          int e0 = 0;
#pragma unroll
          for (int e = PER - 1; e >= 0; --e)
            if (x[e] == m) e0 = e;  // first position holding the max
          best = m;
          best_id = c + e0;
        }
      }
    }
  }
  // fkey of any number is at least fkey(-inf) = 0x007FFFFF > 0, so a thread without a number
  // (key high word 0) ranks below every thread with one
  const int first_id = (int)threadIdx.x * PER;
  unsigned long long key = best_id >= 0 ? ((unsigned long long)fkey(best) << 32) |
                                              (unsigned long long)(0xFFFFFFFFu - (uint32_t)best_id)
                           : first_id < vocab ? (unsigned long long)(0xFFFFFFFFu - (uint32_t)first_id)
                                              : 0ull;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) key = umax64(key, __shfl_xor_sync(0xFFFFFFFFu, key, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = key;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < ARGMAX_THREADS / 32; ++w) key = umax64(key, red[w]);
    am[row] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
  }
}

__global__ void k_tree_walk(const int32_t* __restrict__ parent, const int32_t* __restrict__ token,
                            const int32_t* __restrict__ am, int N, int32_t* __restrict__ argmax_out,
                            int32_t* __restrict__ path, int32_t* __restrict__ len, int32_t* __restrict__ bonus,
                            int32_t* __restrict__ err) {
  __shared__ int32_t s_par[DH_MAX_TREE_NODES];
  __shared__ int32_t s_anc[DH_MAX_TREE_NODES];
  __shared__ int32_t s_dep[DH_MAX_TREE_NODES];
  __shared__ unsigned char s_ok[DH_MAX_TREE_NODES];
  __shared__ int32_t s_a[DH_MAX_TREE_NODES];
  __shared__ unsigned int s_best;
  const int b = blockIdx.x;
  const int n = threadIdx.x;
  const bool live = n < N;
  const size_t base = (size_t)b * N;
  int p = -1;
  if (live) {
    p = parent[base + n];
    s_par[n] = p;
    s_a[n] = am[base + n];
    if (argmax_out) argmax_out[base + n] = s_a[n];
    path[base + n] = -1;
  }
  const bool good = !live || (n == 0 ? p == -1 : (p >= 0 && p < n));
  if (threadIdx.x == 0) s_best = 0u;
  if (!__syncthreads_and(good)) {
    if (n == 0) {
      len[b] = -1;
      bonus[b] = -1;
      if (err) err[b] = DH_ERR_BAD_INPUT;
    }
    return;
  }
  // segment [n, anc): edges all accepted (ok) and their count (dep)
  int anc = -1, dep = 0;
  bool ok = true;
  if (live && n > 0) {
    anc = p;
    dep = 1;
    ok = token[base + n] == s_a[p];
  }
  if (live) { s_anc[n] = anc; s_dep[n] = dep; s_ok[n] = ok; }
  __syncthreads();
  for (;;) {
    const bool more = live && anc >= 0;
    if (!__syncthreads_or(more)) break;
    int na = anc, nd = dep;
    bool nok = ok;
    if (more) {
      na = s_anc[anc];
      nd = dep + s_dep[anc];
      nok = ok && s_ok[anc];
    }
    __syncthreads();
    if (live) { anc = na; dep = nd; ok = nok; s_anc[n] = anc; s_dep[n] = dep; s_ok[n] = ok; }
  }
  if (live && ok) atomicMax(&s_best, ((unsigned int)dep << 16) | (0xFFFFu - (unsigned int)n));
  __syncthreads();
  if (n == 0) {
    const unsigned int key = s_best;
    const int last = (int)(0xFFFFu - (key & 0xFFFFu));
    const int depth = (int)(key >> 16);
    len[b] = depth;
    bonus[b] = s_a[last];
    if (err) err[b] = 0;
    for (int m = last, j = depth; m >= 0 && j >= 0; m = s_par[m], --j) path[base + j] = m;
  }
}

template <typename T>
cudaError_t run(const Ctx& c, const void* logits, const int32_t* parent, const int32_t* token, int B, int N,
                int vocab, int32_t* am_ws, int32_t* argmax_out, int32_t* path, int32_t* len, int32_t* bonus,
                int32_t* err) {
  const long long rows = (long long)B * N;
  prof_before("tree_argmax", c.stream);
  k_tree_argmax<T><<<(unsigned)rows, ARGMAX_THREADS, 0, c.stream>>>(static_cast<const T*>(logits), vocab, am_ws);
  prof_after(c.stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int threads = (N + 31) / 32 * 32;
  prof_before("tree_walk", c.stream);
  k_tree_walk<<<B, threads, 0, c.stream>>>(parent, token, am_ws, N, argmax_out, path, len, bonus, err);
  prof_after(c.stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tree(const Ctx& c, const void* logits, const int32_t* parent, const int32_t* token, int B,
                        int N, int vocab, int dtype, int32_t* am_ws, int32_t* argmax_out, int32_t* path,
                        int32_t* len, int32_t* bonus, int32_t* err) {
  if (dtype == DH_BF16)
    return run<__nv_bfloat16>(c, logits, parent, token, B, N, vocab, am_ws, argmax_out, path, len, bonus, err);
  return run<float>(c, logits, parent, token, B, N, vocab, am_ws, argmax_out, path, len, bonus, err);
}

}  // namespace dh
