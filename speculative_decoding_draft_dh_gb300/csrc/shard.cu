// Vocabulary-sharded draft head: the kernels around the shards' own stage-1 and stage-2 calls.
//
// EAGLE-4 summary page, section "Adaptation has not eliminated high-load regressions" (the
// release serves the target with tensor parallelism over four GPUs), and section "Retrieve
// vocabulary candidates cheaply, then score them exactly": with the vocabulary split over P
// shards (V's columns and W's rows in P contiguous ranges), each shard finds its own K best
// low-rank scores; the global K best are the K best of the union of the shards' lists (a member of
// the global top K is in its own shard's top K), and each candidate's exact logit is computed by
// the shard that owns its W row.  The softmax over the K candidates needs only the row maximum and
// the sum of exponentials, which combine across shards as (max, sum) pairs.
//
// k_add_offset: shard-local ids to global ids.
// k_merge_topk: one block per row ranks the P x K (score, id) entries by counting in the order
//   (score desc, id asc) and writes the K best in order.
// k_localize: global candidate ids to this shard's row index, or -1 where another shard owns them.
// k_shard_stats: one warp per row: owned logits kept, others -inf; the row's (max, sum of exp).
// k_combine_softmax: one warp per row: each candidate's logit from its owner, the shards' pairs
//   combined, probabilities.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int MG_THREADS = 256;

__global__ void k_add_offset(int32_t* __restrict__ idx, long long n, int offset) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int v = idx[i];
    if (v >= 0) idx[i] = v + offset;
  }
}

__global__ void __launch_bounds__(MG_THREADS) k_merge_topk(const int32_t* __restrict__ idx_parts,
                                                         const float* __restrict__ score_parts, int P, int B, int K,
                                                         int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
  extern __shared__ unsigned long long mg[];  // packed (key << 32 | ~id); 0 = no entry
  const int b = blockIdx.x;
  const int n = P * K;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int e = threadIdx.x; e < n; e += MG_THREADS) {
    const int p = e / K, k = e % K;
    const size_t o = ((size_t)p * B + b) * K + k;
    const int v = idx_parts[o];
    const float s = score_parts[o];
    // a padding entry (id < 0) or a NaN score takes no rank
    mg[e] = (v < 0 || s != s) ? 0ull : ((unsigned long long)fkey(s) << 32) | (unsigned long long)(~(uint32_t)v);
  }
  for (int k = threadIdx.x; k < K; k += MG_THREADS) {
    idx_out[(size_t)b * K + k] = -1;
    score_out[(size_t)b * K + k] = -INFINITY;
  }
  __syncthreads();
  int P2 = 1;
  while (P2 < 32 && n * (2 * P2) <= MG_THREADS) P2 <<= 1;
  for (int base = 0; base < n * P2; base += MG_THREADS) {
    const int t = base + (int)threadIdx.x;
    const int i = t / P2, h = t % P2;
    int rank = 0;
    const unsigned long long pi = i < n ? mg[i] : 0ull;
    if (pi)
      for (int j = h; j < n; j += P2) rank += mg[j] > pi ? 1 : 0;
    for (int o = 1; o < P2; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
    if (pi && h == 0 && rank < K) {
      idx_out[(size_t)b * K + rank] = (int32_t)(~(uint32_t)pi);
      score_out[(size_t)b * K + rank] = fkey_inv((uint32_t)(pi >> 32));
    }
  }
}

__global__ void k_localize(const int32_t* __restrict__ idx, long long n, int offset, int vocab_shard,
                           int32_t* __restrict__ local) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const long long v = (long long)idx[i] - offset;
    local[i] = (v >= 0 && v < vocab_shard) ? (int32_t)v : -1;
  }
}

// One warp per row; lane-strided over the K candidates.
__global__ void k_shard_stats(const int32_t* __restrict__ local, int B, int K, float* __restrict__ logits,
                              float* __restrict__ stats) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  float m = -INFINITY;
  for (int k = lane; k < K; k += 32) {
    const size_t o = (size_t)b * K + k;
    const float z = local[o] >= 0 ? logits[o] : -INFINITY;
    logits[o] = z;
    m = fmaxf(m, z);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float s = 0.f;
  if (m != -INFINITY)
    for (int k = lane; k < K; k += 32) s += expf(logits[(size_t)b * K + k] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  if (lane == 0) {
    stats[2 * (size_t)b] = m;
    stats[2 * (size_t)b + 1] = s;
  }
}

__global__ void k_combine_softmax(const float* __restrict__ logits_parts, const float* __restrict__ stats_parts, int P,
                                  int B, int K, float* __restrict__ logits_out, float* __restrict__ probs_out) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  float M = -INFINITY;
  for (int p = 0; p < P; ++p) M = fmaxf(M, stats_parts[2 * ((size_t)p * B + b)]);
  float S = 0.f;
  for (int p = 0; p < P; ++p) {
    const float mp = stats_parts[2 * ((size_t)p * B + b)];
    if (mp != -INFINITY) S += stats_parts[2 * ((size_t)p * B + b) + 1] * expf(mp - M);
  }
  const float inv = 1.f / S;
  for (int k = lane; k < K; k += 32) {
    float z = -INFINITY;
    for (int p = 0; p < P; ++p) z = fmaxf(z, logits_parts[((size_t)p * B + b) * K + k]);
    logits_out[(size_t)b * K + k] = z;
    if (probs_out) probs_out[(size_t)b * K + k] = expf(z - M) * inv;
  }
}

cudaError_t launch_pdl(const Ctx& c, const char* name, dim3 grid, dim3 block, size_t smem, void (*kernel)(),
                       void** args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(name, c.stream);
  cudaError_t e = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kernel), args);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

unsigned grid_for(long long n, int threads, int num_sms) {
  return (unsigned)max(1LL, min((n + threads - 1) / threads, 4LL * num_sms));
}

}  // namespace

cudaError_t launch_add_offset(const Ctx& c, int32_t* idx, long long n, int offset) {
  void* args[] = {&idx, &n, &offset};
  return launch_pdl(c, "shard_offset", dim3(grid_for(n, 256, c.num_sms)), dim3(256), 0,
                    reinterpret_cast<void (*)()>(k_add_offset), args);
}

cudaError_t launch_merge_topk(const Ctx& c, const int32_t* idx_parts, const float* score_parts, int P, int B, int K,
                              int32_t* idx_out, float* score_out) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_merge_topk, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  void* args[] = {&idx_parts, &score_parts, &P, &B, &K, &idx_out, &score_out};
  return launch_pdl(c, "merge_topk", dim3((unsigned)B), dim3(MG_THREADS), (size_t)P * K * 8,
                    reinterpret_cast<void (*)()>(k_merge_topk), args);
}

cudaError_t launch_localize(const Ctx& c, const int32_t* idx, long long n, int offset, int vocab_shard,
                            int32_t* local) {
  void* args[] = {&idx, &n, &offset, &vocab_shard, &local};
  return launch_pdl(c, "shard_localize", dim3(grid_for(n, 256, c.num_sms)), dim3(256), 0,
                    reinterpret_cast<void (*)()>(k_localize), args);
}

cudaError_t launch_shard_stats(const Ctx& c, const int32_t* local, int B, int K, float* logits, float* stats) {
  void* args[] = {&local, &B, &K, &logits, &stats};
  return launch_pdl(c, "shard_stats", dim3((unsigned)((B + 7) / 8)), dim3(256), 0,
                    reinterpret_cast<void (*)()>(k_shard_stats), args);
}

cudaError_t launch_combine_softmax(const Ctx& c, const float* logits_parts, const float* stats_parts, int P, int B,
                                   int K, float* logits_out, float* probs_out) {
  void* args[] = {&logits_parts, &stats_parts, &P, &B, &K, &logits_out, &probs_out};
  return launch_pdl(c, "combine_softmax", dim3((unsigned)((B + 7) / 8)), dim3(256), 0,
                    reinterpret_cast<void (*)()>(k_combine_softmax), args);
}

}  // namespace dh
