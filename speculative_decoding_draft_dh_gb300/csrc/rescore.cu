// Stage 2: exact full-rank logits of the retrieved candidates and their softmax.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the candidates' exact logits come from the original full-rank head.  Section "Why a draft tree
// needs a cost model": products of the resulting draft probabilities estimate the benefit of a
// branch; the softmax here runs over the K candidates of a row at temperature 1.
//
// Gather-GEMV: one warp per (row, candidate) streams W[idx] (d contiguous values) with 16-byte
// loads against h[row] staged in shared memory, accumulates in fp32 and reduces with shuffles.  An index outside [0, vocab)
// is never dereferenced: its logit becomes NaN (and so do the row's probabilities).
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int WARPS = 8;          // candidates per block (one warp each)
constexpr int THREADS = WARPS * 32;
constexpr int MAXW = 20;          // 16-byte W vectors per lane in flight (d = 5120 bf16 in one batch)
constexpr int MAX_D_SMEM = 8192;  // h row staged in shared memory (bf16: 16 KB, fp32: 32 KB)

// Block (b, kb) scores candidates kb*8 .. kb*8+7 of row b.  The block stages h[b] in shared
// memory (before waiting on the previous kernel: h does not depend on it), then each warp streams
// its W row with MAXW 16-byte loads per lane in flight and reduces with shuffles.  With probs
// requested, the block adds its candidate count to the row's ticket; the block completing the row
// computes the softmax and resets the ticket.
template <typename T>
__global__ void __launch_bounds__(THREADS) k_rescore(const T* __restrict__ h, const T* __restrict__ W,
                                                     const int32_t* __restrict__ idx, int d, int vocab, int K,
                                                     float* __restrict__ logits, float* __restrict__ probs,
                                                     uint32_t* __restrict__ tickets) {
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* sh_h = reinterpret_cast<T*>(smem_raw);
  __shared__ float red[WARPS];
  __shared__ float s_bcast;
  __shared__ int s_last;
  const int kblocks = (K + WARPS - 1) / WARPS;
  const int b = blockIdx.x / kblocks, kb = blockIdx.x % kblocks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = kb * WARPS + warp;
  const int n_here = min(WARPS, K - kb * WARPS);
  const T* x = h + (size_t)b * d;
  for (int c = threadIdx.x * PER; c < d; c += THREADS * PER)
    *reinterpret_cast<uint4*>(sh_h + c) = __ldg(reinterpret_cast<const uint4*>(x + c));
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  __syncthreads();
  if (k < K) {
    const int pair = b * K + k;
    const int v = idx[pair];
    const bool ok = v >= 0 && v < vocab;
    float acc = 0.f;
    if (ok) {
      const T* w = W + (size_t)v * d;
      for (int c0 = 0; c0 < d; c0 += 32 * PER * MAXW) {
        uint4 wa[MAXW];
#pragma unroll
        for (int q = 0; q < MAXW; ++q) {
          const int c = c0 + (q * 32 + lane) * PER;
          if (c < d) wa[q] = ld_nc_v4(w + c);
        }
#pragma unroll
        for (int q = 0; q < MAXW; ++q) {
          const int c = c0 + (q * 32 + lane) * PER;
          if (c < d) {
            float wf[PER], xf[PER];
            Elem<T>::unpack(wa[q], wf);
            Elem<T>::unpack(*reinterpret_cast<const uint4*>(sh_h + c), xf);
#pragma unroll
            for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    if (lane == 0) logits[pair] = ok ? acc : __int_as_float(0x7FC00000);
  }
  if (!probs) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&tickets[b], (uint32_t)n_here) + (uint32_t)n_here == (uint32_t)K;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // softmax over the row's K logits (written by other blocks: read through L2)
  const float* z = logits + (size_t)b * K;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < K; i += THREADS) m = fmaxf(m, __ldcg(z + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = red[0];
    for (int i = 1; i < WARPS; ++i) mm = fmaxf(mm, red[i]);
    s_bcast = mm;
  }
  __syncthreads();
  m = s_bcast;
  float ssum = 0.f;
  for (int i = threadIdx.x; i < K; i += THREADS) ssum += expf(__ldcg(z + i) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  __syncthreads();
  if (lane == 0) red[warp] = ssum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < WARPS; ++i) tot += red[i];
    s_bcast = 1.f / tot;
    tickets[b] = 0u;
  }
  __syncthreads();
  const float inv = s_bcast;
  for (int i = threadIdx.x; i < K; i += THREADS) probs[(size_t)b * K + i] = expf(__ldcg(z + i) - m) * inv;
}

// ------------------------------------------------------------------------------------------------
// Deduplicated rescoring for large batches: at B = 512, K = 256 the 131072 (row, candidate) pairs
// name about 88K distinct W rows, so reading each distinct row once saves a third of the traffic.
//   k_link:  one thread per pair pushes the pair onto a per-W-row list (atomic exchange on
//            head[v]); the first pair of a row appends v to the list of distinct rows.
//   k_rescore_uniq: persistent warps take distinct rows in turn, hold the W row in registers and
//            score it against h[b] of every pair on its list; out-of-range ids form one more list
//            whose logits become NaN.  Per-row tickets trigger the softmax as in k_rescore.
// Lists and counters live in the workspace and are left empty for the next call.

struct UniqState {
  uint32_t nuniq, done, bad_head, pad;
};

__global__ void k_link(const int32_t* __restrict__ idx, int BK, int vocab, uint32_t* __restrict__ head,
                       uint32_t* __restrict__ next, uint32_t* __restrict__ uniq, UniqState* __restrict__ st) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= BK) return;
  const int v = idx[p];
  if (v < 0 || v >= vocab) {
    next[p] = atomicExch(&st->bad_head, (uint32_t)p + 1u);
    return;
  }
  const uint32_t old = atomicExch(&head[v], (uint32_t)p + 1u);
  next[p] = old;
  if (old == 0u) uniq[atomicAdd(&st->nuniq, 1u)] = (uint32_t)v;
}

// softmax of row b (K logits, written by other warps: read through L2) by one warp
__device__ void warp_softmax(const float* __restrict__ logits, float* __restrict__ probs, int b, int K) {
  const int lane = threadIdx.x & 31;
  const float* z = logits + (size_t)b * K;
  float m = -INFINITY;
  for (int i = lane; i < K; i += 32) m = fmaxf(m, __ldcg(z + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float ssum = 0.f;
  for (int i = lane; i < K; i += 32) ssum += expf(__ldcg(z + i) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  const float inv = 1.f / ssum;
  for (int i = lane; i < K; i += 32) probs[(size_t)b * K + i] = expf(__ldcg(z + i) - m) * inv;
}

// lane 0 counts one finished pair of row b; returns (to all lanes) whether the row is complete
__device__ __forceinline__ bool finish_pair(uint32_t* tickets, int b, int K, bool with_probs) {
  if (!with_probs) return false;
  uint32_t last = 0;
  if ((threadIdx.x & 31) == 0) {
    __threadfence();
    last = atomicAdd(&tickets[b], 1u) == (uint32_t)(K - 1);
    if (last) __threadfence();
  }
  return __shfl_sync(0xFFFFFFFFu, last, 0) != 0;
}

template <typename T>
__global__ void __launch_bounds__(THREADS) k_rescore_uniq(const T* __restrict__ h, const T* __restrict__ W, int d,
                                                          int K, const uint32_t* __restrict__ uniq,
                                                          uint32_t* __restrict__ head, const uint32_t* __restrict__ next,
                                                          UniqState* __restrict__ st, float* __restrict__ logits,
                                                          float* __restrict__ probs, uint32_t* __restrict__ tickets) {
  constexpr int PER = Elem<T>::PER16;
  constexpr int HB = 5;  // h vectors per lane in flight
  asm volatile("griddepcontrol.wait;" ::: "memory");  // lists come from k_link
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * WARPS + (threadIdx.x >> 5);
  const int nw = gridDim.x * WARPS;
  const uint32_t nuniq = __ldcg(&st->nuniq);
  const bool with_probs = probs != nullptr;
  for (uint32_t u = gw; u <= nuniq; u += nw) {
    if (u == nuniq) {  // out-of-range ids
      uint32_t q = __ldcg(&st->bad_head);
      while (q != 0u) {
        const int pair = (int)q - 1;
        if (lane == 0) logits[pair] = __int_as_float(0x7FC00000);
        if (finish_pair(tickets, pair / K, K, with_probs)) {
          warp_softmax(logits, probs, pair / K, K);
          if (lane == 0) tickets[pair / K] = 0u;
        }
        q = __ldcg(next + pair);
      }
      if (lane == 0) st->bad_head = 0u;
      continue;
    }
    const uint32_t v = __ldcg(uniq + u);
    const T* w = W + (size_t)v * d;
    uint4 wa[MAXW];
#pragma unroll
    for (int i = 0; i < MAXW; ++i) {
      const int c = (i * 32 + lane) * PER;
      if (c < d) wa[i] = ld_nc_v4(w + c);
    }
    uint32_t q = __ldcg(head + v);
    while (q != 0u) {
      const int pair = (int)q - 1;
      const int b = pair / K;
      const T* x = h + (size_t)b * d;
      float acc = 0.f;
#pragma unroll
      for (int i0 = 0; i0 < MAXW; i0 += HB) {
        uint4 xa[HB];
#pragma unroll
        for (int i = 0; i < HB; ++i) {
          const int c = ((i0 + i) * 32 + lane) * PER;
          if (c < d) xa[i] = __ldg(reinterpret_cast<const uint4*>(x + c));
        }
#pragma unroll
        for (int i = 0; i < HB; ++i) {
          const int c = ((i0 + i) * 32 + lane) * PER;
          if (c < d) {
            float wf[PER], xf[PER];
            Elem<T>::unpack(wa[i0 + i], wf);
            Elem<T>::unpack(xa[i], xf);
#pragma unroll
            for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
          }
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (lane == 0) logits[pair] = acc;
      if (finish_pair(tickets, b, K, with_probs)) {
        warp_softmax(logits, probs, b, K);
        if (lane == 0) tickets[b] = 0u;
      }
      q = __ldcg(next + pair);
    }
    if (lane == 0) head[v] = 0u;
  }
  // the last warp out leaves the counters at zero for the next call
  if (lane == 0) {
    __threadfence();
    if (atomicAdd(&st->done, 1u) == (uint32_t)(nw - 1)) {
      st->nuniq = 0u;
      st->done = 0u;
      __threadfence();
    }
  }
}

template <typename T>
cudaError_t run_uniq(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                     float* logits, float* probs, uint32_t* tickets, UniqState* st, uint32_t* head, uint32_t* next,
                     uint32_t* uniq) {
  const int BK = B * K;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((BK + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore_link", c.stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_link, idx, BK, vocab, head, next, uniq, st);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_rescore_uniq<T>, THREADS, 0);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(c.num_sms * max(1, per_sm)));
  cfg.blockDim = dim3(THREADS);
  prof_before("rescore_uniq", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore_uniq<T>, static_cast<const T*>(h), static_cast<const T*>(W), d, K,
                         (const uint32_t*)uniq, head, (const uint32_t*)next, st, logits, probs, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                int K, float* logits, float* probs, uint32_t* tickets) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the blocks may start while the stage-1 kernel drains; they
  // stage h and then wait (griddepcontrol.wait) for its results.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ((K + WARPS - 1) / WARPS)));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)d * sizeof(T);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore<T>, static_cast<const T*>(h), static_cast<const T*>(W), idx, d, vocab, K,
                         logits, probs, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool rescore_supported(int d) { return d <= MAX_D_SMEM; }

// The deduplicated path holds a W row in registers (MAXW 16-byte vectors per lane).
bool rescore_uniq_used(int B, int d, int K, int dtype) {
  const int per = dtype == DH_BF16 ? 8 : 4;
  return (long long)B * K >= 32768 && d <= MAXW * 32 * per;
}

size_t rescore_uniq_bytes(int B, int vocab, int K) {
  return align_up(sizeof(UniqState), 256) + align_up((size_t)vocab * 4, 256) + 2 * align_up((size_t)B * K * 4, 256);
}

cudaError_t launch_rescore_uniq(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets,
                                void* area) {
  char* a = static_cast<char*>(area);
  UniqState* st = reinterpret_cast<UniqState*>(a);
  a += align_up(sizeof(UniqState), 256);
  uint32_t* head = reinterpret_cast<uint32_t*>(a);
  a += align_up((size_t)vocab * 4, 256);
  uint32_t* next = reinterpret_cast<uint32_t*>(a);
  a += align_up((size_t)B * K * 4, 256);
  uint32_t* uniq = reinterpret_cast<uint32_t*>(a);
  if (dtype == DH_BF16)
    return run_uniq<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, st, head, next, uniq);
  return run_uniq<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, st, head, next, uniq);
}

cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                           int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
  return run<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
}

}  // namespace dh
