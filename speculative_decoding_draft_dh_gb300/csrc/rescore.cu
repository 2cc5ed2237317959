// Stage 2: exact full-rank logits of the retrieved candidates and their softmax.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the candidates' exact logits come from the original full-rank head.  Section "Why a draft tree
// needs a cost model": products of the resulting draft probabilities estimate the benefit of a
// branch; the softmax here runs over the K candidates of a row at temperature 1.
//
// Gather-GEMV: one block per (row, candidate) streams W[idx] (d contiguous values) and h[row] with
// 16-byte loads, accumulates in fp32 and reduces with warp shuffles.  An index outside [0, vocab)
// is never dereferenced: its logit becomes NaN (and so do the row's probabilities).
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int THREADS = 128;
constexpr int MAXV = 8;  // 16-byte vectors per thread in flight per batch of the row

// One block per (row, candidate).  Each thread issues up to MAXV 16-byte loads of the W row (and
// the matching h chunk) before using any of them, so a 10 KB row costs one memory round trip.
// With probs requested, the last block of a row to finish (atomic ticket in the workspace)
// computes the row's softmax and resets the ticket for the next call.
template <typename T>
__global__ void __launch_bounds__(THREADS) k_rescore(const T* __restrict__ h, const T* __restrict__ W,
                                                     const int32_t* __restrict__ idx, int d, int vocab, int K,
                                                     float* __restrict__ logits, float* __restrict__ probs,
                                                     uint32_t* __restrict__ tickets) {
  constexpr int PER = Elem<T>::PER16;
  __shared__ float red[THREADS / 32];
  __shared__ float s_bcast;
  __shared__ int s_last;
  const int pair = blockIdx.x;
  const int b = pair / K;
  const T* x = h + (size_t)b * d;
  // h does not depend on the previous kernel on the stream: fetch its first chunk before waiting
  uint4 xa[MAXV];
#pragma unroll
  for (int q = 0; q < MAXV; ++q) {
    const int c = (q * THREADS + (int)threadIdx.x) * PER;
    if (c < d) xa[q] = __ldg(reinterpret_cast<const uint4*>(x + c));
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  const int v = idx[pair];
  const bool ok = v >= 0 && v < vocab;
  float acc = 0.f;
  if (ok) {
    const T* w = W + (size_t)v * d;
    for (int c0 = 0; c0 < d; c0 += THREADS * PER * MAXV) {
      uint4 wa[MAXV];
#pragma unroll
      for (int q = 0; q < MAXV; ++q) {
        const int c = c0 + (q * THREADS + (int)threadIdx.x) * PER;
        if (c < d) {
          wa[q] = ld_nc_v4(w + c);
          if (c0 > 0) xa[q] = __ldg(reinterpret_cast<const uint4*>(x + c));
        }
      }
#pragma unroll
      for (int q = 0; q < MAXV; ++q) {
        const int c = c0 + (q * THREADS + (int)threadIdx.x) * PER;
        if (c < d) {
          float wf[PER], xf[PER];
          Elem<T>::unpack(wa[q], wf);
          Elem<T>::unpack(xa[q], xf);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
        }
      }
    }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < THREADS / 32; ++i) sum += red[i];
    logits[pair] = ok ? sum : __int_as_float(0x7FC00000);
    if (probs) {
      __threadfence();
      s_last = atomicAdd(&tickets[b], 1u) == (uint32_t)(K - 1);
    }
  }
  if (!probs) return;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // softmax over the row's K logits (written by other blocks: read through L2)
  const float* z = logits + (size_t)b * K;
  float m = -INFINITY;
  for (int k = threadIdx.x; k < K; k += THREADS) m = fmaxf(m, __ldcg(z + k));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = red[0];
    for (int i = 1; i < THREADS / 32; ++i) mm = fmaxf(mm, red[i]);
    s_bcast = mm;
  }
  __syncthreads();
  m = s_bcast;
  float ssum = 0.f;
  for (int k = threadIdx.x; k < K; k += THREADS) ssum += expf(__ldcg(z + k) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  __syncthreads();
  if (lane == 0) red[warp] = ssum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < THREADS / 32; ++i) tot += red[i];
    s_bcast = 1.f / tot;
    tickets[b] = 0u;
  }
  __syncthreads();
  const float inv = s_bcast;
  for (int k = threadIdx.x; k < K; k += THREADS) probs[(size_t)b * K + k] = expf(__ldcg(z + k) - m) * inv;
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                int K, float* logits, float* probs, uint32_t* tickets) {
  // Programmatic dependent launch: the blocks may start while the stage-1 kernel drains; they
  // prefetch h and then wait (griddepcontrol.wait) for its results.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * K));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore", c.stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_rescore<T>, static_cast<const T*>(h), static_cast<const T*>(W), idx,
                                     d, vocab, K, logits, probs, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                           int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
  return run<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
}

}  // namespace dh
