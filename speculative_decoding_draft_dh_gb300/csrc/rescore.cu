// Stage 2: exact full-rank logits of the retrieved candidates and their softmax.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the candidates' exact logits come from the original full-rank head.  Section "Why a draft tree
// needs a cost model": products of the resulting draft probabilities estimate the benefit of a
// branch; the softmax here runs over the K candidates of a row at temperature 1.
//
// Gather-GEMV: one warp per (row, candidate) streams W[idx] (d contiguous values) and h[row] with
// 16-byte loads, accumulates in fp32 and reduces with warp shuffles.  An index outside [0, vocab)
// is never dereferenced: its logit becomes NaN.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int WARPS = 4;

template <typename T>
__global__ void __launch_bounds__(WARPS * 32) k_rescore(const T* __restrict__ h, const T* __restrict__ W,
                                                        const int32_t* __restrict__ idx, int BK, int d,
                                                        int vocab, int K, float* __restrict__ logits) {
  constexpr int PER = Elem<T>::PER16;
  const int lane = threadIdx.x & 31;
  const int pair = blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (pair >= BK) return;
  const int b = pair / K;
  const int v = idx[pair];
  if (v < 0 || v >= vocab) {
    if (lane == 0) logits[pair] = __int_as_float(0x7FC00000);
    return;
  }
  const T* w = W + (size_t)v * d;
  const T* x = h + (size_t)b * d;
  float acc = 0.f;
#pragma unroll 4
  for (int c = lane * PER; c < d; c += 32 * PER) {
    const uint4 wa = ld_nc_v4(w + c);
    const uint4 xa = __ldg(reinterpret_cast<const uint4*>(x + c));
    float wf[PER], xf[PER];
    Elem<T>::unpack(wa, wf);
    Elem<T>::unpack(xa, xf);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) logits[pair] = acc;
}

// One warp per row: p = exp(z - max) / sum exp(z - max).  A NaN logit makes the sum, hence every
// probability of the row, NaN.
__global__ void k_softmax(const float* __restrict__ logits, int B, int K, float* __restrict__ probs) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= B) return;
  const float* z = logits + (size_t)row * K;
  float m = -INFINITY;
  for (int k = lane; k < K; k += 32) m = fmaxf(m, z[k]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float s = 0.f;
  for (int k = lane; k < K; k += 32) s += expf(z[k] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
  const float inv = 1.f / s;
  for (int k = lane; k < K; k += 32) probs[(size_t)row * K + k] = expf(z[k] - m) * inv;
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                int K, float* logits, float* probs) {
  const int BK = B * K;
  prof_before("rescore", c.stream);
  k_rescore<T><<<(BK + WARPS - 1) / WARPS, WARPS * 32, 0, c.stream>>>(
      static_cast<const T*>(h), static_cast<const T*>(W), idx, BK, d, vocab, K, logits);
  prof_after(c.stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || probs == nullptr) return e;
  prof_before("softmax", c.stream);
  k_softmax<<<(B + 3) / 4, 128, 0, c.stream>>>(logits, B, K, probs);
  prof_after(c.stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                           int vocab, int K, int dtype, float* logits, float* probs) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs);
  return run<float>(c, h, W, idx, B, d, vocab, K, logits, probs);
}

}  // namespace dh
