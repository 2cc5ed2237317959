// Stage 1a: the low-rank projection t = h U, rounded to the activation dtype.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the low-rank head factors the vocabulary head, and the factor applied first maps the hidden state
// h [B x d] to a rank-r activation t [B x r].  The pages do not state the precision of t; as an
// activation it is rounded to the activation dtype (bf16, round to nearest even) before the
// vocabulary-wide product.
//
// Split-d CUDA-core GEMV/GEMM: block (s, rb) accumulates rows [b0, b0+PB) of h against the d-slice s
// of U in fp32 and writes its partial sums; a second kernel adds the slices of each output with one
// warp in a fixed order (deterministic) and rounds.  U (1.3-5.2 MB) is read exactly once.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int PB = 8;           // rows of h per block
constexpr int TARGET_BLOCKS = 304;

template <typename T>
__global__ void __launch_bounds__(256) k_proj_partial(const T* __restrict__ h, const T* __restrict__ U,
                                                      int B, int d, int r, int nsplit,
                                                      float* __restrict__ partial) {
  extern __shared__ float sh_h[];  // [PB][chunk]
  const int s = blockIdx.x;
  const int b0 = blockIdx.y * PB;
  const int i0 = (int)((long long)d * s / nsplit);
  const int i1 = (int)((long long)d * (s + 1) / nsplit);
  const int chunk = i1 - i0;
  const int nb = min(PB, B - b0);
  for (int e = threadIdx.x; e < PB * chunk; e += blockDim.x) {
    const int b = e / chunk, i = e - b * chunk;
    sh_h[e] = (b < nb) ? Elem<T>::to_f(h[(size_t)(b0 + b) * d + i0 + i]) : 0.f;
  }
  __syncthreads();
  for (int jp = threadIdx.x; jp * 2 < r; jp += blockDim.x) {
    float acc[PB][2];
#pragma unroll
    for (int b = 0; b < PB; ++b) acc[b][0] = acc[b][1] = 0.f;
    const T* up = U + (size_t)i0 * r + 2 * jp;
#pragma unroll 4
    for (int i = 0; i < chunk; ++i) {
      const float u0 = Elem<T>::to_f(up[(size_t)i * r]);
      const float u1 = Elem<T>::to_f(up[(size_t)i * r + 1]);
#pragma unroll
      for (int b = 0; b < PB; ++b) {
        const float hb = sh_h[b * chunk + i];
        acc[b][0] = fmaf(hb, u0, acc[b][0]);
        acc[b][1] = fmaf(hb, u1, acc[b][1]);
      }
    }
#pragma unroll
    for (int b = 0; b < PB; ++b) {
      if (b < nb) {
        // partial layout [B*r][nsplit]: the reduce reads each output's slices contiguously
        float* o = partial + ((size_t)(b0 + b) * r + 2 * jp) * nsplit + s;
        o[0] = acc[b][0];
        o[nsplit] = acc[b][1];
      }
    }
  }
}

// One warp per output: lanes sum strided slices, then a fixed shuffle tree (deterministic).
template <typename T>
__global__ void k_proj_reduce(const float* __restrict__ partial, int BR, int nsplit, T* __restrict__ t) {
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (e >= BR) return;
  const float* p = partial + (size_t)e * nsplit;
  float acc = 0.f;
  for (int s = lane; s < nsplit; s += 32) acc += p[s];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if (lane == 0) t[e] = Elem<T>::from_f(acc);
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* U, int B, int d, int r, float* partial,
                int nsplit, void* t_out) {
  const int nbb = (B + PB - 1) / PB;
  const int chunk_max = (d + nsplit - 1) / nsplit;
  const size_t smem = (size_t)PB * chunk_max * sizeof(float);
  const int threads = min(256, max(32, (r / 2 + 31) / 32 * 32));
  static unsigned long long smem_done = 0;
  if (smem > 48 * 1024) {
    cudaError_t e = allow_max_smem(k_proj_partial<T>, c.device, &smem_done);
    if (e != cudaSuccess) return e;
  }
  prof_before("proj_partial", c.stream);
  k_proj_partial<T><<<dim3(nsplit, nbb), threads, smem, c.stream>>>(
      static_cast<const T*>(h), static_cast<const T*>(U), B, d, r, nsplit, partial);
  prof_after(c.stream);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int BR = B * r;
  prof_before("proj_reduce", c.stream);
  k_proj_reduce<T><<<(BR + 7) / 8, 256, 0, c.stream>>>(partial, BR, nsplit, static_cast<T*>(t_out));
  prof_after(c.stream);
  return cudaGetLastError();
}

}  // namespace

int proj_splits(const Ctx&, int B, int d, int) {
  const int nbb = (B + PB - 1) / PB;
  int ns = (TARGET_BLOCKS + nbb - 1) / nbb;
  ns = max(1, min(ns, d / 16));
  return ns;
}

cudaError_t launch_proj(const Ctx& c, const void* h, const void* U, int B, int d, int r, int dtype,
                        float* partial, int nsplit, void* t_out) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, U, B, d, r, partial, nsplit, t_out);
  return run<float>(c, h, U, B, d, r, partial, nsplit, t_out);
}

}  // namespace dh
