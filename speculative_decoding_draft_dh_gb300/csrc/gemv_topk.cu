// Stage 1b (CUDA-core path): low-rank scores s = t V over the whole vocabulary, reduced on the fly
// to per-group summaries so that the B x vocab score matrix never reaches memory.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the low-rank head scores the full vocabulary only to retrieve candidates.
//
// Each warp owns a tile of 32 x 16 bytes of vocabulary columns (256 bf16 / 128 fp32 ids) and
// streams the r rows of V under it with 16-byte loads, keeping BB rows of scores in registers.
// The scores of each group of 64 ids are folded into a GroupRec (best two (score, id) pairs and the
// third score) by a shuffle butterfly across the lanes that share the group.  The selection kernel
// picks the K candidates from these records and re-scores the rare groups whose third score could
// still reach the candidate set.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int WARPS = 4;
constexpr int BB = 8;  // score rows kept in registers

template <typename T>
__global__ void __launch_bounds__(WARPS * 32) k_scores_summary(const T* __restrict__ t,
                                                               const T* __restrict__ V, int B, int r,
                                                               int vocab, int n_groups,
                                                               GroupRec* __restrict__ recs) {
  constexpr int PER = Elem<T>::PER16;
  constexpr int TILE = 32 * PER;
  constexpr int LPG = GROUP / PER;  // lanes per group
  extern __shared__ float st[];     // [BB][r]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_tiles = (vocab + TILE - 1) / TILE;
  for (int b0 = 0; b0 < B; b0 += BB) {
    const int nb = min(BB, B - b0);
    __syncthreads();
    for (int e = threadIdx.x; e < BB * r; e += blockDim.x) {
      const int b = e / r;
      st[e] = (b < nb) ? Elem<T>::to_f(t[(size_t)(b0 + b) * r + (e - b * r)]) : 0.f;
    }
    __syncthreads();
    for (int tile = blockIdx.x * WARPS + warp; tile < n_tiles; tile += gridDim.x * WARPS) {
      const int c0 = tile * TILE + lane * PER;
      const bool valid = c0 < vocab;  // vocab is a multiple of PER
      float acc[BB][PER];
#pragma unroll
      for (int b = 0; b < BB; ++b)
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[b][e] = 0.f;
      const T* vp = V + (valid ? c0 : 0);
      for (int j = 0; j < r; j += PER) {  // r is a multiple of PER
        uint4 raw[PER];
#pragma unroll
        for (int q = 0; q < PER; ++q)
          raw[q] = valid ? ld_nc_v4(vp + (size_t)(j + q) * vocab) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int q = 0; q < PER; ++q) {
          float x[PER];
          Elem<T>::unpack(raw[q], x);
#pragma unroll
          for (int b = 0; b < BB; ++b) {
            const float tb = st[b * r + j + q];
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[b][e] = fmaf(tb, x[e], acc[b][e]);
          }
        }
      }
#pragma unroll
      for (int b = 0; b < BB; ++b) {
        if (b < nb) {
          Top2 s;
          s.init();
          if (valid) {
#pragma unroll
            for (int e = 0; e < PER; ++e) s.push(acc[b][e], (uint32_t)(c0 + e));
          }
#pragma unroll
          for (int x = 1; x < LPG; x <<= 1) s.merge_shfl(0xFFFFFFFFu, x);
          const int g = c0 / GROUP;
          if ((lane % LPG) == 0 && g < n_groups)
            recs[(size_t)(b0 + b) * n_groups + g] = s.record((uint32_t)g * GROUP);
        }
      }
    }
  }
}

template <typename T>
cudaError_t run(const Ctx& c, const void* t, const void* V, int B, int r, int vocab, GroupRec* recs) {
  constexpr int TILE = 32 * Elem<T>::PER16;
  const int n_tiles = (vocab + TILE - 1) / TILE;
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  int blocks = (n_tiles + WARPS - 1) / WARPS;
  blocks = min(blocks, c.num_sms * 4);
  const size_t smem = (size_t)BB * r * sizeof(float);
  static unsigned long long smem_done = 0;
  if (smem > 48 * 1024) {
    cudaError_t e = allow_max_smem(k_scores_summary<T>, c.device, &smem_done);
    if (e != cudaSuccess) return e;
  }
  prof_before("scores_summary", c.stream);
  k_scores_summary<T><<<blocks, WARPS * 32, smem, c.stream>>>(
      static_cast<const T*>(t), static_cast<const T*>(V), B, r, vocab, n_groups, recs);
  prof_after(c.stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scores_summary(const Ctx& c, const void* t, const void* V, int B, int r, int vocab,
                                  int dtype, GroupRec* recs) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, t, V, B, r, vocab, recs);
  return run<float>(c, t, V, B, r, vocab, recs);
}

}  // namespace dh
