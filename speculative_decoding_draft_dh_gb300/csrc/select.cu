// Stage 1c: exact top-K per row from the group records.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the K retrieved candidates of a row are its K best low-rank scores, in (score desc, id asc) order.
//
// One block per row.  The pool P = the best two (score, id) pairs of every group of 64 ids.
//  1. tau = the K-th best pair of P (radix select on order-preserving keys, then on ids among
//     equal keys).  P holds real scores, so tau ranks at or below the true K-th best score.
//  2. Certificate: a group can hide a member at or above tau only if its third score >= tau.
//     Groups without that property contribute exactly their stored pairs.  The others ("refined"
//     groups) are re-scored exactly from t and V.
//  3. The K best of (stored pairs of the other groups) + (every member of the refined groups) is
//     the exact top-K.  If too many groups need refining, or P has fewer than K pairs, the block
//     re-scores the whole row instead (slow, exact, only reached by adversarial inputs).
//  4. The K winners are sorted by (score desc, id asc) with a bitonic network.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int THREADS = 512;
constexpr int RMAX = 32;                 // refined groups re-scored in shared memory
constexpr int CACHE_GROUPS = 3072;       // records cached in shared memory up to this many groups
constexpr int BITMAP_WORDS = (DH_MAX_VOCAB / GROUP + 31) / 32;

struct Shared {
  uint32_t hist[256];
  uint32_t digit, above, total, cnt, nref;
  int32_t rg[RMAX];
  uint32_t bitmap[BITMAP_WORDS];
  float t[DH_MAX_RANK];
  float rs[RMAX * GROUP];
  uint32_t sk[DH_MAX_K];
  uint32_t si[DH_MAX_K];
};

// k-th largest value of sel(key, id) over the entries for which sel returns true.
// Returns it and sets *n_above to the number of included entries strictly above it.
// Requires at least k included entries (sh.total reports how many there were).
template <class Enum, class Sel>
__device__ uint32_t radix_kth(Enum en, Sel sel, uint32_t k, uint32_t* n_above, Shared& sh) {
  uint32_t prefix = 0, mask = 0, krem = k, above = 0;
  const int lane = threadIdx.x & 31;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    en([&](uint32_t key, uint32_t id) {
      uint32_t x;
      if (sel(key, id, x) && (x & mask) == prefix) atomicAdd(&sh.hist[(x >> shift) & 255u], 1u);
    });
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t c[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { c[q] = sh.hist[255 - 8 * lane - q]; sum += c[q]; }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      if (shift == 24 && lane == 31) sh.total = incl;
      if (excl < krem && krem <= incl) {
        uint32_t run = excl;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run + c[q] >= krem) { sh.digit = 255u - 8u * lane - q; sh.above = run; break; }
          run += c[q];
        }
      }
      if (lane == 31 && incl < krem) { sh.digit = 0; sh.above = incl; }
    }
    __syncthreads();
    const uint32_t dg = sh.digit, ab = sh.above;
    prefix |= dg << shift;
    mask |= 0xFFu << shift;
    krem -= ab;
    above += ab;
    __syncthreads();
  }
  *n_above = above;
  return prefix;
}

// Selects the k best entries (score key desc, id asc) of en, sorts them and writes the row.
template <class Enum>
__device__ void select_sort_write(Enum en, int K, Shared& sh, int32_t* idx_out, float* score_out,
                                  uint32_t* T_out, uint32_t* idthr_out) {
  uint32_t above;
  const uint32_t T = radix_kth(en, [](uint32_t key, uint32_t, uint32_t& x) { x = key; return true; },
                               (uint32_t)K, &above, sh);
  const uint32_t need = (uint32_t)K - above;  // entries with key == T to take, lowest ids first
  uint32_t above2;
  const uint32_t nid = radix_kth(
      en, [T](uint32_t key, uint32_t id, uint32_t& x) { x = ~id; return key == T; }, need, &above2, sh);
  const uint32_t idthr = ~nid;
  if (T_out) { *T_out = T; *idthr_out = idthr; }
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  en([&](uint32_t key, uint32_t id) {
    if (key > T || (key == T && id <= idthr)) {
      const uint32_t pos = atomicAdd(&sh.cnt, 1u);
      if (pos < DH_MAX_K) { sh.sk[pos] = key; sh.si[pos] = id; }
    }
  });
  __syncthreads();
  int P = 1;
  while (P < K) P <<= 1;
  for (int i = K + threadIdx.x; i < P; i += blockDim.x) { sh.sk[i] = 0u; sh.si[i] = 0xFFFFFFFFu; }
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
        const int a = 2 * i - (i & (stride - 1));
        const int b = a + stride;
        const bool up = (a & size) == 0;
        const uint32_t ka = sh.sk[a], kb = sh.sk[b], ia = sh.si[a], ib = sh.si[b];
        const bool b_first = kb > ka || (kb == ka && ib < ia);
        if (b_first == up) { sh.sk[a] = kb; sh.sk[b] = ka; sh.si[a] = ib; sh.si[b] = ia; }
      }
    }
  }
  __syncthreads();
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    idx_out[k] = (int32_t)sh.si[k];
    score_out[k] = fkey_inv(sh.sk[k]);
  }
  __syncthreads();
}

template <typename T>
__device__ __forceinline__ float score_col(const float* t, const T* V, int r, int vocab, int c) {
  float acc = 0.f;
  for (int j = 0; j < r; ++j) acc = fmaf(t[j], Elem<T>::to_f(V[(size_t)j * vocab + c]), acc);
  return acc;
}

template <typename T>
__global__ void __launch_bounds__(THREADS) k_select(const GroupRec* __restrict__ recs, const T* __restrict__ t,
                                                    const T* __restrict__ V, int r, int vocab, int K,
                                                    int32_t* __restrict__ idx_out,
                                                    float* __restrict__ score_out) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Shared& sh = *reinterpret_cast<Shared*>(smem_raw);
  GroupRec* cache = reinterpret_cast<GroupRec*>(smem_raw + align_up(sizeof(Shared), 16));
  const int row = blockIdx.x;
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const GroupRec* rrow = recs + (size_t)row * n_groups;
  const bool cached = n_groups <= CACHE_GROUPS;
  idx_out += (size_t)row * K;
  score_out += (size_t)row * K;

  for (int g = threadIdx.x; g < (int)BITMAP_WORDS; g += blockDim.x) sh.bitmap[g] = 0u;
  for (int j = threadIdx.x; j < r; j += blockDim.x) sh.t[j] = Elem<T>::to_f(t[(size_t)row * r + j]);
  if (cached)
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) cache[g] = rrow[g];
  if (threadIdx.x == 0) sh.nref = 0;
  __syncthreads();
  const GroupRec* src = cached ? cache : rrow;

  auto pool = [&](auto f) {
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      if ((sh.bitmap[g >> 5] >> (g & 31)) & 1u) continue;
      const GroupRec rc = src[g];
      const uint32_t o1 = rc.offs & 0xFFu, o2 = (rc.offs >> 8) & 0xFFu;
      if (o1 != NO_OFFSET) f(fkey(rc.m1), (uint32_t)g * GROUP + o1);
      if (o2 != NO_OFFSET) f(fkey(rc.m2), (uint32_t)g * GROUP + o2);
    }
  };

  // pool size: at least K pairs are needed for tau to exist
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  {
    uint32_t mine = 0;
    pool([&](uint32_t, uint32_t) { ++mine; });
    atomicAdd(&sh.cnt, mine);
  }
  __syncthreads();
  bool full = sh.cnt < (uint32_t)K;
  __syncthreads();

  if (!full) {
    uint32_t above;
    const uint32_t tau = radix_kth(pool, [](uint32_t key, uint32_t, uint32_t& x) { x = key; return true; },
                                   (uint32_t)K, &above, sh);
    // groups that may hide a member at or above tau
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      if (fkey(src[g].m3) >= tau) {
        const uint32_t pos = atomicAdd(&sh.nref, 1u);
        if (pos < RMAX) sh.rg[pos] = g;
        atomicOr(&sh.bitmap[g >> 5], 1u << (g & 31));
      }
    }
    __syncthreads();
    const int nref = (int)sh.nref;
    if (nref == 0) {
      select_sort_write(pool, K, sh, idx_out, score_out, nullptr, nullptr);
      return;
    }
    if (nref <= RMAX) {
      for (int e = threadIdx.x; e < nref * GROUP; e += blockDim.x) {
        const int c = sh.rg[e / GROUP] * GROUP + (e % GROUP);
        sh.rs[e] = (c < vocab) ? score_col(sh.t, V, r, vocab, c) : -INFINITY;
      }
      __syncthreads();
      auto refined = [&](auto f) {
        pool(f);
        for (int e = threadIdx.x; e < nref * GROUP; e += blockDim.x) {
          const int c = sh.rg[e / GROUP] * GROUP + (e % GROUP);
          if (c < vocab) f(fkey(sh.rs[e]), (uint32_t)c);
        }
      };
      select_sort_write(refined, K, sh, idx_out, score_out, nullptr, nullptr);
      return;
    }
    full = true;
  }
  // exact fallback: every id of the row, re-scored on each pass
  auto all = [&](auto f) {
    for (int c = threadIdx.x; c < vocab; c += blockDim.x) f(fkey(score_col(sh.t, V, r, vocab, c)), (uint32_t)c);
  };
  select_sort_write(all, K, sh, idx_out, score_out, nullptr, nullptr);
}

template <typename T>
cudaError_t run(const Ctx& c, const GroupRec* recs, const void* t, const void* V, int B, int r, int vocab,
                int K, int32_t* idx_out, float* score_out) {
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  size_t smem = align_up(sizeof(Shared), 16);
  if (n_groups <= CACHE_GROUPS) smem += (size_t)n_groups * sizeof(GroupRec);
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_select<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  prof_before("select", c.stream);
  k_select<T><<<B, THREADS, smem, c.stream>>>(recs, static_cast<const T*>(t), static_cast<const T*>(V), r,
                                               vocab, K, idx_out, score_out);
  prof_after(c.stream);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_select(const Ctx& c, const GroupRec* recs, const void* t, const void* V, int B, int r,
                          int vocab, int K, int dtype, int32_t* idx_out, float* score_out) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, recs, t, V, B, r, vocab, K, idx_out, score_out);
  return run<float>(c, recs, t, V, B, r, vocab, K, idx_out, score_out);
}

}  // namespace dh
