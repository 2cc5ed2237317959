// Exact top-K selection from group records (shared by the select kernel and the fused
// small-batch kernel).
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the K retrieved candidates of a row are its K best low-rank scores, in (score desc, id asc) order.
//
// select_row() runs on one block (SEL_THREADS threads) per row.  The pool P = the best two
// (score, id) pairs of every group of 64 ids.
//  1. tau = the K-th best pair of P (radix select on order-preserving keys, then on ids among
//     equal keys).  P holds real scores, so tau ranks at or below the true K-th best score.
//  2. Certificate: a group can hide a member at or above tau only if its third score >= tau.
//     Groups without that property contribute exactly their stored pairs.  The others ("refined"
//     groups) are re-scored exactly from t and V.
//  3. The K best of (stored pairs of the other groups) + (every member of the refined groups) is
//     the exact top-K.  If too many groups need refining, or P has fewer than K pairs, the block
//     re-scores the whole row instead (slow, exact, only reached by adversarial inputs).
//  4. The K winners are sorted by (score desc, id asc) with a bitonic network.
#pragma once

#include "dh_internal.cuh"

namespace dh {
namespace sel {

constexpr int SEL_THREADS = 512;
constexpr int RMAX = 32;                 // refined groups re-scored in shared memory
constexpr int CACHE_GROUPS = 3072;       // records cached in shared memory up to this many groups
constexpr int BITMAP_WORDS = (DH_MAX_VOCAB / GROUP + 31) / 32;

constexpr int HIST_BINS = 4096;  // widest radix digit (12 bits)

struct Shared {
  uint32_t hist[HIST_BINS];
  uint32_t wsum[SEL_THREADS / 32];
  uint32_t digit, run, bincount, total, cnt, nref;
  int32_t rg[RMAX];
  uint32_t bitmap[BITMAP_WORDS];
  float t[DH_MAX_RANK];
  float rs[RMAX * GROUP];
  uint32_t sk[DH_MAX_K];
  uint32_t si[DH_MAX_K];
};

// Histogram increment (shared-memory atomic; 12-bit digits spread the keys over enough bins that
// conflicts stay low).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin) { atomicAdd(&hist[bin], 1u); }

// Result of a radix selection of the k-th largest value x over the included entries.
//   total      number of included entries (if total < k nothing else is meaningful)
//   exact_ge   true: exactly k entries have x >= thr
//              false: thr is the k-th largest value, `above` entries have x > thr and the
//              k - above entries still to take have x == thr (more than that many do)
struct Kth {
  uint32_t thr, above, total;
  bool exact_ge;
};

// Finds, over the bins of sh.hist[0..nbins) read from the highest down, the bin where the running
// count reaches krem; sets sh.digit, sh.run (count above it), sh.bincount and, if set_total,
// sh.total.  Each of the nbins / 8 first threads owns 8 consecutive bins.
__device__ __forceinline__ void find_digit(Shared& sh, int nbins, uint32_t krem, bool set_total) {
  const int users = nbins / 8;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t c[8], sum = 0;
  if ((int)threadIdx.x < users) {
#pragma unroll
    for (int q = 0; q < 8; ++q) { c[q] = sh.hist[nbins - 1 - 8 * (int)threadIdx.x - q]; sum += c[q]; }
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  uint32_t before = 0;
  if (users > 32) {
    if (lane == 31) sh.wsum[warp] = incl;
    __syncthreads();
    for (int w = 0; w < warp; ++w) before += sh.wsum[w];
  }
  incl += before;
  const uint32_t excl = incl - sum;
  if ((int)threadIdx.x < users) {
    if (set_total && (int)threadIdx.x == users - 1) sh.total = incl;
    if (excl < krem && krem <= incl) {
      uint32_t run = excl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (run + c[q] >= krem) {
          sh.digit = (uint32_t)(nbins - 1 - 8 * (int)threadIdx.x - q); sh.run = run; sh.bincount = c[q];
          break;
        }
        run += c[q];
      }
    }
    if ((int)threadIdx.x == users - 1 && incl < krem) { sh.digit = 0; sh.run = incl; sh.bincount = 0; }
  }
}

// MSB-first radix select with digits of 12, 12 and 8 bits.  sel(key, id, x) decides inclusion and
// sets x.  Stops as soon as the bin holding the k-th value contains exactly the entries still
// needed.
template <class Enum, class Sel>
__device__ Kth radix_kth(Enum en, Sel sel, uint32_t k, Shared& sh) {
  constexpr int SHIFTS[3] = {20, 8, 0};
  constexpr int BITS[3] = {12, 12, 8};
  uint32_t prefix = 0, mask = 0, krem = k, above = 0;
  Kth res;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = SHIFTS[pass], nbins = 1 << BITS[pass];
    const uint32_t dmask = (uint32_t)nbins - 1u;
    for (int i = threadIdx.x; i < nbins; i += blockDim.x) sh.hist[i] = 0;
    __syncthreads();
    en([&](uint32_t key, uint32_t id) {
      uint32_t x;
      if (sel(key, id, x) && (x & mask) == prefix) hist_add(sh.hist, (x >> shift) & dmask);
    });
    __syncthreads();
    find_digit(sh, nbins, krem, pass == 0);
    __syncthreads();
    const uint32_t dg = sh.digit, run = sh.run, bc = sh.bincount, total = sh.total;
    __syncthreads();
    if (pass == 0 && total < k) {
      res.thr = 0; res.above = 0; res.total = total; res.exact_ge = false;
      return res;
    }
    prefix |= dg << shift;
    mask |= dmask << shift;
    krem -= run;
    above += run;
    if (bc == krem) {
      res.thr = prefix; res.above = above; res.total = total; res.exact_ge = true;
      return res;
    }
  }
  res.thr = prefix; res.above = above; res.total = sh.total; res.exact_ge = false;
  return res;
}

// (key, id) ranks before (key2, id2): larger key first, then smaller id.
__device__ __forceinline__ bool key_before(uint32_t ka, uint32_t ia, uint32_t kb, uint32_t ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Sorts sh.sk/sh.si[0..K) (padded to a power of two) into ranking order.  K <= 64: one warp with
// shuffles; larger K: a block-wide bitonic network in shared memory.
__device__ inline void sort_selected(Shared& sh, int K) {
  int P = 1;
  while (P < K) P <<= 1;
  for (int i = K + threadIdx.x; i < P; i += blockDim.x) { sh.sk[i] = 0u; sh.si[i] = 0xFFFFFFFFu; }
  __syncthreads();
  if (P <= 64) {
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      uint32_t k0 = 0, i0 = 0xFFFFFFFFu, k1 = 0, i1 = 0xFFFFFFFFu;
      if (2 * lane < P) { k0 = sh.sk[2 * lane]; i0 = sh.si[2 * lane]; }
      if (2 * lane + 1 < P) { k1 = sh.sk[2 * lane + 1]; i1 = sh.si[2 * lane + 1]; }
      for (int size = 2; size <= 64; size <<= 1) {
        for (int j = size >> 1; j > 0; j >>= 1) {
          if (j == 1) {
            const int p0 = 2 * lane;
            const bool up = (p0 & size) == 0;
            const bool b_first = key_before(k1, i1, k0, i0);
            if (b_first == up) {
              uint32_t tk = k0, ti = i0;
              k0 = k1; i0 = i1; k1 = tk; i1 = ti;
            }
          } else {
            const int src = lane ^ (j >> 1);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              uint32_t& mk = e ? k1 : k0;
              uint32_t& mi = e ? i1 : i0;
              const uint32_t ok_ = __shfl_sync(0xFFFFFFFFu, mk, src);
              const uint32_t oi = __shfl_sync(0xFFFFFFFFu, mi, src);
              const int p = 2 * lane + e;
              const bool up = (p & size) == 0;
              const bool lower = (p & j) == 0;
              const bool mine_first = key_before(mk, mi, ok_, oi);
              const bool keep_first = (up == lower);
              if (keep_first != mine_first) { mk = ok_; mi = oi; }
            }
          }
        }
      }
      if (2 * lane < P) { sh.sk[2 * lane] = k0; sh.si[2 * lane] = i0; }
      if (2 * lane + 1 < P) { sh.sk[2 * lane + 1] = k1; sh.si[2 * lane + 1] = i1; }
    }
    __syncthreads();
    return;
  }
  for (int size = 2; size <= P; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < P / 2; i += blockDim.x) {
        const int a0 = 2 * i - (i & (stride - 1));
        const int b0 = a0 + stride;
        const bool up = (a0 & size) == 0;
        const uint32_t ka = sh.sk[a0], kb = sh.sk[b0], ia = sh.si[a0], ib = sh.si[b0];
        if (key_before(kb, ib, ka, ia) == up) { sh.sk[a0] = kb; sh.sk[b0] = ka; sh.si[a0] = ib; sh.si[b0] = ia; }
      }
    }
  }
  __syncthreads();
}

// Selects the K best entries (score key desc, id asc) of en, sorts them and writes the row; the
// K-th best key goes to *thr_out.  Returns false (and writes nothing) if en holds fewer than K.
template <class Enum>
__device__ bool select_sort_write(Enum en, int K, Shared& sh, int32_t* idx_out, float* score_out,
                                  uint32_t* thr_out) {
  const Kth a = radix_kth(en, [](uint32_t key, uint32_t, uint32_t& x) { x = key; return true; },
                          (uint32_t)K, sh);
  if (a.total < (uint32_t)K) return false;
  const uint32_t T = a.thr;
  uint32_t idthr = 0;  // among key == T, take ~id >= idthr (the lowest ids)
  if (!a.exact_ge) {
    const Kth b = radix_kth(
        en, [T](uint32_t key, uint32_t id, uint32_t& x) { x = ~id; return key == T; }, (uint32_t)K - a.above,
        sh);
    idthr = b.thr;
  }
  const bool exact = a.exact_ge;
  if (threadIdx.x == 0) sh.cnt = 0;
  __syncthreads();
  en([&](uint32_t key, uint32_t id) {
    if (exact ? key >= T : (key > T || (key == T && ~id >= idthr))) {
      const uint32_t pos = atomicAdd(&sh.cnt, 1u);
      if (pos < DH_MAX_K) { sh.sk[pos] = key; sh.si[pos] = id; }
    }
  });
  __syncthreads();
  sort_selected(sh, K);
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    idx_out[k] = (int32_t)sh.si[k];
    score_out[k] = fkey_inv(sh.sk[k]);
  }
  if (thr_out) *thr_out = sh.sk[K - 1];  // the exact K-th best key of en
  __syncthreads();
  return true;
}

template <typename T>
__device__ __forceinline__ float score_col(const float* t, const T* V, int r, int vocab, int c) {
  float acc = 0.f;
#pragma unroll 16
  for (int j = 0; j < r; ++j) acc = fmaf(t[j], Elem<T>::to_f(V[(size_t)j * vocab + c]), acc);
  return acc;
}

// Exact scores of the 64 ids of group g (ids >= vocab give -inf) into out[0..64).  The block's
// warps split the r rows of V: warp w covers rows [w*rw, (w+1)*rw) with all its loads in flight
// (lane i reads the two ids 2i, 2i+1), then the per-warp partial sums are added in warp order
// (a fixed order, so the result is deterministic).  scratch: SEL_THREADS / 32 * 64 floats.
template <typename T>
__device__ void score_group(const float* t, const T* __restrict__ V, int r, int vocab, int g, float* out,
                            float* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int rw = (r + nw - 1) / nw;
  const int j0 = warp * rw, j1 = min(r, j0 + rw);
  const int c = g * GROUP + 2 * lane;
  float a0 = 0.f, a1 = 0.f;
  constexpr int BATCH = 16;
  for (int jb = j0; jb < j1; jb += BATCH) {
    float v0[BATCH], v1[BATCH];
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int j = jb + q;
      v0[q] = (j < j1 && c < vocab) ? Elem<T>::to_f(V[(size_t)j * vocab + c]) : 0.f;
      v1[q] = (j < j1 && c + 1 < vocab) ? Elem<T>::to_f(V[(size_t)j * vocab + c + 1]) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < BATCH; ++q) {
      const int j = jb + q;
      const float tj = (j < j1) ? t[j] : 0.f;
      a0 = fmaf(tj, v0[q], a0);
      a1 = fmaf(tj, v1[q], a1);
    }
  }
  scratch[warp * 64 + 2 * lane] = a0;
  scratch[warp * 64 + 2 * lane + 1] = a1;
  __syncthreads();
  if (threadIdx.x < 64) {
    float s = 0.f;
    for (int w = 0; w < nw; ++w) s += scratch[w * 64 + threadIdx.x];
    out[threadIdx.x] = (g * GROUP + (int)threadIdx.x < vocab) ? s : -INFINITY;
  }
  __syncthreads();
}



// Shared memory select_row needs: the Shared block plus, when n_groups <= CACHE_GROUPS, a copy of
// the row's records.
__host__ __device__ constexpr size_t select_smem_bytes(int n_groups) {
  return align_up(sizeof(Shared), 16) + (n_groups <= CACHE_GROUPS ? (size_t)n_groups * sizeof(GroupRec) : 0);
}

// Exact top-K of one row.  smem: select_smem_bytes(n_groups) bytes, 16-byte aligned.
// t_row: the row's projection (r values of the activation dtype); rrow: its n_groups records.
template <typename T>
__device__ void select_row(unsigned char* smem, const GroupRec* __restrict__ rrow, const T* __restrict__ t_row,
                           const T* __restrict__ V, int r, int vocab, int K, int32_t* __restrict__ idx_out,
                           float* __restrict__ score_out) {
  Shared& sh = *reinterpret_cast<Shared*>(smem);
  GroupRec* cache = reinterpret_cast<GroupRec*>(smem + align_up(sizeof(Shared), 16));
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const bool cached = n_groups <= CACHE_GROUPS;

  for (int g = threadIdx.x; g < (int)BITMAP_WORDS; g += blockDim.x) sh.bitmap[g] = 0u;
  for (int j = threadIdx.x; j < r; j += blockDim.x) sh.t[j] = Elem<T>::to_f(t_row[j]);
  if (cached) {
    constexpr int PER_THREAD = (CACHE_GROUPS + SEL_THREADS - 1) / SEL_THREADS;
    GroupRec tmp[PER_THREAD];
#pragma unroll
    for (int q = 0; q < PER_THREAD; ++q) {
      const int g = threadIdx.x + q * SEL_THREADS;
      if (g < n_groups) tmp[q] = rrow[g];
    }
#pragma unroll
    for (int q = 0; q < PER_THREAD; ++q) {
      const int g = threadIdx.x + q * SEL_THREADS;
      if (g < n_groups) cache[g] = tmp[q];
    }
  }
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

  uint32_t tau = 0;
  if (select_sort_write(pool, K, sh, idx_out, score_out, &tau)) {
    // Certificate: groups that may hide a member ranking at or above tau (third score >= tau).
    // tau is at or below the true K-th score, so without such groups the pool's top K is exact.
    for (int g = threadIdx.x; g < n_groups; g += blockDim.x) {
      if (fkey(src[g].m3) >= tau) {
        const uint32_t pos = atomicAdd(&sh.nref, 1u);
        if (pos < RMAX) sh.rg[pos] = g;
        atomicOr(&sh.bitmap[g >> 5], 1u << (g & 31));
      }
    }
    __syncthreads();
    const int nref = (int)sh.nref;
    if (nref == 0) return;
    if (nref <= RMAX) {
      for (int i = 0; i < nref; ++i)
        score_group(sh.t, V, r, vocab, sh.rg[i], sh.rs + i * GROUP, reinterpret_cast<float*>(sh.hist));
      auto refined = [&](auto f) {
        pool(f);  // skips the refined groups (bitmap)
        for (int e = threadIdx.x; e < nref * GROUP; e += blockDim.x) {
          const int c = sh.rg[e / GROUP] * GROUP + (e % GROUP);
          if (c < vocab) f(fkey(sh.rs[e]), (uint32_t)c);
        }
      };
      select_sort_write(refined, K, sh, idx_out, score_out, nullptr);
      return;
    }
  }
  // exact fallback: every id of the row, re-scored on each pass
  auto all = [&](auto f) {
    for (int c = threadIdx.x; c < vocab; c += blockDim.x) f(fkey(score_col(sh.t, V, r, vocab, c)), (uint32_t)c);
  };
  select_sort_write(all, K, sh, idx_out, score_out, nullptr);
}

}  // namespace sel
}  // namespace dh
