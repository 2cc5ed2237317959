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

#include <cstddef>

#include "dh_internal.cuh"

namespace dh {
namespace sel {

constexpr int SEL_THREADS = 512;
constexpr int RMAX = 32;                 // refined groups re-scored in shared memory
constexpr int CACHE_GROUPS = 3072;       // records cached in shared memory up to this many groups
constexpr int BITMAP_WORDS = (DH_MAX_VOCAB / GROUP + 31) / 32;

constexpr int HIST_BINS = 4096;  // widest radix digit (12 bits)

struct Shared {
  alignas(16) uint32_t hist[HIST_BINS];  // also the fast path's packed 64-bit entries
  uint32_t wsum[SEL_THREADS / 32];
  uint32_t wmin[SEL_THREADS / 32], wmax[SEL_THREADS / 32];
  uint32_t digit, run, bincount, total, cnt, nref, tau_key;
  int32_t rg[RMAX];
  uint32_t bitmap[BITMAP_WORDS];
  float t[DH_MAX_RANK];
  alignas(16) float rs[RMAX * GROUP];  // also the fast path's packed boundary entries
  alignas(16) uint32_t sk[DH_MAX_K];
  uint32_t si[DH_MAX_K];
};

static_assert(offsetof(Shared, rs) % 8 == 0 && offsetof(Shared, hist) % 8 == 0, "64-bit views need 8-byte alignment");

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
// sh.total.  Each of the first nbins / per threads owns per consecutive bins (per = 8, or more when
// the block has fewer than nbins / 8 threads).
__device__ __forceinline__ void find_digit(Shared& sh, int nbins, uint32_t krem, bool set_total) {
  const int per = max(8, nbins / (int)blockDim.x);
  const int users = nbins / per;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int top = nbins - 1 - per * (int)threadIdx.x;  // this thread's highest bin
  uint32_t sum = 0;
  if ((int)threadIdx.x < users)
    for (int q = 0; q < per; ++q) sum += sh.hist[top - q];
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
      for (int q = 0; q < per; ++q) {
        const uint32_t cq = sh.hist[top - q];
        if (run + cq >= krem) {
          sh.digit = (uint32_t)(top - q); sh.run = run; sh.bincount = cq;
          break;
        }
        run += cq;
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

// Appends for the lanes whose pred is set: returns each such lane's position in the list whose
// length is *counter (one shared atomic per warp).  Called by all 32 lanes of the warp.
__device__ __forceinline__ uint32_t warp_append(bool pred, uint32_t* counter) {
  const int lane = threadIdx.x & 31;
  const uint32_t b = __ballot_sync(0xFFFFFFFFu, pred);
  uint32_t base = 0;
  if (lane == 0 && b) base = atomicAdd(counter, (uint32_t)__popc(b));
  base = __shfl_sync(0xFFFFFFFFu, base, 0);
  return base + (uint32_t)__popc(b & ((1u << lane) - 1u));
}

// Rank of entry i among sp[0..K) by counting (the number of larger packed values), with P threads
// per entry: thread h of the entry counts over j = h, h + P, h + 2P, ... (the P threads of an
// entry read consecutive words, so their loads do not collide in a shared-memory bank), and the
// P partial counts are added with shuffles.  Every thread of the warp takes part.
__device__ __forceinline__ int rank_by_count(const unsigned long long* sp, int K, int P, int i, int h,
                                             unsigned long long* pi_out) {
  int rank = 0;
  unsigned long long pi = 0;
  if (i < K) {
    pi = sp[i];
    if (K <= 8 * P) {  // at most 8 steps: a plain loop measured faster than an unrolled one
      for (int j = h; j < K; j += P) rank += sp[j] > pi ? 1 : 0;
    } else {
#pragma unroll 8
      for (int j = h; j < K; j += P) rank += sp[j] > pi ? 1 : 0;
    }
  }
  for (int o = 1; o < P; o <<= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
  *pi_out = pi;
  return rank;
}

// Sorts sh.sk/sh.si[0..K) into ranking order by counting: with (key, id) packed as
// key << 32 | ~id (ranking order = descending packed value; ids are unique, so the packed values
// are distinct), an entry's rank is the number of entries with a larger packed value.  P threads
// share an entry (P = the largest power of two <= 32 with K * P <= blockDim.x).  Uses sh.hist as
// scratch.
__device__ inline void sort_selected(Shared& sh, int K) {
  unsigned long long* sp = reinterpret_cast<unsigned long long*>(sh.hist);  // K <= DH_MAX_K entries
  for (int i = threadIdx.x; i < K; i += blockDim.x)
    sp[i] = ((unsigned long long)sh.sk[i] << 32) | (unsigned long long)(~sh.si[i]);
  __syncthreads();
  int P = 1;
  while (P < 32 && K * (2 * P) <= (int)blockDim.x) P <<= 1;
  for (int base = 0; base < K * P; base += blockDim.x) {
    const int t = base + (int)threadIdx.x;
    const int i = t / P, h = t % P;
    unsigned long long pi;
    const int rank = rank_by_count(sp, K, P, i, h, &pi);
    if (i < K && h == 0) {
      sh.sk[rank] = (uint32_t)(pi >> 32);
      sh.si[rank] = ~(uint32_t)pi;
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

// Fast path for a pool that fits in registers (at most FP_ENT entries per thread).  MSB-first
// radix select over y = key - (smallest key of the pool), 256 bins per level: level 0 takes the 8
// bits of y below the top bit of the pool's key range (so the bins span the pool's own range; the
// pool holds each group's best two scores, and its keys crowd into a narrow band of the float
// range), each further level the next 8 bits.  The descent stops at the first level whose boundary
// bin (the bin holding the K-th entry) has at most FP_RANK entries.  Entries above the boundary
// bin are selected, the boundary bin's entries ranked by counting and the best K - above of them
// taken; the K winners are then ranked by counting and written out in order.  Entries are packed
// as key << 32 | ~id, so ranking order is descending packed value.  With 256 bins one warp scans a
// level's histogram, and a level costs two block barriers.  Returns false (nothing written) when
// the pool has fewer than K entries or the boundary bin still holds more than FP_BOUND entries
// after the last level (many equal keys); the caller then runs the generic radix selection.  On
// success the K selected entries are also left in sh.sk/sh.si, in ranking order.
constexpr int FP_ENT = 12;
constexpr int FP_BINS = 256;
constexpr int FP_BITS = 8;
constexpr int FP_BOUND = 512;  // largest boundary bin ranked by counting (after the last level)
constexpr int FP_RANK = 64;    // a level whose boundary bin holds at most this many ends the descent

__device__ __forceinline__ unsigned long long pack_entry(uint32_t key, uint32_t id) {
  return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}

template <class Load>
__device__ bool fast_select(Load load, int n_entries_max, int K, Shared& sh, int32_t* idx_out, float* score_out,
                            uint32_t* thr_out) {
  if (n_entries_max > FP_ENT * (int)blockDim.x) return false;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  uint32_t* hist = sh.hist;
  uint32_t key[FP_ENT], id[FP_ENT];
  load(key, id);  // key 0 = no entry
  for (int i = threadIdx.x; i < FP_BINS; i += blockDim.x) hist[i] = 0;  // visible after the next barrier
  // the pool's key range
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < FP_ENT; ++q)
    if (key[q]) { kmin = min(kmin, key[q]); kmax = max(kmax, key[q]); }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) { sh.wmin[warp] = kmin; sh.wmax[warp] = kmax; }
  __syncthreads();
  for (int w = 0; w < nw; ++w) { kmin = min(kmin, sh.wmin[w]); kmax = max(kmax, sh.wmax[w]); }
  if (kmax == 0u) return false;  // empty pool (uniform: every thread read the same values)
#pragma unroll
  for (int q = 0; q < FP_ENT; ++q) key[q] = key[q] ? key[q] - kmin + 1u : 0u;  // y + 1 (0 = no entry)
  const uint32_t range = kmax - kmin + 1u;
  int shift = range >= 0x80000000u ? 32 - FP_BITS : max(0, (32 - __clz((int)range)) - FP_BITS);
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K, above = 0, bc = 0;
  const uint32_t dmask = (uint32_t)FP_BINS - 1u;
  bool first = true;
#pragma unroll 1
  for (;;) {
#pragma unroll
    for (int q = 0; q < FP_ENT; ++q)
      if (key[q] && (key[q] & mask) == prefix) atomicAdd(&hist[(key[q] >> shift) & dmask], 1u);
    __syncthreads();
    find_digit(sh, FP_BINS, krem, first);  // 256 bins: one warp, no barrier inside
    __syncthreads();
    const uint32_t D = sh.digit, run = sh.run, total = sh.total;
    bc = sh.bincount;
    if (first && total < (uint32_t)K) return false;
    first = false;
    prefix |= D << shift;
    mask |= dmask << shift;
    krem -= run;
    above += run;
    if (bc <= (uint32_t)FP_RANK || shift == 0) break;  // ranking the boundary bin by counting is cheap
    shift = max(0, shift - FP_BITS);
    for (int i = threadIdx.x; i < FP_BINS; i += blockDim.x) hist[i] = 0;  // the scan is done with it
    __syncthreads();
  }
  if (bc > (uint32_t)FP_BOUND) return false;
  // compaction: block scan of the per-thread counts (above the bin in the low 16 bits, in the
  // boundary bin in the high 16 bits), then every thread writes its entries at its offsets
  unsigned long long* sp = reinterpret_cast<unsigned long long*>(sh.hist);  // the K winners
  unsigned long long* bp = reinterpret_cast<unsigned long long*>(sh.rs);    // the boundary bin
  uint32_t nu = 0, nb = 0;
#pragma unroll
  for (int q = 0; q < FP_ENT; ++q) {
    const uint32_t mk = key[q] & mask;
    nu += (key[q] && mk > prefix) ? 1u : 0u;
    nb += (key[q] && mk == prefix) ? 1u : 0u;
  }
  const uint32_t mine = nu | (nb << 16);
  uint32_t incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  uint32_t before = 0;
  for (int w = 0; w < warp; ++w) before += sh.wsum[w];
  const uint32_t excl = before + incl - mine;
  uint32_t pu = excl & 0xFFFFu, pb = excl >> 16;
#pragma unroll
  for (int q = 0; q < FP_ENT; ++q) {
    const uint32_t mk = key[q] & mask;
    const uint32_t k0 = key[q] - 1u + kmin;  // the original key
    if (key[q] && mk > prefix) sp[pu++] = pack_entry(k0, id[q]);
    else if (key[q] && mk == prefix) bp[pb++] = pack_entry(k0, id[q]);
  }
  __syncthreads();
  // the boundary entries ranking below the first K - above of the bin are dropped; the others go
  // after the entries above the bin (their rank among the bin's entries is unique)
  const int need = K - (int)above;
  {
    int P = 1;
    while (P < 32 && (int)bc * (2 * P) <= (int)blockDim.x) P <<= 1;
    for (int base = 0; base < (int)bc * P; base += blockDim.x) {
      const int t = base + (int)threadIdx.x;
      const int i = t / P, h = t % P;
      unsigned long long pi;
      const int rank = rank_by_count(bp, (int)bc, P, i, h, &pi);
      if (i < (int)bc && h == 0 && rank < need) sp[above + rank] = pi;
    }
  }
  __syncthreads();
  // rank the K winners by counting (P threads per entry, partial counts added with shuffles) and
  // write them out in order
  int P = 1;
  while (P < 32 && K * (2 * P) <= (int)blockDim.x) P <<= 1;
  for (int base = 0; base < K * P; base += blockDim.x) {
    const int t = base + (int)threadIdx.x;
    const int i = t / P, h = t % P;
    unsigned long long pi;
    const int rank = rank_by_count(sp, K, P, i, h, &pi);
    if (i < K && h == 0) {
      const uint32_t kk = (uint32_t)(pi >> 32), ii = ~(uint32_t)pi;
      idx_out[rank] = (int32_t)ii;
      score_out[rank] = fkey_inv(kk);
      sh.sk[rank] = kk;
      sh.si[rank] = ii;
      if (rank == K - 1) sh.tau_key = kk;
    }
  }
  __syncthreads();
  if (thr_out) *thr_out = sh.tau_key;
  return true;
}

template <typename T>
__device__ __forceinline__ float score_col(const float* t, const T* V, int r, int vocab, int c) {
  float acc = 0.f;
#pragma unroll 16
  for (int j = 0; j < r; ++j) acc = fmaf(t[j], Elem<T>::to_f(V[(size_t)j * vocab + c]), acc);
  return acc;
}

// Four consecutive values of a V row as floats (8-byte load for bf16, 16-byte for fp32; the
// address is a multiple of 4 elements and rows start 16-byte aligned).
template <typename T>
__device__ __forceinline__ void load4(const T* p, float* x);
template <>
__device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16* p, float* x) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  x[0] = __uint_as_float(u.x << 16);
  x[1] = __uint_as_float(u.x & 0xFFFF0000u);
  x[2] = __uint_as_float(u.y << 16);
  x[3] = __uint_as_float(u.y & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void load4<float>(const float* p, float* x) {
  const float4 u = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = u.x;
  x[1] = u.y;
  x[2] = u.z;
  x[3] = u.w;
}

// Exact scores of the 64 ids of each of the n groups gs[0..n) (ids >= vocab give -inf) into
// out[i*64 .. i*64 + 64), n <= SG_BATCH.  The r rows of V are split over SG_PARTS parts (part w
// covers rows [w*rw, (w+1)*rw)); the block's warps take the (group, part) items in turn, so the
// loads of every group are in flight together, two rows per instruction (lanes 0-15 the even rows,
// 16-31 the odd ones; lane i loads ids 4(i mod 16) .. +3), up to 16 loads per lane.  The two halves
// are added with one shuffle, then each group's parts in part order: a fixed order whatever the
// block size, so blocks of 256 and 512 threads give the same scores.
// scratch: SG_BATCH * SG_PARTS * 64 floats.  vocab is a multiple of 4.
constexpr int SG_PARTS = 16;
constexpr int SG_BATCH = 4;
static_assert(SG_BATCH * SG_PARTS * 64 <= HIST_BINS, "the scratch is the histogram area");

template <typename T>
__device__ void score_groups(const float* t, const T* __restrict__ V, int r, int vocab, const int32_t* gs, int n,
                             float* out, float* scratch) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int rw = (r + SG_PARTS - 1) / SG_PARTS;
  const int half = lane >> 4;
  for (int item = warp; item < n * SG_PARTS; item += nw) {
    const int gi = item / SG_PARTS, part = item % SG_PARTS;
    const int c = gs[gi] * GROUP + 4 * (lane & 15);
    const bool cok = c < vocab;
    const int j0 = part * rw, j1 = min(r, j0 + rw);
    float a[4] = {0.f, 0.f, 0.f, 0.f};
    constexpr int BATCH = 16;
    for (int jb = j0; jb < j1; jb += 2 * BATCH) {
      float v[BATCH][4];
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        const int j = jb + 2 * q + half;
        if (j < j1 && cok) {
          load4<T>(V + (size_t)j * vocab + c, v[q]);
        } else {
          v[q][0] = v[q][1] = v[q][2] = v[q][3] = 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < BATCH; ++q) {
        const int j = jb + 2 * q + half;
        const float tj = (j < j1) ? t[j] : 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) a[e] = fmaf(tj, v[q][e], a[e]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) a[e] += __shfl_xor_sync(0xFFFFFFFFu, a[e], 16);
    if (lane < 16) {
#pragma unroll
      for (int e = 0; e < 4; ++e) scratch[item * 64 + 4 * lane + e] = a[e];
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n * 64; e += blockDim.x) {
    const int gi = e / 64, col = e % 64;
    float sum = 0.f;
    for (int w = 0; w < SG_PARTS; ++w) sum += scratch[(gi * SG_PARTS + w) * 64 + col];
    out[e] = (gs[gi] * GROUP + col < vocab) ? sum : -INFINITY;
  }
  __syncthreads();
}

// Shared memory select_row needs: the Shared block plus, when n_groups <= CACHE_GROUPS, a copy of
// the row's records.
__host__ __device__ constexpr size_t select_smem_bytes(int n_groups) {
  return align_up(sizeof(Shared), 16) + (n_groups <= CACHE_GROUPS ? (size_t)n_groups * sizeof(GroupRec) : 0);
}

// Exact top-K of one row by a block of NT threads (NT = blockDim.x).  smem: select_smem_bytes(n_groups)
// bytes, 16-byte aligned.  t_row: the row's projection (r values of the activation dtype), or
// nullptr with acc_row set: the row's slice of the small-batch projection's fixed-point
// accumulators (copies BR apart), which this block reads and then clears.  rrow: the row's
// n_groups records.  The register fast path is used when NT threads can hold the cached records
// (SEL_THREADS threads); otherwise the generic radix path.
template <typename T, int NT = SEL_THREADS>
__device__ void select_row(unsigned char* smem, const GroupRec* __restrict__ rrow, const T* __restrict__ t_row,
                           unsigned long long* __restrict__ acc_row, int BR, const T* __restrict__ V, int r,
                           int vocab, int K, int32_t* __restrict__ idx_out, float* __restrict__ score_out) {
  Shared& sh = *reinterpret_cast<Shared*>(smem);
  GroupRec* cache = reinterpret_cast<GroupRec*>(smem + align_up(sizeof(Shared), 16));
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const bool cached = n_groups <= CACHE_GROUPS;

  for (int g = threadIdx.x; g < (int)BITMAP_WORDS; g += blockDim.x) sh.bitmap[g] = 0u;
  if (acc_row) {
    for (int j = threadIdx.x; j < r; j += blockDim.x) {
      sh.t[j] = acc_to_t<T>(acc_row, BR, j);
#pragma unroll
      for (int q = 0; q < ACC_COPIES; ++q) acc_row[(size_t)q * BR + j] = 0ull;  // zero for the next call
    }
  } else {
    for (int j = threadIdx.x; j < r; j += blockDim.x) sh.t[j] = Elem<T>::to_f(t_row[j]);
  }
  // the row's records: in registers (thread i holds groups i, i + NT, ...) for the fast path and
  // the certificate, and copied to shared memory for the generic path and the refinement
  constexpr int PER_THREAD = (CACHE_GROUPS + NT - 1) / NT;
  constexpr bool FAST = 2 * PER_THREAD <= FP_ENT;
  constexpr int REGS = FAST ? PER_THREAD : 1;
  GroupRec tmp[REGS];
  if (cached && FAST) {
#pragma unroll
    for (int q = 0; q < REGS; ++q) {
      const int g = threadIdx.x + q * NT;
      if (g < n_groups) tmp[q] = rrow[g];
    }
#pragma unroll
    for (int q = 0; q < REGS; ++q) {
      const int g = threadIdx.x + q * NT;
      if (g < n_groups) cache[g] = tmp[q];
    }
  } else if (cached) {
    for (int g = threadIdx.x; g < n_groups; g += NT) cache[g] = rrow[g];
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
  auto load_pool = [&](uint32_t* key, uint32_t* id) {
#pragma unroll
    for (int q = 0; q < FP_ENT / 2; ++q) {
      const int g = threadIdx.x + q * NT;
      key[2 * q] = key[2 * q + 1] = 0u;
      id[2 * q] = id[2 * q + 1] = 0xFFFFFFFFu;
      if (q < REGS && g < n_groups) {
        const GroupRec rc = tmp[q];
        const uint32_t o1 = rc.offs & 0xFFu, o2 = (rc.offs >> 8) & 0xFFu;
        if (o1 != NO_OFFSET) { key[2 * q] = fkey(rc.m1); id[2 * q] = (uint32_t)g * GROUP + o1; }
        if (o2 != NO_OFFSET) { key[2 * q + 1] = fkey(rc.m2); id[2 * q + 1] = (uint32_t)g * GROUP + o2; }
      }
    }
  };
  bool selected = FAST && cached && fast_select(load_pool, 2 * n_groups, K, sh, idx_out, score_out, &tau);
  if (threadIdx.x == 0) sh.nref = 0;
  __syncthreads();
  if (!selected) selected = select_sort_write(pool, K, sh, idx_out, score_out, &tau);
  if (selected) {
    // Certificate: groups that may hide a member ranking at or above tau (third score >= tau).
    // tau is at or below the true K-th score, so without such groups the pool's top K is exact.
    auto mark = [&](int g) {
      const uint32_t pos = atomicAdd(&sh.nref, 1u);
      if (pos < RMAX) sh.rg[pos] = g;
      atomicOr(&sh.bitmap[g >> 5], 1u << (g & 31));
    };
    if (cached && FAST) {
#pragma unroll
      for (int q = 0; q < REGS; ++q) {
        const int g = threadIdx.x + q * NT;
        if (g < n_groups && fkey(tmp[q].m3) >= tau) mark(g);
      }
    } else {
      for (int g = threadIdx.x; g < n_groups; g += blockDim.x)
        if (fkey(src[g].m3) >= tau) mark(g);
    }
    __syncthreads();
    const int nref = (int)sh.nref;
    if (nref == 0) return;
    if (nref <= RMAX) {
      for (int i = 0; i < nref; i += SG_BATCH)
        score_groups(sh.t, V, r, vocab, sh.rg + i, min(SG_BATCH, nref - i), sh.rs + i * GROUP,
                     reinterpret_cast<float*>(sh.hist));
      // Candidates: the K selected pool entries outside the refined groups (sh.sk/si still hold the
      // selection) and the refined groups' members at or above tau.  Every entry of the exact top-K
      // is among them; when they number at least K (always, unless re-scoring moved a selected
      // score below tau by rounding) the top K by rank counting is the result.
      unsigned long long* cp = reinterpret_cast<unsigned long long*>(sh.hist);  // packed candidates
      constexpr int CMAX = HIST_BINS / 2;
      if (threadIdx.x == 0) sh.cnt = 0;
      __syncthreads();
      for (int k0 = 0; k0 < K; k0 += blockDim.x) {
        const int k = k0 + threadIdx.x;
        bool take = false;
        if (k < K) {
          const uint32_t g = sh.si[k] / GROUP;
          take = !((sh.bitmap[g >> 5] >> (g & 31)) & 1u);
        }
        const uint32_t pos = warp_append(take, &sh.cnt);
        if (take) cp[pos] = pack_entry(sh.sk[k], sh.si[k]);
      }
      for (int e0 = 0; e0 < nref * GROUP; e0 += blockDim.x) {
        const int e = e0 + threadIdx.x;
        bool take = false;
        uint32_t key = 0;
        int c = 0;
        if (e < nref * GROUP) {
          c = sh.rg[e / GROUP] * GROUP + (e % GROUP);
          key = fkey(sh.rs[e]);
          take = c < vocab && key >= tau;
        }
        const uint32_t pos = warp_append(take, &sh.cnt);
        if (take && pos < CMAX) cp[pos] = pack_entry(key, (uint32_t)c);
      }
      __syncthreads();
      const int n = (int)sh.cnt;
      __syncthreads();
      if (n >= K && n <= CMAX) {
        // rank every candidate among the n by counting, P threads per candidate
        int P = 1;
        while (P < 32 && n * (2 * P) <= (int)blockDim.x) P <<= 1;
        for (int base = 0; base < n * P; base += blockDim.x) {
          const int t = base + (int)threadIdx.x;
          const int i = t / P, h = t % P;
          unsigned long long pi;
          const int rank = rank_by_count(cp, n, P, i, h, &pi);
          if (i < n && h == 0 && rank < K) {
            idx_out[rank] = (int32_t)(~(uint32_t)pi);
            score_out[rank] = fkey_inv((uint32_t)(pi >> 32));
          }
        }
        return;
      }
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
