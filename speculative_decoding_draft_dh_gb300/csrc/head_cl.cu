// Small batches: selection and exact rescoring fused into one kernel, one thread-block cluster of
// 16, 8 or 4 CTAs per row.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the K candidates of a row are its K best low-rank scores (score desc, id asc); their exact
// logits come from the full-rank head, and the softmax runs over the K candidates.
//
// At batch 1 the selection is a short chain of dependent steps over about 4700 pool entries, and
// each kernel boundary in the pipeline costs one to two microseconds.  Here the cluster's CTAs
// split the row's group records and select cooperatively through distributed shared memory, with
// the steps of the register fast path of the selection kernel (radix levels over the pool's own
// key range, compaction, ranking by counting):
//  - the key range is combined in the leader CTA (rank 0) behind one cluster barrier;
//  - each radix level: every CTA histograms its own entries locally, and after one cluster barrier
//    every CTA sums the CTAs' histograms and finds the boundary bin itself;
//  - compaction writes the entries above and in the boundary bin into every CTA's lists;
//  - every CTA ranks the boundary bin itself, so it knows the K winners and tau, checks the
//    certificate on its groups and scores its share of the winners against h (staged in shared
//    memory before the wait on the previous kernel), storing the logits into the leader, while the
//    leader ranks the winners and writes them in order;
//  - after one more barrier the leader orders the logits and computes the softmax.
// A row whose certificate finds groups to re-score, or whose pool is degenerate, is selected again
// by the leader alone with the block selection (select_row: exact, with refinement and full
// rescan) and then rescored.
//
// Cluster barriers are hardware barriers that every CTA passes unconditionally, so they always
// complete.
#include <cooperative_groups.h>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "select.cuh"

namespace dh {
namespace {

namespace cg = cooperative_groups;

// A cluster has 16 CTAs where the GPU can schedule such clusters (a non-portable size: the CTAs
// must share a GPC), else 8 or 4; each thread holds 16 / CTAS group records, so every size covers
// 4096 groups.  Spreading the candidates' W rows over 16 SMs halves each SM's share of the
// rescoring loads (20.1 against 20.4 µs per call at batch 1).
constexpr int HC_THREADS = 256;
constexpr int HC_WARPS = HC_THREADS / 32;
constexpr int HC_MAX_GROUPS = 16 * HC_THREADS;  // 4096 groups: vocab <= 262144
constexpr int HC_MAX_K = 256;
constexpr int HC_BINS = 256;
constexpr int HC_BITS = 8;
static_assert(HC_BINS == HC_THREADS, "one bin per thread in the level scan");
constexpr int HC_RANK = 64;    // a level whose boundary bin holds at most this many ends the descent
constexpr int HC_BOUND = 512;  // largest boundary bin ranked by counting

// Control block: every CTA has one; the leader's is the one in use.
struct HeadCtl {
  uint32_t hist[2][HC_BINS];  // this CTA's histograms (even and odd levels)
  uint32_t wsc[HC_WARPS];     // per-warp totals of the bin scan
  uint32_t kmin, kmax;
  uint32_t digit, run, bincount, total;
  uint32_t n_above, n_bound, nref, tau_key;
  uint32_t wmin[HC_WARPS], wmax[HC_WARPS];
  alignas(16) unsigned long long sp[HC_MAX_K];  // the K winners, packed key << 32 | ~id (unsorted)
  alignas(16) unsigned long long bp[HC_BOUND];  // the boundary bin
  alignas(16) unsigned long long wb[HC_MAX_K];  // the boundary bin's winners, best first
  float z[HC_MAX_K];                            // the row's logits in rank order (leader)
  float zu[HC_MAX_K];                           // the logits by winner position (leader)
  int32_t rk[HC_MAX_K];                         // rank of each winner position (leader)
};

struct HeadParams {
  const GroupRec* recs;     // [B][n_groups]
  const uint32_t* gkeys;    // [B][n_groups] the groups' best keys (fast selection), or null
  unsigned long long* acc;  // the small-batch projection's fixed-point accumulators (cleared here), or
  const void* t;            // t [B][r] in the activation dtype (tensor-core stage 1)
  const void* V;
  const void* h;
  const void* W;
  int B, d, r, vocab, K, n_groups;
  int32_t* idx_out;
  float* score_out;
  float* logits;
  float* probs;  // may be null
};

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk prefetch of [p, p + bytes) into L2 (p 16-byte aligned, bytes a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ unsigned long long pack(uint32_t key, uint32_t id) {
  return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}

// One warp's dot product of h (in shared memory) with W row v, in the rescoring kernels' order:
// each lane keeps MAXW 16-byte loads of the row in flight, accumulates in fp32, and the warp
// reduces with xor shuffles (every lane gets the sum).  The same order gives bit-identical logits.
template <typename T>
__device__ __forceinline__ float row_dot(const T* __restrict__ W, int v, int d, const T* hs, int lane) {
  constexpr int PER = Elem<T>::PER16;
  constexpr int MAXW = 20;
  const T* w = W + (size_t)v * d;
  float acc = 0.f;
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
        Elem<T>::unpack(*reinterpret_cast<const uint4*>(hs + c), xf);
#pragma unroll
        for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// Dynamic shared memory layout: control block, h, then the block selection's area (leader only).
__host__ __device__ constexpr size_t hc_h_offset() { return align_up(sizeof(HeadCtl), 128); }
__host__ __device__ constexpr size_t hc_fb_offset(int d, int elem) {
  return hc_h_offset() + align_up((size_t)d * elem, 128);
}

// Block-local state of the fast selection.
struct FastShared {
  uint32_t hist[HC_BINS];
  uint32_t wsc[HC_WARPS], wmin[HC_WARPS], wmax[HC_WARPS];
  uint32_t digit, run, bincount, total, nb, theta;
  uint32_t bk[HC_RANK];  // the last level's bin
};

// Fast selection from the groups' best keys (written by the small-batch scores kernel).
// theta = the K-th largest of the row's group bests; each CTA finds it alone (radix levels over
// the keys' own range with block barriers, then ranking inside the last bin).  The K groups whose
// bests reach theta put K pool entries at or above it, so the pool's K-th best is >= theta and
// every entry of the pool's top K is >= theta: the entries >= theta (K to 2K of them on random
// rows) are compacted into every CTA's list behind one cluster barrier and ranked there, which
// also orders them.  Then the certificate, the exact logits of the winners (each CTA its share)
// and one more cluster barrier; the leader computes the softmax.  Returns true when the row must
// take the leader's exact selection instead: more than HC_BOUND entries reach theta, fewer than K
// groups hold entries, or the certificate flags a group.  Every CTA takes the same decision at
// the same barrier.
template <typename T, int HC_CTAS, int HC_RPT, int HC_ENT>
__device__ __forceinline__ bool head_fast(const HeadParams& p, cg::cluster_group& cl, HeadCtl& my, HeadCtl& L,
                                          FastShared& fs, const T* hs, int b, int g0, int g1,
                                          const GroupRec (&rec)[HC_RPT], const uint32_t (&key)[HC_ENT],
                                          const uint32_t (&id)[HC_ENT]) {
  constexpr int GK = HC_MAX_GROUPS / HC_THREADS;  // group keys per thread
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K, n_groups = p.n_groups;
  const bool leader = cl.block_rank() == 0;
  // every group's best key of the row (written by the previous kernel: read through L2)
  const uint32_t* grow = p.gkeys + (size_t)b * n_groups;
  uint32_t y[GK];
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < GK; ++q) {
    const int g = (int)threadIdx.x + q * HC_THREADS;
    y[q] = g < n_groups ? __ldcg(grow + g) : 0u;
    if (y[q]) { kmin = min(kmin, y[q]); kmax = max(kmax, y[q]); }
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) { fs.wmin[warp] = kmin; fs.wmax[warp] = kmax; }
  fs.hist[threadIdx.x] = 0u;
  if (threadIdx.x == 0) fs.nb = 0u;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < HC_WARPS; ++w) { kmin = min(kmin, fs.wmin[w]); kmax = max(kmax, fs.wmax[w]); }
  // every CTA's control block is zeroed (the initial arrive) before the compaction writes into it
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  bool ok = kmax != 0u;
  uint32_t theta = 0u;
  if (ok) {
#pragma unroll
    for (int q = 0; q < GK; ++q) y[q] = y[q] ? y[q] - kmin + 1u : 0u;  // 0 = empty group
    const uint32_t range = kmax - kmin + 1u;
    int shift = range >= 0x80000000u ? 32 - HC_BITS : max(0, (32 - __clz((int)range)) - HC_BITS);
    uint32_t prefix = 0u, mask = 0u, krem = (uint32_t)K, bc = 0u;
    bool first = true;
#pragma unroll 1
    for (;;) {
#pragma unroll
      for (int q = 0; q < GK; ++q)
        if (y[q] && (y[q] & mask) == prefix) atomicAdd(&fs.hist[(y[q] >> shift) & (HC_BINS - 1)], 1u);
      __syncthreads();
      const int bin = HC_BINS - 1 - (int)threadIdx.x;  // from the top
      const uint32_t cnt = fs.hist[bin];
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) fs.wsc[warp] = incl;
      __syncthreads();
      uint32_t before = 0u;
#pragma unroll
      for (int w = 0; w < HC_WARPS; ++w) before += w < warp ? fs.wsc[w] : 0u;
      incl += before;
      if (incl - cnt < krem && krem <= incl) { fs.digit = (uint32_t)bin; fs.run = incl - cnt; fs.bincount = cnt; }
      if (threadIdx.x == HC_THREADS - 1) fs.total = incl;
      fs.hist[bin] = 0u;  // this thread's own bin, for the next level
      __syncthreads();
      if (first && fs.total < (uint32_t)K) { ok = false; break; }  // fewer nonempty groups than K
      first = false;
      prefix |= fs.digit << shift;
      mask |= (uint32_t)(HC_BINS - 1) << shift;
      krem -= fs.run;
      bc = fs.bincount;
      if (bc <= (uint32_t)HC_RANK || shift == 0) break;
      shift = max(0, shift - HC_BITS);
    }
    if (ok) {
      uint32_t ty = prefix;  // shift 0: every key of the last bin equals prefix
      if (shift > 0) {
        // the last bin holds at most HC_RANK keys: the krem-th largest of them by counting
#pragma unroll
        for (int q = 0; q < GK; ++q)
          if (y[q] && (y[q] & mask) == prefix) fs.bk[atomicAdd(&fs.nb, 1u)] = y[q];
        __syncthreads();
        if (threadIdx.x < bc) {
          const uint32_t yi = fs.bk[threadIdx.x];
          uint32_t rank = 0u;
          for (uint32_t j = 0; j < bc; ++j) {
            const uint32_t yj = fs.bk[j];
            rank += (yj > yi || (yj == yi && j < threadIdx.x)) ? 1u : 0u;
          }
          if (rank == krem - 1u) fs.theta = yi;
        }
        __syncthreads();
        ty = fs.theta;
      }
      theta = ty - 1u + kmin;
    }
  }
  // the pool entries at or above theta into every CTA's list (positions from warp ballots and one
  // remote atomic per warp on the leader's counter); their W rows start towards L2 now
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll
  for (int q = 0; q < HC_ENT; ++q) {
    const bool c = ok && key[q] && key[q] >= theta;
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, c);
    uint32_t base = 0u;
    if (lane == 0 && bal) base = atomicAdd(&L.n_bound, (uint32_t)__popc(bal));
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    if (c) {
      const uint32_t pos = base + (uint32_t)__popc(bal & below);
      if (pos < (uint32_t)HC_BOUND) {
        const unsigned long long e = pack(key[q], id[q]);
#pragma unroll
        for (int c2 = 0; c2 < HC_CTAS; ++c2) *cl.map_shared_rank(&my.bp[pos], (unsigned)c2) = e;
      }
      if (id[q] < (uint32_t)p.vocab)
        prefetch_l2(static_cast<const T*>(p.W) + (size_t)id[q] * p.d, (uint32_t)(p.d * sizeof(T)));
    }
  }
  cluster_sync_all();
  const uint32_t n_cand = L.n_bound;  // the leader passes one more barrier below before it exits
  if (!ok || n_cand > (uint32_t)HC_BOUND || n_cand < (uint32_t)K) return true;
  // rank the candidates by counting: winner of rank k < K into sp[k] (every CTA, its own copy)
  {
    int P = 1;
    while (P < 32 && (int)n_cand * (2 * P) <= HC_THREADS) P <<= 1;
    for (int base = 0; base < (int)n_cand * P; base += HC_THREADS) {
      const int t = base + (int)threadIdx.x;
      const int i = t / P, hh = t % P;
      unsigned long long pi;
      const int rank = sel::rank_by_count(my.bp, (int)n_cand, P, i, hh, &pi);
      if (i < (int)n_cand && hh == 0 && rank < K) my.sp[rank] = pi;
    }
  }
  __syncthreads();
  // certificate: a group whose third score reaches tau (the K-th best) may hide a top-K member
  const uint32_t tau = (uint32_t)(my.sp[K - 1] >> 32);
  bool flag = false;
#pragma unroll
  for (int q = 0; q < HC_RPT; ++q)
    flag |= (g0 + (int)threadIdx.x + q * HC_THREADS) < g1 && fkey(rec[q].m3) >= tau;
  const uint32_t fm = __ballot_sync(0xFFFFFFFFu, flag);
  if (lane == 0 && fm)
#pragma unroll
    for (int c2 = 0; c2 < HC_CTAS; ++c2) atomicAdd(cl.map_shared_rank(&my.nref, (unsigned)c2), (uint32_t)__popc(fm));
  // exact logits of this CTA's winners, written out and stored into the leader for the softmax
  const int crank = (int)cl.block_rank();
  float* zl = cl.map_shared_rank(&my.z[0], 0u);
  for (int k = warp * HC_CTAS + crank; k < K; k += HC_CTAS * HC_WARPS) {
    const unsigned long long e = my.sp[k];
    const int v = (int)(~(uint32_t)e);
    const bool okv = v >= 0 && v < p.vocab;
    const float acc = okv ? row_dot<T>(static_cast<const T*>(p.W), v, p.d, hs, lane) : 0.f;
    const float z = okv ? acc : __int_as_float(0x7FC00000);
    if (lane == 0) {
      p.idx_out[(size_t)b * K + k] = v;
      p.score_out[(size_t)b * K + k] = fkey_inv((uint32_t)(e >> 32));
      p.logits[(size_t)b * K + k] = z;
      zl[k] = z;
    }
  }
  cluster_sync_all();
  if (my.nref != 0u) return true;
  if (!leader) return false;
  // the row's accumulators are cleared for the next call (select_row does it on the other branch)
  if (p.acc) {
    const int BR = p.B * p.r;
    unsigned long long* acc_row = p.acc + (size_t)b * p.r;
    for (int j = threadIdx.x; j < p.r; j += HC_THREADS)
#pragma unroll
      for (int q = 0; q < ACC_COPIES; ++q) acc_row[(size_t)q * BR + j] = 0ull;
  }
  if (p.probs && warp == 0) warp_softmax(my.z, K, p.probs + (size_t)b * K);
  return false;
}

template <typename T, int HC_CTAS>
__global__ void __launch_bounds__(HC_THREADS, 1) k_head_cl(HeadParams p) {
  constexpr int HC_RPT = 16 / HC_CTAS;  // group records per thread
  constexpr int HC_ENT = 2 * HC_RPT;    // pool entries per thread
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ __align__(128) unsigned char smem[];
  cg::cluster_group cl = cg::this_cluster();
  const uint32_t crank = cl.block_rank();
  const bool leader = crank == 0;
  const int b = (int)(blockIdx.x / HC_CTAS);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K, n_groups = p.n_groups, BR = p.B * p.r;
  HeadCtl& my = *reinterpret_cast<HeadCtl*>(smem);
  HeadCtl& L = *cl.map_shared_rank(&my, 0u);
  T* hs = reinterpret_cast<T*>(smem + hc_h_offset());
  unsigned char* fb = smem + hc_fb_offset(p.d, (int)sizeof(T));
  const GroupRec* rrow = p.recs + (size_t)b * n_groups;
  unsigned long long* acc_row = p.acc ? p.acc + (size_t)b * p.r : nullptr;
  const T* t_row = p.acc ? nullptr : static_cast<const T*>(p.t) + (size_t)b * p.r;

  // zero this CTA's control block; the barrier's wait (below) makes the leader's visible
  for (int i = threadIdx.x; i < HC_BINS; i += HC_THREADS) my.hist[0][i] = my.hist[1][i] = 0u;
  if (threadIdx.x == 0) {
    my.kmin = 0xFFFFFFFFu;
    my.kmax = 0u;
    my.n_above = my.n_bound = my.nref = 0u;
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // h does not depend on the previous kernels
  const T* hrow = static_cast<const T*>(p.h) + (size_t)b * p.d;
  for (int c = threadIdx.x * PER; c < p.d; c += HC_THREADS * PER)
    *reinterpret_cast<uint4*>(hs + c) = __ldg(reinterpret_cast<const uint4*>(hrow + c));
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the records come from the scores kernel

  // this CTA's slice of the row's groups
  const int slice = (n_groups + HC_CTAS - 1) / HC_CTAS;
  const int g0 = (int)crank * slice, g1 = min(n_groups, g0 + slice);
  GroupRec rec[HC_RPT];
  uint32_t key[HC_ENT], id[HC_ENT];
#pragma unroll
  for (int q = 0; q < HC_RPT; ++q) {
    const int g = g0 + threadIdx.x + q * HC_THREADS;
    key[2 * q] = key[2 * q + 1] = 0u;
    id[2 * q] = id[2 * q + 1] = 0xFFFFFFFFu;
    rec[q].m3 = -INFINITY;
    if (g < g1) {
      rec[q] = rrow[g];
      const uint32_t o1 = rec[q].offs & 0xFFu, o2 = (rec[q].offs >> 8) & 0xFFu;
      if (o1 != NO_OFFSET) { key[2 * q] = fkey(rec[q].m1); id[2 * q] = (uint32_t)g * GROUP + o1; }
      if (o2 != NO_OFFSET) { key[2 * q + 1] = fkey(rec[q].m2); id[2 * q + 1] = (uint32_t)g * GROUP + o2; }
    }
  }
  bool fallback = false;
  if (p.gkeys) {
    __shared__ FastShared fs;
    if (!head_fast<T, HC_CTAS, HC_RPT, HC_ENT>(p, cl, my, L, fs, hs, b, g0, g1, rec, key, id)) return;
    fallback = true;
  } else {
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int q = 0; q < HC_ENT; ++q)
    if (key[q]) { kmin = min(kmin, key[q]); kmax = max(kmax, key[q]); }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) { my.wmin[warp] = kmin; my.wmax[warp] = kmax; }
  __syncthreads();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every control block is zeroed
  if (threadIdx.x == 0) {
    for (int w = 0; w < HC_WARPS; ++w) { kmin = min(kmin, my.wmin[w]); kmax = max(kmax, my.wmax[w]); }
    if (kmax) {
      atomicMin(&L.kmin, kmin);
      atomicMax(&L.kmax, kmax);
    }
  }
  cluster_sync_all();
  kmin = L.kmin;
  kmax = L.kmax;

  // ---------------------------------------------------------------- cooperative radix descent
  fallback = kmax == 0u;  // empty pool
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)K, above = 0, bc = 0;
  if (!fallback) {
#pragma unroll
    for (int q = 0; q < HC_ENT; ++q) key[q] = key[q] ? key[q] - kmin + 1u : 0u;  // y + 1 (0 = no entry)
    const uint32_t range = kmax - kmin + 1u;
    int shift = range >= 0x80000000u ? 32 - HC_BITS : max(0, (32 - __clz((int)range)) - HC_BITS);
    const uint32_t dmask = (uint32_t)HC_BINS - 1u;
    bool first = true;
    int lvl = 0;
#pragma unroll 1
    for (;;) {
      // each CTA histograms its own entries; after the barrier every CTA sums the CTAs' histograms
      // and finds the digit itself, so a level costs one cluster barrier
      uint32_t* hb = my.hist[lvl & 1];
#pragma unroll
      for (int q = 0; q < HC_ENT; ++q)
        if (key[q] && (key[q] & mask) == prefix) atomicAdd(&hb[(key[q] >> shift) & dmask], 1u);
      cluster_sync_all();
      const int bin = HC_BINS - 1 - (int)threadIdx.x;  // thread t takes bin 255 - t: scan from the top
      uint32_t cnt = 0;
#pragma unroll
      for (int c = 0; c < HC_CTAS; ++c) cnt += cl.map_shared_rank(hb, (unsigned)c)[bin];
      // the other buffer was last read (by every CTA) before this level's barrier
      my.hist[(lvl & 1) ^ 1][threadIdx.x] = 0u;
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) my.wsc[warp] = incl;
      __syncthreads();
      uint32_t before = 0, total = 0;
#pragma unroll
      for (int w = 0; w < HC_WARPS; ++w) {
        const uint32_t x = my.wsc[w];
        before += w < warp ? x : 0u;
        total += x;
      }
      incl += before;
      if (incl - cnt < krem && krem <= incl) {
        my.digit = (uint32_t)bin;
        my.run = incl - cnt;
        my.bincount = cnt;
      }
      __syncthreads();
      ++lvl;
      if (first && total < (uint32_t)K) { fallback = true; break; }
      const uint32_t D = my.digit, run = my.run;
      bc = my.bincount;
      first = false;
      prefix |= D << shift;
      mask |= dmask << shift;
      krem -= run;
      above += run;
      if (bc <= (uint32_t)HC_RANK || shift == 0) break;
      shift = max(0, shift - HC_BITS);
    }
    if (bc > (uint32_t)HC_BOUND) fallback = true;
  }
  // every CTA took the same decisions from the same histograms
  if (!fallback) {
    // compaction into every CTA's lists (positions from warp ballots, one remote atomic per warp
    // on the leader's counters, each entry stored into all CTAs)
    const uint32_t below = (1u << lane) - 1u;
#pragma unroll
    for (int q = 0; q < HC_ENT; ++q) {
      const uint32_t mk = key[q] & mask;
      const bool up = key[q] && mk > prefix, bd = key[q] && mk == prefix;
      const uint32_t bu = __ballot_sync(0xFFFFFFFFu, up), bb = __ballot_sync(0xFFFFFFFFu, bd);
      uint32_t base_u = 0, base_b = 0;
      if (lane == 0) {
        if (bu) base_u = atomicAdd(&L.n_above, (uint32_t)__popc(bu));
        if (bb) base_b = atomicAdd(&L.n_bound, (uint32_t)__popc(bb));
      }
      base_u = __shfl_sync(0xFFFFFFFFu, base_u, 0);
      base_b = __shfl_sync(0xFFFFFFFFu, base_b, 0);
      if (up || bd) {
        const unsigned long long e = pack(key[q] - 1u + kmin, id[q]);
        unsigned long long* dst = up ? &my.sp[base_u + __popc(bu & below)] : &my.bp[base_b + __popc(bb & below)];
#pragma unroll
        for (int c = 0; c < HC_CTAS; ++c) *cl.map_shared_rank(dst, (unsigned)c) = e;
      }
    }
    cluster_sync_all();
    // Every CTA now holds the winners above the boundary bin (sp[0, above)) and the boundary bin
    // (bp[0, bc)).  Each ranks the bin itself, so it knows all K winners, and tau (the K-th best
    // key: the worst boundary winner) without waiting for the leader's sort.
    const int need = K - (int)above;  // at least one: the boundary bin holds the K-th entry
    {
      int P = 1;
      while (P < 32 && (int)bc * (2 * P) <= HC_THREADS) P <<= 1;
      for (int base = 0; base < (int)bc * P; base += HC_THREADS) {
        const int t = base + (int)threadIdx.x;
        const int i = t / P, hh = t % P;
        unsigned long long pi;
        const int rank = sel::rank_by_count(my.bp, (int)bc, P, i, hh, &pi);
        if (i < (int)bc && hh == 0 && rank < need) my.wb[rank] = pi;
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < need; i += HC_THREADS) my.sp[above + i] = my.wb[i];
    // Candidate positions of this CTA's warps: when the other CTAs have a warp for every
    // candidate, the leader, which sorts, scores none; otherwise every CTA scores.  Warp w of
    // scoring CTA c takes k = w * n_sc + c, k + n_sc * HC_WARPS, ...
    const bool leader_sorts_only = K <= (HC_CTAS - 1) * HC_WARPS;
    const int n_sc = leader_sorts_only ? HC_CTAS - 1 : HC_CTAS;
    const int c_sc = leader_sorts_only ? (int)crank - 1 : (int)crank;  // -1: the leader
    const int k_first = c_sc < 0 ? K : warp * n_sc + c_sc;
    // this CTA's candidates' W rows start towards L2 now (the certificate comes before the dot
    // products)
    if (lane == 0)
      for (int k = k_first; k < K; k += n_sc * HC_WARPS) {
        const int v = (int)(~(uint32_t)(k < (int)above ? my.sp[k] : my.wb[k - (int)above]));
        if (v >= 0 && v < p.vocab)
          prefetch_l2(static_cast<const T*>(p.W) + (size_t)v * p.d, (uint32_t)(p.d * sizeof(T)));
      }
    const uint32_t tau = (uint32_t)(my.wb[need - 1] >> 32);
    // certificate: a group whose third score reaches tau may hide a member of the top K
    bool mine = false;
#pragma unroll
    for (int q = 0; q < HC_RPT; ++q) mine |= fkey(rec[q].m3) >= tau && (g0 + (int)threadIdx.x + q * HC_THREADS) < g1;
    // every CTA's own count gets the flags, so that after the barrier below each CTA reads only
    // its own shared memory (the leader may exit as soon as it has passed that barrier)
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, mine);
    if (lane == 0 && bm)
#pragma unroll
      for (int c = 0; c < HC_CTAS; ++c) atomicAdd(cl.map_shared_rank(&my.nref, (unsigned)c), (uint32_t)__popc(bm));
    __syncthreads();  // sp[0, K) complete in this CTA
    if (leader) {
      // the winners' order: rank by counting, outputs written in rank order
      int P = 1;
      while (P < 32 && K * (2 * P) <= HC_THREADS) P <<= 1;
      for (int base = 0; base < K * P; base += HC_THREADS) {
        const int t = base + (int)threadIdx.x;
        const int i = t / P, hh = t % P;
        unsigned long long pi;
        const int rank = sel::rank_by_count(my.sp, K, P, i, hh, &pi);
        if (i < K && hh == 0) {
          p.idx_out[(size_t)b * K + rank] = (int32_t)(~(uint32_t)pi);
          p.score_out[(size_t)b * K + rank] = fkey_inv((uint32_t)(pi >> 32));
          my.rk[i] = rank;
        }
      }
    }
    // exact logits of the winners by position, into the leader, while it sorts; they are used
    // unless the certificate sends the row to the leader's block selection
    for (int k = k_first; k < K; k += n_sc * HC_WARPS) {
      const int v = (int)(~(uint32_t)my.sp[k]);
      const bool ok = v >= 0 && v < p.vocab;
      const float acc = ok ? row_dot<T>(static_cast<const T*>(p.W), v, p.d, hs, lane) : 0.f;
      if (lane == 0) L.zu[k] = ok ? acc : __int_as_float(0x7FC00000);
    }
    cluster_sync_all();
    fallback = my.nref != 0u;
    if (!fallback) {
      if (!leader) return;
      // zero the row's accumulators for the next call (select_row does it on the other branch)
      if (acc_row)
        for (int j = threadIdx.x; j < p.r; j += HC_THREADS)
#pragma unroll
          for (int q = 0; q < ACC_COPIES; ++q) acc_row[(size_t)q * BR + j] = 0ull;
      for (int k = threadIdx.x; k < K; k += HC_THREADS) {
        const float z = my.zu[k];
        my.z[my.rk[k]] = z;
        p.logits[(size_t)b * K + my.rk[k]] = z;
      }
      __syncthreads();
      if (p.probs && warp == 0) warp_softmax(my.z, K, p.probs + (size_t)b * K);
      return;
    }
  }
  }  // the cooperative radix selection
  // the leader selects the row alone: exact, with refinement or a full rescan as needed
  if (leader)
    sel::select_row<T, HC_THREADS>(fb, rrow, t_row, acc_row, BR, static_cast<const T*>(p.V), p.r, p.vocab, K,
                                   p.idx_out + (size_t)b * K, p.score_out + (size_t)b * K);
  cluster_sync_all();

  // ---------------------------------------------------------------- exact logits and softmax
  const int32_t* cand = p.idx_out + (size_t)b * K;
  for (int k = warp * HC_CTAS + (int)crank; k < K; k += HC_CTAS * HC_WARPS) {
    const int v = cand[k];
    const bool ok = v >= 0 && v < p.vocab;
    const float acc = ok ? row_dot<T>(static_cast<const T*>(p.W), v, p.d, hs, lane) : 0.f;
    const float z = ok ? acc : __int_as_float(0x7FC00000);
    if (lane == 0) {
      p.logits[(size_t)b * K + k] = z;
      L.z[k] = z;
    }
  }
  cluster_sync_all();
  if (!leader || !p.probs || warp != 0) return;
  warp_softmax(my.z, K, p.probs + (size_t)b * K);
}

template <typename T, int CTAS>
cudaError_t launch(const Ctx& c, const HeadParams& p, size_t smem) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CTAS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * CTAS));
  cfg.blockDim = dim3(HC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_before("head_cluster", c.stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_head_cl<T, CTAS>, p);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Clusters of CTAS CTAs with this shared memory that run at once on the device (0 if none).
template <typename T, int CTAS>
int clusters_at_once(int device, size_t smem) {
  unsigned long long done = 0;  // the query needs the kernel's shared memory limit raised
  if (allow_max_smem(k_head_cl<T, CTAS>, device, &done) != cudaSuccess) return 0;
  if (CTAS > 8 &&
      cudaFuncSetAttribute(k_head_cl<T, CTAS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    return 0;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CTAS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CTAS);
  cfg.blockDim = dim3(HC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_head_cl<T, CTAS>, &cfg) != cudaSuccess) n = 0;
  return n;
}

// Cluster size for B rows: 16 CTAs when all B clusters of 16 run at once, else 8 when all B
// clusters of 8 do, else 4 for up to 2048 (row, candidate) pairs when all B clusters of 4 do, else
// 0 (the batch goes to the selection and rescoring kernels).  Four CTAs score eight or more
// candidates per warp, one row after another; that pays against the two kernels up to about 2048
// pairs (32 rows x 64: 31.0 against 39.0 µs per call; 16 x 64: 29.3 against 32.6) but not beyond
// (64 x 128: 77.6 against 56.4).  The device's capacities are queried once per device and element
// type (set-up calls: shared memory limit, the non-portable size, the occupancy query).
// The DH_HEAD_CTAS switch (8 or 4) skips the larger forms (tests).
template <typename T>
int choose_ctas(const Ctx& c, int B, int K, int d, int n_groups) {
  const size_t smem = hc_fb_offset(d, (int)sizeof(T)) + sel::select_smem_bytes(n_groups);
  static std::mutex mu;
  static int cap[64][3] = {};  // [device]: clusters of 16, 8 and 4 at once, +1 (0: not queried)
  static size_t smem_at[64] = {};
  if (c.device < 0 || c.device >= 64) return 0;
  int n16, n8, n4;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (cap[c.device][0] == 0 || smem_at[c.device] < smem) {
      cap[c.device][0] = clusters_at_once<T, 16>(c.device, smem) + 1;
      cap[c.device][1] = clusters_at_once<T, 8>(c.device, smem) + 1;
      cap[c.device][2] = clusters_at_once<T, 4>(c.device, smem) + 1;
      smem_at[c.device] = smem;
      (void)cudaGetLastError();  // a refused query leaves no sticky error behind
    }
    n16 = cap[c.device][0] - 1;
    n8 = cap[c.device][1] - 1;
    n4 = cap[c.device][2] - 1;
  }
  const int most = tuning().head_ctas_max;
  if (most >= 16 && B <= n16) return 16;
  if (most >= 8 && B <= n8) return 8;
  if (most >= 4 && B <= n4 && (long long)B * K <= 2048) return 4;
  return 0;
}

template <typename T>
cudaError_t run(const Ctx& c, const HeadParams& p, int ctas) {
  const size_t smem = hc_fb_offset(p.d, (int)sizeof(T)) + sel::select_smem_bytes(p.n_groups);
  if (ctas == 4) return launch<T, 4>(c, p, smem);
  return ctas == 16 ? launch<T, 16>(c, p, smem) : launch<T, 8>(c, p, smem);
}

}  // namespace

int head_cluster_ctas(const Ctx& c, int B, int K, int d, int vocab, int dtype) {
  // a wave of clusters holds at most one row per 4 SMs: larger batches need no query
  if (B > c.num_sms / 4) return 0;
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  return dtype == DH_BF16 ? choose_ctas<__nv_bfloat16>(c, B, K, d, n_groups)
                          : choose_ctas<float>(c, B, K, d, n_groups);
}

bool head_cluster_supported(int B, int d, int vocab, int K, int dtype) {
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const size_t smem = hc_fb_offset(d, dtype == DH_BF16 ? 2 : 4) + sel::select_smem_bytes(n_groups);
  return B >= 1 && K <= HC_MAX_K && n_groups <= HC_MAX_GROUPS && n_groups <= sel::CACHE_GROUPS &&
         d <= 8192 && smem <= 200 * 1024;
}

cudaError_t launch_head_cluster(const Ctx& c, int ctas, const GroupRec* recs, const uint32_t* gkeys,
                                unsigned long long* acc, const void* t, const void* V, const void* h, const void* W,
                                int B, int d, int r, int vocab, int K, int dtype, int32_t* idx_out, float* score_out,
                                float* logits, float* probs) {
  if (ctas != 4 && ctas != 8 && ctas != 16) return cudaErrorInvalidValue;
  HeadParams p;
  p.recs = recs;
  p.gkeys = gkeys;
  p.acc = acc;
  p.t = t;
  p.V = V;
  p.h = h;
  p.W = W;
  p.B = B;
  p.d = d;
  p.r = r;
  p.vocab = vocab;
  p.K = K;
  p.n_groups = (vocab + GROUP - 1) / GROUP;
  p.idx_out = idx_out;
  p.score_out = score_out;
  p.logits = logits;
  p.probs = probs;
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, p, ctas);
  return run<float>(c, p, ctas);
}

}  // namespace dh
