// Small batches: selection and exact rescoring fused into one kernel, one thread-block cluster of
// 16, 8 or 4 CTAs per row.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the K candidates of a row are its K best low-rank scores (score desc, id asc); their exact
// logits come from the full-rank head, and the softmax runs over the K candidates.
//
// At batch 1 the selection is a short chain of dependent steps, and each kernel boundary or
// cluster barrier costs about half a microsecond to a microsecond.  Two selections run here:
//  - the fast selection (the default: the stage-1 scores kernels, small-batch or tensor-core, also
//    write every group's best key when this kernel follows): every CTA selects the K winners itself (a bound from K disjoint subsets of
//    the groups' best keys, one histogram, then the records of the few candidate groups, read
//    through L2, ranked by counting), so the CTAs exchange nothing until the exact logits; each CTA
//    starts the W rows of its share of the candidate groups towards L2 as soon as it knows them,
//    scores its share of the winners against h (bulk-copied into shared memory at the start), and
//    stores the logits into the leader (rank 0), which computes the softmax after one cluster
//    barrier;
//  - the cooperative radix selection (DH_HEAD_SELECT=radix): the CTAs split the row's group records;
//    the key range is combined in the leader behind one cluster barrier; each radix level every CTA
//    histograms its own entries and, after one cluster barrier, sums the CTAs' histograms and finds
//    the boundary bin itself; compaction writes the entries above and in the boundary bin into
//    every CTA's lists; every CTA ranks the boundary bin, knows the K winners and tau, checks the
//    certificate on its groups and scores its share of the winners while the leader ranks them;
//    after one more barrier the leader orders the logits and computes the softmax.
// A row whose certificate (fast selection) finds groups to re-score is refined in place by every
// CTA (those groups scored exactly, the winners ranked again), then rescored.  A row the radix
// certificate flags, or whose pool is degenerate, or that the in-place refinement cannot settle, is
// selected again by the leader alone with the block selection (select_row: exact, with refinement
// and full rescan) and then rescored.
//
// Cluster barriers are hardware barriers.  Each path has a fixed sequence of them, and every CTA of
// a cluster takes the same path: its decisions come from the same data in every CTA (the fast
// selection, the in-place refinement) or from state combined across the cluster (the radix
// selection), so the barriers always complete.
#include <cooperative_groups.h>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "select.cuh"
#include "sm100.cuh"

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
  alignas(16) unsigned long long cmp[HC_BOUND];  // fast selection: the candidates, compacted
  uint32_t cnt[16];                              // fast selection: each CTA's candidate count
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
  int* status;  // workspace status word
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
      if (c < d) acc = Elem<T>::dot16(*reinterpret_cast<const uint4*>(hs + c), wa[q], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// The same dot product with the W row in shared memory (lane-strided 16-byte chunks in row_dot's
// order, fp32 fused multiply-adds, the same xor reduction): bit-identical to row_dot.
template <typename T>
__device__ __forceinline__ float row_dot_smem(const T* wrow, int d, const T* hs, int lane) {
  constexpr int PER = Elem<T>::PER16;
  float acc = 0.f;
  for (int c = lane * PER; c < d; c += 32 * PER)
    acc = Elem<T>::dot16(*reinterpret_cast<const uint4*>(hs + c), *reinterpret_cast<const uint4*>(wrow + c), acc);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// Dynamic shared memory layout: control block, h, then the block selection's area (leader only).
__host__ __device__ constexpr size_t hc_h_offset() { return align_up(sizeof(HeadCtl), 128); }
__host__ __device__ constexpr size_t hc_fb_offset(int d, int elem) {
  return hc_h_offset() + align_up((size_t)d * elem, 128);
}
__host__ __device__ constexpr size_t hc_smem_bytes(int d, int elem, int n_groups) {
  return hc_fb_offset(d, elem) + sel::select_smem_bytes(n_groups);
}

constexpr int HC_GK = HC_MAX_GROUPS / HC_THREADS;  // group keys per thread in the fast selection
constexpr int HC_FBITS = 11;
constexpr int HC_FBINS = 1 << HC_FBITS;  // the fast selection's histogram
constexpr int HC_FBPT = HC_FBINS / HC_THREADS;
static_assert(HC_FBPT == 8, "each thread scans two 16-byte vectors of bins");
constexpr int HC_CG = 384;  // candidate groups of the fast selection (K <= 256 plus the boundary bin)
constexpr uint64_t HC_WAIT_NS = 2000000000ull;  // limit of the wait for h's bulk copy (2 s)

// Block-local state of the fast selection.
struct FastShared {
  alignas(16) uint32_t hist[HC_FBINS];
  alignas(16) unsigned long long ce[2 * HC_CG];  // the candidate entries, packed key << 32 | ~id
  uint32_t smax[HC_MAX_K];                       // the largest key of each of the K subsets
  int32_t cg[HC_CG];                             // the candidate groups
  uint32_t cm3[HC_CG];                           // their third-best keys (certificate)
  uint32_t wsc[HC_WARPS];
  uint32_t bb;     // the boundary bin
  uint32_t n_ent;  // candidate entries
  uint32_t n_cg;   // candidate groups (for the refinement)
  int refine;      // the certificate flagged a group: the row is refined after the fast path
  uint64_t wbar[HC_WARPS];  // each warp's first winner's W row, bulk-copied into the selection area
};

// 16-byte asynchronous copy global -> shared, read through L2 (completed by cp.async.wait_all).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_u32(dst)), "l"(src) : "memory");
}

// Bounded wait for a bulk copy into shared memory; a copy that does not land in time raises
// DH_ERR_TIMEOUT in the status word, and the thread waits once more so that the copy has landed
// (or the second limit has passed) before the CTA reuses or releases the memory.
__device__ __forceinline__ bool wait_copy(uint64_t* bar, int* status) {
  if (sm100::mbar_wait(bar, 0, HC_WAIT_NS)) return true;
  if ((threadIdx.x & 31) == 0) atomicOr(status, 1 << DH_ERR_TIMEOUT);
  sm100::mbar_wait(bar, 0, HC_WAIT_NS);
  return false;
}

// In-place refinement of a row the fast selection's certificate flags (in every CTA, from the fast
// selection's winners, candidate groups and tau): the flagged groups' members are scored exactly
// with the block selection's score_groups, and the K winners are ranked again among the winners
// outside those groups and the flagged groups' members at or above tau.  That is select_row's own
// refinement on the same candidates, so the winners are the same.  `area` is the selection area,
// laid out as select_row's Shared block (its W-row slots must have landed).  Returns false where
// select_row would settle the row another way (more than RMAX flagged groups, or a candidate count
// outside [K, CMAX]); the block selection then takes the row.
template <typename T>
__device__ bool refine_in_place(const HeadParams& p, HeadCtl& my, const FastShared& fs, unsigned char* area, int b,
                                uint32_t n_cg, uint32_t tau) {
  sel::Shared& sh = *reinterpret_cast<sel::Shared*>(area);
  const int K = p.K, r = p.r;
  for (int w = threadIdx.x; w < (int)sel::BITMAP_WORDS; w += HC_THREADS) sh.bitmap[w] = 0u;
  if (p.acc) {
    const unsigned long long* acc_row = p.acc + (size_t)b * r;
    for (int j = threadIdx.x; j < r; j += HC_THREADS) sh.t[j] = acc_to_t<T>(acc_row, p.B * r, j);
  } else {
    const T* t_row = static_cast<const T*>(p.t) + (size_t)b * r;
    for (int j = threadIdx.x; j < r; j += HC_THREADS) sh.t[j] = Elem<T>::to_f(t_row[j]);
  }
  if (threadIdx.x == 0) sh.nref = 0u;
  __syncthreads();
  for (uint32_t i = threadIdx.x; i < n_cg; i += HC_THREADS) {
    if (fs.cm3[i] >= tau) {
      const int g = fs.cg[i];
      const uint32_t pos = atomicAdd(&sh.nref, 1u);
      if (pos < (uint32_t)sel::RMAX) sh.rg[pos] = g;
      atomicOr(&sh.bitmap[g >> 5], 1u << (g & 31));
    }
  }
  __syncthreads();
  const int nref = (int)sh.nref;
  if (nref > sel::RMAX) return false;
  const T* V = static_cast<const T*>(p.V);
  for (int i = 0; i < nref; i += sel::SG_BATCH)
    sel::score_groups(sh.t, V, r, p.vocab, sh.rg + i, min(sel::SG_BATCH, nref - i), sh.rs + i * GROUP,
                      reinterpret_cast<float*>(sh.hist));
  unsigned long long* cp = reinterpret_cast<unsigned long long*>(sh.hist);  // the candidates, packed
  constexpr int CMAX = sel::HIST_BINS / 2;
  if (threadIdx.x == 0) sh.cnt = 0u;
  __syncthreads();
  for (int k0 = 0; k0 < K; k0 += HC_THREADS) {
    const int k = k0 + (int)threadIdx.x;
    bool take = false;
    unsigned long long e = 0ull;
    if (k < K) {
      e = my.sp[k];
      const uint32_t g = (~(uint32_t)e) / GROUP;
      take = !((sh.bitmap[g >> 5] >> (g & 31)) & 1u);
    }
    const uint32_t pos = sel::warp_append(take, &sh.cnt);
    if (take && pos < (uint32_t)CMAX) cp[pos] = e;
  }
  for (int e0 = 0; e0 < nref * GROUP; e0 += HC_THREADS) {
    const int e = e0 + (int)threadIdx.x;
    bool take = false;
    uint32_t key = 0u;
    int c = 0;
    if (e < nref * GROUP) {
      c = sh.rg[e / GROUP] * GROUP + (e % GROUP);
      key = fkey(sh.rs[e]);
      take = c < p.vocab && key >= tau;
    }
    const uint32_t pos = sel::warp_append(take, &sh.cnt);
    if (take && pos < (uint32_t)CMAX) cp[pos] = pack(key, (uint32_t)c);
  }
  __syncthreads();
  const int n = (int)sh.cnt;
  if (n < K || n > CMAX) return false;
  int P = 1;
  while (P < 32 && n * (2 * P) <= HC_THREADS) P <<= 1;
  for (int base = 0; base < n * P; base += HC_THREADS) {
    const int t = base + (int)threadIdx.x;
    const int i = t / P, h = t % P;
    unsigned long long pi;
    const int rank = sel::rank_by_count(cp, n, P, i, h, &pi);
    if (i < n && h == 0 && rank < K) my.sp[rank] = pi;
  }
  __syncthreads();
  return true;
}

// Fast selection from the groups' best keys (written by the small-batch scores kernel).  Every CTA
// selects the row's K winners itself, from every group's best key and the records of a few groups,
// so the CTAs exchange nothing before the exact logits:
//  1. A lower bound lo on theta, the K-th largest group best: the keys are split into K disjoint
//     subsets (thread t's keys form part of subset t mod K); each subset's largest key is a
//     distinct key, so K keys reach the smallest of them.  On random rows about the top tenth
//     of the keys reach lo.
//  2. One histogram of the keys at or above lo, in bins of 2^sh keys over [lo, largest key]
//     (monotone in the key), and a block scan from the top: the boundary bin bb holds theta, and
//     theta' = lo + bb 2^sh <= theta.  The K groups whose bests reach theta put K pool entries at
//     or above theta', so every entry of the pool's top K is at or above theta', and only groups
//     whose best reaches theta' (the candidate groups: about K) hold such entries.
//  3. The candidate groups' records (copied into shared memory through L2 as soon as lo is known,
//     for every group whose best reaches lo, while the histogram is built): their entries at or
//     above theta' are collected (their W rows start towards L2, each group's by one CTA) and ranked by counting,
//     which also orders the K winners.  Certificate: a group whose third score reaches tau (the
//     K-th winner's) may hide a member of the top K; only a candidate group can (its third score is
//     at most its best).
//  4. Each CTA scores winners k = warp x CTAs + rank and writes them in rank order; the logits go to
//     the leader.  One cluster barrier; the leader computes the softmax.
// Returns true when the row must take the leader's exact selection instead: fewer than K groups
// hold entries, more than HC_CG groups reach theta', or the certificate flags a group.  Every CTA
// takes the same decision from the same data.
template <typename T, int HC_CTAS>
__device__ __forceinline__ bool head_fast(const HeadParams& p, cg::cluster_group& cl, HeadCtl& my, FastShared& fs,
                                          const T* hs, uint64_t* hbar, T* slots, int b, const uint32_t (&y)[HC_GK]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = p.K;
  const int crank = (int)cl.block_rank();
  const bool leader = crank == 0;
  const GroupRec* rrow = p.recs + (size_t)b * p.n_groups;
  // ---- 1. lo: the smallest of the K subsets' largest keys (an empty subset leaves it 0)
  uint32_t ymax = 0u;
#pragma unroll
  for (int q = 0; q < HC_GK; ++q) ymax = max(ymax, y[q]);
  if (ymax) atomicMax(&fs.smax[threadIdx.x % K], ymax);
  __syncthreads();
  uint32_t lo = 0xFFFFFFFFu, hi = 0u;
  for (int s = lane; s < K; s += 32) {
    const uint32_t v = fs.smax[s];
    lo = min(lo, v);
    hi = max(hi, v);
  }
  lo = max(__reduce_min_sync(0xFFFFFFFFu, lo), 1u);  // key 0 marks an empty group
  hi = __reduce_max_sync(0xFFFFFFFFu, hi);
  // the records of the groups whose bests reach lo (every candidate group among them; about a
  // tenth of the row) start towards the selection area now, indexed by group, while the
  // histogram is built
  GroupRec* recs_s = reinterpret_cast<GroupRec*>(slots);
#pragma unroll
  for (int q = 0; q < HC_GK; ++q) {
    const int g = (int)threadIdx.x + q * HC_THREADS;
    if (y[q] && y[q] >= lo) cp_async16(&recs_s[g], rrow + g);
  }
  // ---- 2. histogram of the keys in [lo, hi], bins of 2^sh keys
  const uint32_t span = hi >= lo ? hi - lo : 0u;
  const int sh = max(0, (32 - __clz((int)span)) - HC_FBITS);
  if (hi >= lo)
#pragma unroll
    for (int q = 0; q < HC_GK; ++q)
      if (y[q] >= lo) atomicAdd(&fs.hist[(y[q] - lo) >> sh], 1u);
  __syncthreads();
  // thread t scans bins [HC_FBINS - 8(t + 1), HC_FBINS - 8t), from the top
  const int base = HC_FBINS - HC_FBPT * ((int)threadIdx.x + 1);
  const uint4 h0 = *reinterpret_cast<const uint4*>(&fs.hist[base]);
  const uint4 h1 = *reinterpret_cast<const uint4*>(&fs.hist[base + 4]);
  const uint32_t c[HC_FBPT] = {h1.w, h1.z, h1.y, h1.x, h0.w, h0.z, h0.y, h0.x};  // bins base+7 .. base
  uint32_t own = 0u;
#pragma unroll
  for (int j = 0; j < HC_FBPT; ++j) own += c[j];
  uint32_t incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) fs.wsc[warp] = incl;
  __syncthreads();
  uint32_t before = 0u, total = 0u;
#pragma unroll
  for (int w = 0; w < HC_WARPS; ++w) {
    before += w < warp ? fs.wsc[w] : 0u;
    total += fs.wsc[w];
  }
  uint32_t run = before + incl - own;  // keys in the bins above this thread's
#pragma unroll
  for (int j = 0; j < HC_FBPT; ++j) {
    if (run < (uint32_t)K && run + c[j] >= (uint32_t)K) fs.bb = (uint32_t)(base + HC_FBPT - 1 - j);
    run += c[j];
  }
  if (threadIdx.x == 0) fs.n_ent = 0u;
  __syncthreads();
  const bool ok = hi >= lo && total >= (uint32_t)K;  // else fewer than K groups hold entries
  const uint32_t theta = ok ? lo + (fs.bb << sh) : 0xFFFFFFFFu;
  // ---- 3. the candidate groups (block scan for their positions), their records, their entries
  uint32_t mine = 0u;
#pragma unroll
  for (int q = 0; q < HC_GK; ++q) mine += (y[q] && y[q] >= theta) ? 1u : 0u;
  incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) fs.wsc[warp] = incl;
  __syncthreads();
  before = 0u;
  total = 0u;
#pragma unroll
  for (int w = 0; w < HC_WARPS; ++w) {
    before += w < warp ? fs.wsc[w] : 0u;
    total += fs.wsc[w];
  }
  uint32_t pos = before + incl - mine;
#pragma unroll
  for (int q = 0; q < HC_GK; ++q) {
    if (y[q] && y[q] >= theta) {
      if (pos < (uint32_t)HC_CG) fs.cg[pos] = (int)threadIdx.x + q * HC_THREADS;
      ++pos;
    }
  }
  const uint32_t n_cg = total;
  bool fall = !ok || n_cg > (uint32_t)HC_CG;
  if (threadIdx.x == 0) {
    fs.n_cg = n_cg;
    fs.refine = 0;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (!fall) {
    for (uint32_t i = threadIdx.x; i < n_cg; i += HC_THREADS) {
      const int g = fs.cg[i];
      const GroupRec r = recs_s[g];
      fs.cm3[i] = fkey(r.m3);
      const uint32_t o1 = r.offs & 0xFFu, o2 = (r.offs >> 8) & 0xFFu;
      const uint32_t k2 = o2 != NO_OFFSET ? fkey(r.m2) : 0u;
      const bool two = k2 && k2 >= theta;
      const uint32_t slot = atomicAdd(&fs.n_ent, two ? 2u : 1u);  // at most 2 n_cg <= 2 HC_CG entries
      const uint32_t v1 = (uint32_t)g * GROUP + o1, v2 = (uint32_t)g * GROUP + o2;
      fs.ce[slot] = pack(fkey(r.m1), v1);
      if (two) fs.ce[slot + 1] = pack(k2, v2);
      if (g % HC_CTAS == crank) {  // each candidate group's W rows towards L2, by one CTA
        const T* W = static_cast<const T*>(p.W);
        const uint32_t row_bytes = (uint32_t)(p.d * sizeof(T));
        if (v1 < (uint32_t)p.vocab) prefetch_l2(W + (size_t)v1 * p.d, row_bytes);
        if (two && v2 < (uint32_t)p.vocab) prefetch_l2(W + (size_t)v2 * p.d, row_bytes);
      }
    }
  }
  __syncthreads();
  // ---- 4. rank the entries: the K winners in order; the certificate
  bool flag = false;
  if (!fall) {
    const int n_ent = (int)fs.n_ent;  // at least n_cg >= K
    int P = 1;
    while (P < 32 && n_ent * (2 * P) <= HC_THREADS) P <<= 1;
    for (int base2 = 0; base2 < n_ent * P; base2 += HC_THREADS) {
      const int t = base2 + (int)threadIdx.x;
      const int i = t / P, hh = t % P;
      unsigned long long pi;
      const int rank = sel::rank_by_count(fs.ce, n_ent, P, i, hh, &pi);
      if (i < n_ent && hh == 0 && rank < K) my.sp[rank] = pi;
    }
    __syncthreads();
  }
  // each warp's first winner's W row starts into the warp's slot of the selection area now (a bulk
  // copy), ahead of the certificate and the cluster wait
  const uint32_t row_bytes = (uint32_t)(p.d * sizeof(T));
  const int n_slot = min(HC_WARPS, (int)(sel::select_smem_bytes(p.n_groups) / row_bytes));
  const int k_first = warp * HC_CTAS + crank;
  bool slotted = false;
  if (!fall && warp < n_slot && k_first < K) {
    const int v = (int)(~(uint32_t)my.sp[k_first]);
    slotted = v >= 0 && v < p.vocab;
    if (slotted && lane == 0) {
      sm100::fence_proxy_async_smem();  // the records read from this area are done with (barriers above)
      sm100::mbar_arrive_expect_tx(&fs.wbar[warp], row_bytes);
      sm100::bulk_load(slots + (size_t)warp * p.d, static_cast<const T*>(p.W) + (size_t)v * p.d, row_bytes,
                       &fs.wbar[warp]);
    }
  }
  if (!fall) {
    const uint32_t tau = (uint32_t)(my.sp[K - 1] >> 32);
    for (uint32_t i = threadIdx.x; i < n_cg; i += HC_THREADS) flag |= fs.cm3[i] >= tau;
  }
  // fall is uniform over the block (from shared state): one block-wide vote, on the certificate; a
  // flagged row leaves the fast path and is refined by the caller (refine_in_place)
  if (!fall && __syncthreads_or(flag)) {
    if (threadIdx.x == 0) fs.refine = 1;
    fall = true;
  }
  // every CTA has started (the arrive at its start) before any CTA writes into the leader
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (fall) {
    if (slotted) wait_copy(&fs.wbar[warp], p.status);  // landed before the selection area is reused
    __syncthreads();
    return true;
  }
  // ---- 5. exact logits of winners k = warp x CTAs + rank, in rank order; into the leader
  wait_copy(hbar, p.status);
  float* zl = cl.map_shared_rank(&my.z[0], 0u);
  for (int k = k_first; k < K; k += HC_CTAS * HC_WARPS) {
    const unsigned long long e = my.sp[k];
    const int v = (int)(~(uint32_t)e);
    const bool okv = v >= 0 && v < p.vocab;
    float acc = 0.f;
    if (k == k_first && slotted) {
      wait_copy(&fs.wbar[warp], p.status);
      acc = row_dot_smem<T>(slots + (size_t)warp * p.d, p.d, hs, lane);
    } else if (okv) {
      acc = row_dot<T>(static_cast<const T*>(p.W), v, p.d, hs, lane);
    }
    const float z = okv ? acc : __int_as_float(0x7FC00000);
    if (lane == 0) {
      p.idx_out[(size_t)b * K + k] = v;
      p.score_out[(size_t)b * K + k] = fkey_inv((uint32_t)(e >> 32));
      p.logits[(size_t)b * K + k] = z;
      zl[k] = z;
    }
  }
  cluster_sync_all();
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

  __shared__ FastShared fs;
  __shared__ uint64_t hbar;  // h's bulk copy into shared memory
  if (p.gkeys) {
    for (int i = threadIdx.x; i < HC_FBINS; i += HC_THREADS) fs.hist[i] = 0u;
    for (int i = threadIdx.x; i < HC_MAX_K; i += HC_THREADS) fs.smax[i] = 0u;
  }
  // zero this CTA's control block; the barrier's wait (below) makes the leader's visible
  for (int i = threadIdx.x; i < HC_BINS; i += HC_THREADS) my.hist[0][i] = my.hist[1][i] = 0u;
  if (threadIdx.x == 0) {
    my.kmin = 0xFFFFFFFFu;
    my.kmax = 0u;
    my.n_above = my.n_bound = my.nref = 0u;
    // h does not depend on the previous kernels: one bulk copy, waited for before the first dot
    // product (every path waits, so no copy is in flight when the CTA exits)
    const uint32_t h_bytes = (uint32_t)(p.d * sizeof(T));
    sm100::mbar_init(&hbar, 1);
    if (p.gkeys)
      for (int w = 0; w < HC_WARPS; ++w) sm100::mbar_init(&fs.wbar[w], 1);
    sm100::fence_barrier_init();
    sm100::mbar_arrive_expect_tx(&hbar, h_bytes);
    sm100::bulk_load(hs, static_cast<const T*>(p.h) + (size_t)b * p.d, h_bytes, &hbar);
  }
  __syncthreads();
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  // the next kernel may launch now: every kernel of the library that follows waits
  // (griddepcontrol.wait) for this grid before it reads anything, so its launch latency is hidden
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the records come from the scores kernel

  bool fallback = false;
  if (p.gkeys) {
    // every group's best key of the row
    uint32_t gk[HC_GK];
    const uint32_t* grow = p.gkeys + (size_t)b * n_groups;
#pragma unroll
    for (int q = 0; q < HC_GK; ++q) {
      const int g = (int)threadIdx.x + q * HC_THREADS;
      gk[q] = g < n_groups ? __ldcg(grow + g) : 0u;
    }
    if (!head_fast<T, HC_CTAS>(p, cl, my, fs, hs, &hbar, reinterpret_cast<T*>(fb), b, gk)) return;
    fallback = true;
  } else {
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
    wait_copy(&hbar, p.status);
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
  // A row the fast selection's certificate flagged is refined in place by every CTA (its W-row slots
  // have landed); each reaches the same winners from the same data, as it reached the same decision
  // to refine, and scores its share of them.
  if (p.gkeys && fs.refine &&
      refine_in_place<T>(p, my, fs, fb, b, fs.n_cg, (uint32_t)(my.sp[K - 1] >> 32))) {
    wait_copy(&hbar, p.status);
    float* zl = cl.map_shared_rank(&my.z[0], 0u);
    for (int k = warp * HC_CTAS + (int)crank; k < K; k += HC_CTAS * HC_WARPS) {
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
    if (!leader) return;
    if (acc_row)  // zeroed for the next call (select_row does it on the other branch)
      for (int j = threadIdx.x; j < p.r; j += HC_THREADS)
#pragma unroll
        for (int q = 0; q < ACC_COPIES; ++q) acc_row[(size_t)q * BR + j] = 0ull;
    if (p.probs && warp == 0) warp_softmax(my.z, K, p.probs + (size_t)b * K);
    return;
  }
  // otherwise the leader selects the row alone: exact, with refinement or a full rescan as needed
  if (leader)
    sel::select_row<T, HC_THREADS>(fb, rrow, t_row, acc_row, BR, static_cast<const T*>(p.V), p.r, p.vocab, K,
                                   p.idx_out + (size_t)b * K, p.score_out + (size_t)b * K);
  cluster_sync_all();

  // ---------------------------------------------------------------- exact logits and softmax
  const int32_t* cand = p.idx_out + (size_t)b * K;
  wait_copy(&hbar, p.status);
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
  cudaError_t e = carveout_max_shared(reinterpret_cast<const void*>(k_head_cl<T, CTAS>), c.device);
  if (e != cudaSuccess) return e;
  prof_before("head_cluster", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_head_cl<T, CTAS>, p);
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

// Largest K for which the fused head is chosen by default.  Above it the two kernels are as fast or
// faster (µs per call in CUDA graphs at d 5120, vocab 151936, fused against two kernels: 8 x 192:
// 40.9 / 40.5; at K = 256, 33.8 / 32.2 at B = 2 and 47.1 / 46.1 at B = 8), while up to K = 128 the
// fused head is as fast or faster at every batch that fits one wave (3 x 96: 24.3 / 28.6; 8 x 128:
// 33.9 / 34.7; 16 x 128: 39.3 / 40.0).
constexpr int HC_AUTO_MAX_K = 128;

// Cluster size for B rows: 16 CTAs when all B clusters of 16 run at once, else 8 when all B
// clusters of 8 do, else 4 when all B clusters of 4 do, for up to 8192 (row, candidate) pairs with
// K <= 64 and 2048 above, else 2 when all B clusters of 2 do and K <= 64, else 0 (the batch goes to
// the selection and rescoring kernels); 0 as well above HC_AUTO_MAX_K candidates unless
// DH_FORCE_HEAD=cluster.  Small clusters score several candidates per warp, one after another.
// Measured per call in CUDA graphs at d 5120, vocab 151936, fused against two kernels, with 4 CTAs:
// 33 x 64: 30.9 / 39.6 µs; 36 x 64: 32.0 / 39.7; but 24 x 128: 43.8 / 42.1; with 2 CTAs: 40 x 64:
// 36.9 / 40.6; 64 x 64: 38.2 / 42.6; 76 x 64: 43.8 / 48.3; but 40 x 128: 51.7 / 47.8.  Clusters in
// two waves lose (4 CTAs, 64 x 128: 58.1 / 52.5).  The device's capacities are queried once per
// device and element type (set-up calls: shared memory limit, the non-portable size, the occupancy
// query).  The DH_HEAD_CTAS switch (8, 4 or 2) skips the larger forms (tests).
template <typename T>
int choose_ctas(const Ctx& c, int B, int K, int d, int n_groups) {
  const size_t smem = hc_smem_bytes(d, (int)sizeof(T), n_groups);
  static std::mutex mu;
  static int cap[64][4] = {};  // [device]: clusters of 16, 8, 4 and 2 at once, +1 (0: not queried)
  static size_t smem_at[64] = {};
  if (c.device < 0 || c.device >= 64) return 0;
  int n16, n8, n4, n2;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (cap[c.device][0] == 0 || smem_at[c.device] < smem) {
      cap[c.device][0] = clusters_at_once<T, 16>(c.device, smem) + 1;
      cap[c.device][1] = clusters_at_once<T, 8>(c.device, smem) + 1;
      cap[c.device][2] = clusters_at_once<T, 4>(c.device, smem) + 1;
      cap[c.device][3] = clusters_at_once<T, 2>(c.device, smem) + 1;
      smem_at[c.device] = smem;
      (void)cudaGetLastError();  // a refused query leaves no sticky error behind
    }
    n16 = cap[c.device][0] - 1;
    n8 = cap[c.device][1] - 1;
    n4 = cap[c.device][2] - 1;
    n2 = cap[c.device][3] - 1;
  }
  const bool forced = tuning().head_cluster;  // wherever it fits, whatever the candidates
  if (K > HC_AUTO_MAX_K && !forced) return 0;
  const int most = tuning().head_ctas_max;
  if (most >= 16 && B <= n16) return 16;
  if (most >= 8 && B <= n8) return 8;
  if (most >= 4 && B <= n4 && (forced || (long long)B * K <= (K <= 64 ? 8192 : 2048))) return 4;
  if (most >= 2 && B <= n2 && (forced || K <= 64)) return 2;
  return 0;
}

template <typename T>
cudaError_t run(const Ctx& c, const HeadParams& p, int ctas) {
  const size_t smem = hc_smem_bytes(p.d, (int)sizeof(T), p.n_groups);
  if (ctas == 4) return launch<T, 4>(c, p, smem);
  if (ctas == 2) return launch<T, 2>(c, p, smem);
  return ctas == 16 ? launch<T, 16>(c, p, smem) : launch<T, 8>(c, p, smem);
}

}  // namespace

int head_cluster_ctas(const Ctx& c, int B, int K, int d, int vocab, int dtype) {
  // a wave of clusters holds at most one row per 2 SMs: larger batches need no query
  if (B > c.num_sms / 2) return 0;
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  return dtype == DH_BF16 ? choose_ctas<__nv_bfloat16>(c, B, K, d, n_groups)
                          : choose_ctas<float>(c, B, K, d, n_groups);
}

bool head_cluster_supported(int B, int d, int vocab, int K, int dtype) {
  const int n_groups = (vocab + GROUP - 1) / GROUP;
  const size_t smem = hc_smem_bytes(d, dtype == DH_BF16 ? 2 : 4, n_groups);
  return B >= 1 && K <= HC_MAX_K && n_groups <= HC_MAX_GROUPS && n_groups <= sel::CACHE_GROUPS &&
         d <= 8192 && smem <= 200 * 1024;
}

cudaError_t launch_head_cluster(const Ctx& c, int ctas, const GroupRec* recs, const uint32_t* gkeys,
                                unsigned long long* acc, const void* t, const void* V, const void* h, const void* W,
                                int B, int d, int r, int vocab, int K, int dtype, int32_t* idx_out, float* score_out,
                                float* logits, float* probs, int* status) {
  if (ctas != 2 && ctas != 4 && ctas != 8 && ctas != 16) return cudaErrorInvalidValue;
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
  p.status = status;
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, p, ctas);
  return run<float>(c, p, ctas);
}

}  // namespace dh
