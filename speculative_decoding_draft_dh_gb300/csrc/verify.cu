// Chain verification at positive temperature: speculative sampling over L drafted tokens per request.
//
// EAGLE-4 summary page, section "Distribution preservation has algorithmic and implementation
// conditions": at positive temperature the target verifies the drafted tokens and a rejection
// correction keeps the target's output distribution; each round's depth is fixed before the round.
// For a chain this is standard speculative sampling (Leviathan, Kalman and Matias 2023; Chen et al.
// 2023): with p_i = softmax(l_i / T) the target's distribution after the prefix and x_0..x_{i-1},
// and q_i the draft's distribution (K candidate ids with their probabilities), token i is accepted
// when u_i < p_i(x_i) / q_i(x_i); after the first rejection at n the emitted token is drawn from
// max(0, p_n - q_n), after L acceptances from p_L, by inverse CDF in vocabulary order with the
// uniform w_b.
//
// k_verify_stats (one block per target row, HBM-bound: the whole step's traffic): each warp reads
//   segments of 32 lanes x SEG_VECS 16-byte vectors (1024 bf16 or 512 fp32 ids, lane l holding
//   vectors l, l + 32, ... so every load is coalesced), and writes per segment its maximum of
//   z = l * log2(e) / T and the sum of 2^(z - max); one warp reduction pair per segment of 1024
//   ids keeps the shuffle chains short against the 2^x evaluations.  The warps stream the
//   (row, segment) items of all rows grid-stride, so no wave of blocks is left half empty.  Every
//   target row is needed: which row the chain stops at is known only after all acceptance tests.
// k_verify_walk (one block per request): warp i combines row i's segment pairs into the row's
//   maximum and sum (fixed order) and evaluates the acceptance test of position i; the first
//   failure gives n.  The draw's weights are per segment: the segment sums rescaled to
//   the row's maximum, minus min(p, q) at the candidates of position n (none after L acceptances).
//   A block scan over the segments in vocabulary order finds the segment where the running sum
//   crosses w_b times the total; one warp then recomputes that segment's weights id by id, scans
//   them and finds the token.  All sums run in a fixed order, so results repeat bit for bit.
#include "dh_internal.cuh"

namespace dh {
namespace {

constexpr int VS_THREADS = 512;
constexpr int SEG_VECS = 4;    // 16-byte vectors per lane in a segment
constexpr int VW_THREADS = 256;
constexpr int VW_MAX_L = 64;   // drafted tokens per request
constexpr float LOG2E = 1.4426950408889634f;

// 2^x on the special-function unit, subnormal results flushed to zero (one instruction; the terms
// it flushes are below 2^-126 of the row maximum's and do not move a sum).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (m, s) <- the pair of the union: max and the sum rescaled to it (an empty side has m = -inf, s = 0).
__device__ __forceinline__ void combine(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;
  s = (m == -INFINITY ? 0.f : s * ex2(m - mn)) + (m2 == -INFINITY ? 0.f : s2 * ex2(m2 - mn));
  m = mn;
}

template <typename T>
__global__ void __launch_bounds__(VS_THREADS) k_verify_stats(const T* __restrict__ logits, int vocab, float c,
                                                           int n_seg, int n_items, float2* __restrict__ seg_stats) {
  constexpr int PER = Elem<T>::PER16;
  constexpr int SEG = 32 * PER * SEG_VECS;
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (VS_THREADS / 32);
  const int w0 = blockIdx.x * (VS_THREADS / 32) + (threadIdx.x >> 5);
  // launched with programmatic dependent launch: the logits may come from the kernel before this
  // one, which may also still read the workspace, so nothing is loaded or stored before the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the loads of item g (row g / n_seg, segment g % n_seg): its SEG_VECS vectors per lane
  auto load = [&](int g, uint4 (&u)[SEG_VECS]) {
    const int row = g / n_seg, sgi = g - row * n_seg;
#pragma unroll
    for (int v = 0; v < SEG_VECS; ++v) {
      const int id = sgi * SEG + (v * 32 + lane) * PER;
      u[v] = (g < n_items && id < vocab) ? ld_nc_v4(logits + (size_t)row * vocab + id) : make_uint4(0, 0, 0, 0);
    }
  };
  // the walk kernel's blocks may launch as these retire (they wait for the statistics themselves)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  uint4 cur[SEG_VECS], nxt[SEG_VECS];
  load(w0, cur);
  for (int g = w0; g < n_items; g += nw) {
    load(g + nw, nxt);  // the next item's loads are in flight while this one is reduced
    const int sgi = g % n_seg;
    // the maximum of the raw logits (the scale c > 0 keeps the order), then
    // sum 2^(l c - m c) with one fused multiply-add per term; only the last segment of a row has ids
    // past the vocabulary, whose terms are left out
    float z[SEG_VECS][PER];
    float m = -INFINITY;
    const bool full = (sgi + 1) * SEG <= vocab;
#pragma unroll
    for (int v = 0; v < SEG_VECS; ++v) {
      Elem<T>::unpack(cur[v], z[v]);
      if (!full) {
        const int id = sgi * SEG + (v * 32 + lane) * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) z[v][e] = id < vocab ? z[v][e] : -INFINITY;
      }
#pragma unroll
      for (int e = 0; e < PER; ++e) m = fmaxf(m, z[v][e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float mc = m * c;
    float sum = 0.f;
    if (m != -INFINITY)
#pragma unroll
      for (int v = 0; v < SEG_VECS; ++v)
#pragma unroll
        for (int e = 0; e < PER; ++e) sum += ex2(fmaf(z[v][e], c, -mc));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane == 0) seg_stats[g] = make_float2(m == -INFINITY ? m : mc, sum);
#pragma unroll
    for (int v = 0; v < SEG_VECS; ++v) cur[v] = nxt[v];
  }
}

// A row's (max, sum) from its segments' pairs, by one warp: lane l combines segments l, l + 32, ...
// in order, then the lanes' pairs combine in a fixed butterfly order (every lane gets the result).
__device__ __forceinline__ float2 row_pair(const float2* seg, int n_seg) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY, s = 0.f;
  for (int i = lane; i < n_seg; i += 32) {
    const float2 q = seg[i];
    combine(m, s, q.x, q.y);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o), s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
    // the lower lane's pair first, so both lanes compute the same value
    if (lane & o) {
      float mm = m2, ss = s2;
      combine(mm, ss, m, s);
      m = mm; s = ss;
    } else {
      combine(m, s, m2, s2);
    }
  }
  return make_float2(m, s);
}

struct WalkParams {
  const void* logits;
  const int32_t* cand_idx;
  const float* cand_prob;
  const int32_t* draft;
  const float* u_accept;
  const float* u_sample;
  const float2* seg_stats;
  int L, vocab, K, n_seg;
  float c;
  int32_t* n_accept;
  int32_t* token;
};

template <typename T>
__device__ __forceinline__ float logit_at(const T* row, int v) {
  return Elem<T>::to_f(row[v]);
}

// Exclusive scan of x over the block in thread order (warp shuffles, then the warp totals): a
// fixed order, so it repeats bit for bit.  Returns this thread's exclusive prefix and sets *total.
__device__ __forceinline__ float block_excl_scan(float x, float* wtot, float* total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  float before = 0.f, all = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += wtot[w];
    all += wtot[w];
  }
  __syncthreads();  // wtot may be reused by the next scan
  *total = all;
  return before + incl - x;
}

template <typename T>
__global__ void __launch_bounds__(VW_THREADS) k_verify_walk(WalkParams p) {
  // the next kernel may launch as these blocks start (every library kernel launched with
  // programmatic dependent launch waits for this grid before it touches what it touches)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int PER = Elem<T>::PER16;
  constexpr int SEG = 32 * PER * SEG_VECS;
  constexpr int LANE_IDS = PER * SEG_VECS;  // ids of a segment per lane in the final rescan
  extern __shared__ float sw[];             // per-segment weights (n_seg)
  __shared__ int s_n, s_seg, s_last;
  __shared__ float s_corr[DH_MAX_K];   // -min(p, q) at each candidate id's first occurrence, else 0
  __shared__ int32_t s_cid[DH_MAX_K];  // the id at its first occurrence, else -1
  __shared__ float s_q[DH_MAX_K];      // q(v) summed over the id's occurrences (first occurrence)
  __shared__ float s_wtot[VW_THREADS / 32];
  __shared__ float s_local;
  __shared__ float2 s_row[VW_MAX_L + 1];  // each target row's (max, sum)
  __shared__ float s_qx[VW_MAX_L], s_lx[VW_MAX_L];  // q_i(x_i) and the logit of x_i in row i
  const int b = blockIdx.x;
  const int L = p.L, K = p.K, n_seg = p.n_seg;
  const T* rows = static_cast<const T*>(p.logits) + (size_t)b * (L + 1) * p.vocab;
  const float2* segs = p.seg_stats + (size_t)b * (L + 1) * n_seg;
  if (threadIdx.x == 0) { s_n = L; s_seg = 0x7FFFFFFF; s_last = -1; }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // before the wait (none of it depends on the statistics): warp i sums q_i(x_i) over the
  // candidate list and reads the logit of x_i
  for (int i = warp; i < L; i += VW_THREADS / 32) {
    const int x = p.draft[(size_t)b * L + i];
    const int32_t* ci = p.cand_idx + ((size_t)b * L + i) * K;
    const float* cq = p.cand_prob + ((size_t)b * L + i) * K;
    float qx = 0.f;
    for (int k = lane; k < K; k += 32)
      if (ci[k] == x) qx += cq[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qx += __shfl_xor_sync(0xFFFFFFFFu, qx, o);
    if (lane == 0) {
      const bool in_range = x >= 0 && x < p.vocab;
      s_qx[i] = in_range ? qx : 0.f;  // outside the vocabulary: accepted, as q(x) = 0
      s_lx[i] = in_range ? logit_at(rows + (size_t)i * p.vocab, x) : 0.f;
    }
  }
  // the statistics come from k_verify_stats (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // warp i combines row i's segment pairs, then takes the acceptance test of position i
  for (int i = warp; i <= L; i += VW_THREADS / 32) {
    const float2 rp = row_pair(segs + (size_t)i * n_seg, n_seg);
    if (lane == 0) {
      s_row[i] = rp;
      if (i < L) {
        const float qx = s_qx[i];
        const float px = ex2(s_lx[i] * p.c - rp.x) / rp.y;
        const bool accepted = qx <= 0.f || p.u_accept[(size_t)b * L + i] < px / qx;
        if (!accepted) atomicMin(&s_n, i);
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  const T* row = rows + (size_t)n * p.vocab;
  const float2 st = s_row[n];
  const float inv_s = 1.f / st.y;
  const float2* seg = segs + (size_t)n * n_seg;
  // the candidates of position n (none after L acceptances), staged in shared memory
  const int Kn = n < L ? K : 0;
  const int32_t* cidx = p.cand_idx + ((size_t)b * L + (n < L ? n : 0)) * K;
  const float* cprob = p.cand_prob + ((size_t)b * L + (n < L ? n : 0)) * K;
  for (int k = threadIdx.x; k < Kn; k += VW_THREADS) {
    s_cid[k] = cidx[k];
    s_q[k] = cprob[k];
  }
  __syncthreads();
  // -min(p(v), q(v)) at each id's first occurrence, with q(v) summed over the id's occurrences
  float corr_k = 0.f, q_k = 0.f;
  int id_k = -1;
  for (int k = threadIdx.x; k < Kn; k += VW_THREADS) {
    const int v = s_cid[k];
    bool first = v >= 0 && v < p.vocab;
    float q = 0.f;
    for (int k2 = 0; k2 < Kn && first; ++k2) {
      if (s_cid[k2] != v) continue;
      if (k2 < k) first = false;
      q += s_q[k2];
    }
    const float pv = first ? ex2(logit_at(row, v) * p.c - st.x) * inv_s : 0.f;
    id_k = first ? v : -1;
    corr_k = first ? -fminf(pv, q) : 0.f;
    q_k = q;
  }
  __syncthreads();  // every thread has read s_cid / s_q
  for (int k = threadIdx.x; k < Kn; k += VW_THREADS) {
    s_cid[k] = id_k;
    s_corr[k] = corr_k;
    s_q[k] = q_k;
  }
  __syncthreads();
  // per-segment weights: the segment's p-mass plus the corrections of its candidates (in k order);
  // thread t owns segments [t * per, (t + 1) * per) and sums them in order
  const int per = (n_seg + VW_THREADS - 1) / VW_THREADS;
  const int sa = min(n_seg, (int)threadIdx.x * per), sb = min(n_seg, sa + per);
  auto seg_mass = [&](int s) {
    const float2 sg = seg[s];
    return sg.x == -INFINITY ? 0.f : sg.y * ex2(sg.x - st.x) * inv_s;
  };
  float tsum = 0.f;
  for (int s = sa; s < sb; ++s) {
    float w = seg_mass(s);
    for (int k = 0; k < Kn; ++k)
      if (s_cid[k] >= 0 && s_cid[k] / SEG == s) w += s_corr[k];
    w = fmaxf(w, 0.f);
    sw[s] = w;
    tsum += w;
  }
  float total;
  float excl = block_excl_scan(tsum, s_wtot, &total);
  // a zero residual (p_n = q_n on the candidates, no mass elsewhere): draw from p_n itself
  const bool use_p = !(total > 0.f);
  if (use_p) {
    tsum = 0.f;
    for (int s = sa; s < sb; ++s) {
      sw[s] = seg_mass(s);
      tsum += sw[s];
    }
    excl = block_excl_scan(tsum, s_wtot, &total);
  }
  const float target = p.u_sample[b] * total;
  // the segment where the running sum passes target: the thread whose range holds it walks its
  // segments (rounding may leave no claimant, or two: the lowest segment wins)
  int mine = -1, last_pos = -1;
  float before = 0.f;
  if (sb > sa && excl <= target && target < excl + tsum) {
    float run = excl;
    for (int s = sa; s < sb; ++s) {
      if (sw[s] > 0.f && run + sw[s] > target) { mine = s; before = run; break; }
      run += sw[s];
    }
  }
  for (int s = sa; s < sb; ++s)
    if (sw[s] > 0.f) last_pos = s;
  if (mine >= 0) atomicMin(&s_seg, mine);
  if (last_pos >= 0) atomicMax(&s_last, last_pos);
  __syncthreads();
  const bool claimed = s_seg != 0x7FFFFFFF;
  if (mine >= 0 && mine == s_seg) s_local = target - before;
  __syncthreads();
  // warp 0 recomputes the chosen segment's weights id by id (lane l: ids [l * LANE_IDS, (l + 1) *
  // LANE_IDS) of the segment, in order) and finds the token
  if (warp == 0) {
    const int sg = claimed ? s_seg : (s_last < 0 ? 0 : s_last);
    const float local = claimed ? s_local : INFINITY;  // unclaimed: the segment's last positive id
    const int id0 = sg * SEG + lane * LANE_IDS;
    float w[LANE_IDS];
#pragma unroll
    for (int v = 0; v < SEG_VECS; ++v) {
      const int id = id0 + v * PER;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (id < p.vocab) u = *reinterpret_cast<const uint4*>(row + id);
      Elem<T>::unpack(u, w + v * PER);
#pragma unroll
      for (int e = 0; e < PER; ++e) w[v * PER + e] = id + e < p.vocab ? ex2(w[v * PER + e] * p.c - st.x) * inv_s : 0.f;
    }
    if (!use_p) {
      for (int k = 0; k < Kn; ++k) {
        const int v = s_cid[k];  // first occurrences only
        if (v < id0 || v >= id0 + LANE_IDS) continue;
#pragma unroll
        for (int e = 0; e < LANE_IDS; ++e)
          if (id0 + e == v) w[e] = fmaxf(w[e] + s_corr[k], 0.f);
      }
    }
    float lsum = 0.f;
#pragma unroll
    for (int e = 0; e < LANE_IDS; ++e) lsum += w[e];
    float incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const float ex = incl - lsum;
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, lsum > 0.f && ex <= local && local < incl);
    int tok = -1;
    if (bm) {
      const int src = __ffs(bm) - 1;
      if (lane == src) {
        float run = ex;
#pragma unroll
        for (int e = 0; e < LANE_IDS; ++e) {
          if (tok < 0 && w[e] > 0.f && run + w[e] > local) tok = id0 + e;
          run += w[e];
        }
        if (tok < 0)
#pragma unroll
          for (int e = 0; e < LANE_IDS; ++e)
            if (w[e] > 0.f) tok = id0 + e;
      }
      tok = __shfl_sync(0xFFFFFFFFu, tok, src);
    } else {
      // past the segment's recomputed sum (rounding, or no claimant): its last positive id
      int lastv = -1;
#pragma unroll
      for (int e = 0; e < LANE_IDS; ++e)
        if (w[e] > 0.f) lastv = id0 + e;
      lastv = __reduce_max_sync(0xFFFFFFFFu, lastv);
      tok = lastv < 0 ? sg * SEG : lastv;
    }
    if (lane == 0) {
      p.n_accept[b] = n;
      p.token[b] = tok;
    }
  }
}

// Staged form of the walk (K <= VW_FK candidates per position and L K <= VW_CAP in all): before
// its wait on the statistics, the block prepares every position's candidate list, so that after
// the wait nothing of it needs memory: warp i sorts position i's entries by (id, k) (ranking by
// counting), marks each id's first entry with q summed over the id's entries, and loads that id's
// logit in row i.  After the wait: the rows' pairs and the acceptance tests give n as before; the
// corrections -min(p, q) of position n's entries follow from shared memory, and, with the entries
// in id order, each segment's corrections form one run, summed in order by the thread at its start.
// Row n is prefetched into L2 for the final rescan of the claiming segment, whose corrections are
// found by a binary search of the sorted ids.  Results repeat bit for bit (fixed orders throughout);
// they agree with the general form of the walk to rounding.
constexpr int VW_FK = 128;   // candidates per position on the staged path
constexpr int VW_CAP = 2048;  // staged entries over all positions

__device__ __forceinline__ void prefetch_l2_bytes(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

template <typename T>
__global__ void __launch_bounds__(VW_THREADS) k_verify_walk_staged(WalkParams p) {
  // the next kernel may launch as these blocks start (every library kernel launched with
  // programmatic dependent launch waits for this grid before it touches what it touches)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int PER = Elem<T>::PER16;
  constexpr int SEG = 32 * PER * SEG_VECS;
  constexpr int LANE_IDS = PER * SEG_VECS;
  constexpr int NOID = 0x7FFFFFFF;           // sort key of an id outside the vocabulary (last)
  extern __shared__ float sw[];             // [n_seg] segment weights, then [n_seg] correction sums
  __shared__ int32_t e_v[VW_CAP];           // each position's entries sorted by (id, k)
  __shared__ float e_q[VW_CAP];             // at an id's first entry: q(id) over its entries; else -1
  __shared__ float e_l[VW_CAP];             // at an id's first entry: the id's logit in the row
  __shared__ float s_corr[VW_FK];           // corrections of position n's entries (sorted order)
  __shared__ int s_n, s_seg, s_last;
  __shared__ float s_wtot[VW_THREADS / 32];
  __shared__ float s_local;
  __shared__ float2 s_row[VW_MAX_L + 1];
  __shared__ float s_qx[VW_MAX_L], s_lx[VW_MAX_L];
  const int b = blockIdx.x;
  const int L = p.L, K = p.K, n_seg = p.n_seg;
  float* cseg = sw + n_seg;
  const T* rows = static_cast<const T*>(p.logits) + (size_t)b * (L + 1) * p.vocab;
  const float2* segs = p.seg_stats + (size_t)b * (L + 1) * n_seg;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) { s_n = L; s_seg = 0x7FFFFFFF; s_last = -1; }
  for (int s = threadIdx.x; s < n_seg; s += VW_THREADS) cseg[s] = 0.f;
  // ---- before the wait: q_i(x_i), the logit of x_i, and position i's sorted entries (warp i)
  for (int i = warp; i < L; i += VW_THREADS / 32) {
    const int x = p.draft[(size_t)b * L + i];
    const int32_t* ci = p.cand_idx + ((size_t)b * L + i) * K;
    const float* cq = p.cand_prob + ((size_t)b * L + i) * K;
    const T* row = rows + (size_t)i * p.vocab;
    const int base = i * K;
    float qx = 0.f;
    for (int k = lane; k < K; k += 32) {
      const int v = ci[k];
      const float q = cq[k];
      if (v == x) qx += q;
      e_v[base + k] = (v >= 0 && v < p.vocab) ? v : NOID;
      e_q[base + k] = q;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) qx += __shfl_xor_sync(0xFFFFFFFFu, qx, o);
    if (lane == 0) {
      const bool in_range = x >= 0 && x < p.vocab;
      s_qx[i] = in_range ? qx : 0.f;  // outside the vocabulary: accepted, as q(x) = 0
      s_lx[i] = in_range ? logit_at(row, x) : 0.f;
    }
    __syncwarp();
    // rank by (id, k): at most VW_FK / 32 entries per lane
    int rk[VW_FK / 32], kv[VW_FK / 32];
    float kq[VW_FK / 32];
#pragma unroll
    for (int j = 0; j < VW_FK / 32; ++j) {
      const int k = lane + 32 * j;
      rk[j] = -1;
      if (k < K) {
        kv[j] = e_v[base + k];
        kq[j] = e_q[base + k];
        int r = 0;
        for (int k2 = 0; k2 < K; ++k2) {
          const int v2 = e_v[base + k2];
          r += (v2 < kv[j] || (v2 == kv[j] && k2 < k)) ? 1 : 0;
        }
        rk[j] = r;
      }
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < VW_FK / 32; ++j)
      if (rk[j] >= 0) {
        e_v[base + rk[j]] = kv[j];
        e_q[base + rk[j]] = kq[j];
      }
    __syncwarp();
    // first entries: q summed over the id's run (k order), and the id's logit
    float fq[VW_FK / 32], fl[VW_FK / 32];
#pragma unroll
    for (int j = 0; j < VW_FK / 32; ++j) {
      const int r = lane + 32 * j;
      fq[j] = -1.f;
      fl[j] = 0.f;
      if (r < K) {
        const int v = e_v[base + r];
        if (v != NOID && (r == 0 || e_v[base + r - 1] != v)) {
          float q = 0.f;
          for (int r2 = r; r2 < K && e_v[base + r2] == v; ++r2) q += e_q[base + r2];
          fq[j] = q;
          fl[j] = logit_at(row, v);
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < VW_FK / 32; ++j) {
      const int r = lane + 32 * j;
      if (r < K) {
        e_q[base + r] = fq[j];
        e_l[base + r] = fl[j];
      }
    }
  }
  // the statistics come from k_verify_stats (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // ---- warp i combines row i's segment pairs, then takes the acceptance test of position i
  for (int i = warp; i <= L; i += VW_THREADS / 32) {
    const float2 rp = row_pair(segs + (size_t)i * n_seg, n_seg);
    if (lane == 0) {
      s_row[i] = rp;
      if (i < L) {
        const float qx = s_qx[i];
        const float px = ex2(s_lx[i] * p.c - rp.x) / rp.y;
        const bool accepted = qx <= 0.f || p.u_accept[(size_t)b * L + i] < px / qx;
        if (!accepted) atomicMin(&s_n, i);
      }
    }
  }
  __syncthreads();
  const int n = s_n;
  const T* row = rows + (size_t)n * p.vocab;
  // row n towards L2 for the final rescan (64 KB pieces)
  if (warp == VW_THREADS / 32 - 1) {
    const uint32_t row_bytes = (uint32_t)((size_t)p.vocab * sizeof(T));  // a multiple of 16
    for (uint32_t off = (uint32_t)lane * 65536u; off < row_bytes; off += 32u * 65536u)
      prefetch_l2_bytes(reinterpret_cast<const char*>(row) + off, min(65536u, row_bytes - off));
  }
  const float2 st = s_row[n];
  const float inv_s = 1.f / st.y;
  const float2* seg = segs + (size_t)n * n_seg;
  const int Kn = n < L ? K : 0;
  const int base = n < L ? n * K : 0;
  // ---- corrections -min(p, q) of position n's entries, then each segment's run summed in order
  for (int r = threadIdx.x; r < Kn; r += VW_THREADS) {
    const float q = e_q[base + r];
    s_corr[r] = q >= 0.f ? -fminf(ex2(e_l[base + r] * p.c - st.x) * inv_s, q) : 0.f;
  }
  __syncthreads();
  for (int r = threadIdx.x; r < Kn; r += VW_THREADS) {
    const int v = e_v[base + r];
    if (v == NOID) continue;
    const int sg = v / SEG;
    if (r > 0 && e_v[base + r - 1] / SEG == sg) continue;  // not the start of its segment's run
    float cs = 0.f;
    for (int r2 = r; r2 < Kn && e_v[base + r2] != NOID && e_v[base + r2] / SEG == sg; ++r2) cs += s_corr[r2];
    cseg[sg] = cs;
  }
  __syncthreads();
  // ---- per-segment weights; thread t owns segments [t * per, (t + 1) * per)
  const int per = (n_seg + VW_THREADS - 1) / VW_THREADS;
  const int sa = min(n_seg, (int)threadIdx.x * per), sb = min(n_seg, sa + per);
  auto seg_mass = [&](int s) {
    const float2 sg = seg[s];
    return sg.x == -INFINITY ? 0.f : sg.y * ex2(sg.x - st.x) * inv_s;
  };
  float tsum = 0.f;
  for (int s = sa; s < sb; ++s) {
    const float w = fmaxf(seg_mass(s) + cseg[s], 0.f);
    sw[s] = w;
    tsum += w;
  }
  float total;
  float excl = block_excl_scan(tsum, s_wtot, &total);
  // a zero residual (p_n = q_n on the candidates, no mass elsewhere): draw from p_n itself
  const bool use_p = !(total > 0.f);
  if (use_p) {
    tsum = 0.f;
    for (int s = sa; s < sb; ++s) {
      sw[s] = seg_mass(s);
      tsum += sw[s];
    }
    excl = block_excl_scan(tsum, s_wtot, &total);
  }
  const float target = p.u_sample[b] * total;
  int mine = -1, last_pos = -1;
  float before = 0.f;
  if (sb > sa && excl <= target && target < excl + tsum) {
    float run = excl;
    for (int s = sa; s < sb; ++s) {
      if (sw[s] > 0.f && run + sw[s] > target) { mine = s; before = run; break; }
      run += sw[s];
    }
  }
  for (int s = sa; s < sb; ++s)
    if (sw[s] > 0.f) last_pos = s;
  if (mine >= 0) atomicMin(&s_seg, mine);
  if (last_pos >= 0) atomicMax(&s_last, last_pos);
  __syncthreads();
  const bool claimed = s_seg != 0x7FFFFFFF;
  if (mine >= 0 && mine == s_seg) s_local = target - before;
  __syncthreads();
  // ---- warp 0 recomputes the chosen segment's weights id by id and finds the token
  if (warp == 0) {
    const int sg = claimed ? s_seg : (s_last < 0 ? 0 : s_last);
    const float local = claimed ? s_local : INFINITY;  // unclaimed: the segment's last positive id
    const int id0 = sg * SEG + lane * LANE_IDS;
    float w[LANE_IDS];
#pragma unroll
    for (int v = 0; v < SEG_VECS; ++v) {
      const int id = id0 + v * PER;
      uint4 u = make_uint4(0, 0, 0, 0);
      if (id < p.vocab) u = *reinterpret_cast<const uint4*>(row + id);
      Elem<T>::unpack(u, w + v * PER);
#pragma unroll
      for (int e = 0; e < PER; ++e) w[v * PER + e] = id + e < p.vocab ? ex2(w[v * PER + e] * p.c - st.x) * inv_s : 0.f;
    }
    if (!use_p && Kn > 0) {
      // the segment's entries: the first sorted entry with id >= sg * SEG (binary search), onwards
      int lo = 0, hi = Kn;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (e_v[base + mid] < sg * SEG) lo = mid + 1; else hi = mid;
      }
      for (int r = lo; r < Kn; ++r) {
        const int v = e_v[base + r];
        if (v == NOID || v >= (sg + 1) * SEG) break;
        if (e_q[base + r] < 0.f || v < id0 || v >= id0 + LANE_IDS) continue;  // not a first entry, or another lane's
#pragma unroll
        for (int e = 0; e < LANE_IDS; ++e)
          if (id0 + e == v) w[e] = fmaxf(w[e] + s_corr[r], 0.f);
      }
    }
    float lsum = 0.f;
#pragma unroll
    for (int e = 0; e < LANE_IDS; ++e) lsum += w[e];
    float incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const float ex = incl - lsum;
    const uint32_t bm = __ballot_sync(0xFFFFFFFFu, lsum > 0.f && ex <= local && local < incl);
    int tok = -1;
    if (bm) {
      const int src = __ffs(bm) - 1;
      if (lane == src) {
        float run = ex;
#pragma unroll
        for (int e = 0; e < LANE_IDS; ++e) {
          if (tok < 0 && w[e] > 0.f && run + w[e] > local) tok = id0 + e;
          run += w[e];
        }
        if (tok < 0)
#pragma unroll
          for (int e = 0; e < LANE_IDS; ++e)
            if (w[e] > 0.f) tok = id0 + e;
      }
      tok = __shfl_sync(0xFFFFFFFFu, tok, src);
    } else {
      int lastv = -1;
#pragma unroll
      for (int e = 0; e < LANE_IDS; ++e)
        if (w[e] > 0.f) lastv = id0 + e;
      lastv = __reduce_max_sync(0xFFFFFFFFu, lastv);
      tok = lastv < 0 ? sg * SEG : lastv;
    }
    if (lane == 0) {
      p.n_accept[b] = n;
      p.token[b] = tok;
    }
  }
}

template <typename T>
cudaError_t run(const Ctx& c, const void* logits, int B, int L, int vocab, int K, const int32_t* cand_idx,
                const float* cand_prob, const int32_t* draft, const float* u_accept, const float* u_sample,
                float temperature, int32_t* n_accept, int32_t* token, float2* seg_stats) {
  constexpr int SEG = 32 * Elem<T>::PER16 * SEG_VECS;
  const int n_seg = (vocab + SEG - 1) / SEG;
  const float cf = LOG2E / temperature;
  const int n_items = B * (L + 1) * n_seg;  // < 2^31: checked by the caller
  // persistent grid: two blocks per SM stream the (row, segment) items
  const int per_block = VS_THREADS / 32;
  const unsigned grid = (unsigned)max(1, min(2 * c.num_sms, (n_items + per_block - 1) / per_block));
  cudaError_t e;
  {  // programmatic dependent launch: the launch overlaps the previous kernel's tail
    cudaLaunchAttribute sa[1];
    sa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    sa[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t sc = {};
    sc.gridDim = dim3(grid);
    sc.blockDim = dim3(VS_THREADS);
    sc.stream = c.stream;
    sc.attrs = sa;
    sc.numAttrs = 1;
    prof_before("verify_stats", c.stream);
    e = cudaLaunchKernelEx(&sc, k_verify_stats<T>, static_cast<const T*>(logits), vocab, cf, n_seg, n_items,
                           seg_stats);
    prof_after(c.stream);
  }
  if (e != cudaSuccess) return e;
  WalkParams wp;
  wp.logits = logits;
  wp.cand_idx = cand_idx;
  wp.cand_prob = cand_prob;
  wp.draft = draft;
  wp.u_accept = u_accept;
  wp.u_sample = u_sample;
  wp.seg_stats = seg_stats;
  wp.L = L;
  wp.vocab = vocab;
  wp.K = K;
  wp.n_seg = n_seg;
  wp.c = cf;
  wp.n_accept = n_accept;
  wp.token = token;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)B);
  cfg.blockDim = dim3(VW_THREADS);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool staged = K <= VW_FK && (long long)L * K <= VW_CAP;
  static unsigned long long smem_done = 0, smem_done_st = 0;
  if (staged) {
    cfg.dynamicSmemBytes = 2 * (size_t)n_seg * sizeof(float);
    e = allow_max_smem(k_verify_walk_staged<T>, c.device, &smem_done_st);
  } else {
    cfg.dynamicSmemBytes = (size_t)n_seg * sizeof(float);
    e = allow_max_smem(k_verify_walk<T>, c.device, &smem_done);
  }
  if (e != cudaSuccess) return e;
  prof_before("verify_walk", c.stream);
  e = staged ? cudaLaunchKernelEx(&cfg, k_verify_walk_staged<T>, wp) : cudaLaunchKernelEx(&cfg, k_verify_walk<T>, wp);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

int verify_segments(int vocab, int dtype) {
  const int seg = 32 * (dtype == DH_BF16 ? 8 : 4) * SEG_VECS;
  return (vocab + seg - 1) / seg;
}

cudaError_t launch_verify(const Ctx& c, const void* logits, int dtype, int B, int L, int vocab, int K,
                          const int32_t* cand_idx, const float* cand_prob, const int32_t* draft, const float* u_accept,
                          const float* u_sample, float temperature, int32_t* n_accept, int32_t* token,
                          float2* seg_stats) {
  if (dtype == DH_BF16)
    return run<__nv_bfloat16>(c, logits, B, L, vocab, K, cand_idx, cand_prob, draft, u_accept, u_sample, temperature,
                              n_accept, token, seg_stats);
  return run<float>(c, logits, B, L, vocab, K, cand_idx, cand_prob, draft, u_accept, u_sample, temperature, n_accept,
                    token, seg_stats);
}

}  // namespace dh
