// Stage 2: exact full-rank logits of the retrieved candidates and their softmax.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the candidates' exact logits come from the original full-rank head.  Section "Why a draft tree
// needs a cost model": products of the resulting draft probabilities estimate the benefit of a
// branch; the softmax here runs over the K candidates of a row at temperature 1.
//
// Gather-GEMV: one warp per (row, candidate) streams W[idx] (d contiguous values) with 16-byte
// loads against h[row] staged in shared memory, accumulates in fp32 and reduces with shuffles.  An index outside [0, vocab)
// is never dereferenced: its logit becomes NaN (and so do the row's probabilities).
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>

#include "dh_internal.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

constexpr int WARPS = 8;          // candidates per block (one warp each), larger batches
constexpr int THREADS = WARPS * 32;
constexpr int MAXW = 20;          // 16-byte W vectors per lane in flight (d = 5120 bf16 in one batch)
constexpr int MAX_D_SMEM = 8192;  // h row staged in shared memory (bf16: 16 KB, fp32: 32 KB)

// One warp's dot product of h (staged in shared memory) with W row v: each lane keeps MAXW
// 16-byte loads of the row in flight, then the warp reduces with shuffles (every lane gets the sum).
template <typename T>
__device__ __forceinline__ float warp_row_dot(const T* __restrict__ W, int v, int d, const T* sh_h, int lane) {
  constexpr int PER = Elem<T>::PER16;
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
      if (c < d) acc = Elem<T>::dot16(*reinterpret_cast<const uint4*>(sh_h + c), wa[q], acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  return acc;
}

// Block (b, kb) scores candidates kb*8 .. kb*8+7 of row b.  The block stages h[b] in shared
// memory (before waiting on the previous kernel: h does not depend on it), then each warp streams
// its W row with MAXW 16-byte loads per lane in flight and reduces with shuffles.  With probs
// requested, the block adds its candidate count to the row's ticket; the block completing the row
// computes the softmax and resets the ticket.
template <typename T, int NWARP>
__global__ void __launch_bounds__(NWARP * 32) k_rescore(const T* __restrict__ h, const T* __restrict__ W,
                                                     const int32_t* __restrict__ idx, int d, int vocab, int K,
                                                     float* __restrict__ logits, float* __restrict__ probs,
                                                     uint32_t* __restrict__ tickets) {
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* sh_h = reinterpret_cast<T*>(smem_raw);
  __shared__ int s_last;
  const int kblocks = (K + NWARP - 1) / NWARP;
  const int b = blockIdx.x / kblocks, kb = blockIdx.x % kblocks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = kb * NWARP + warp;
  const int n_here = min(NWARP, K - kb * NWARP);
  const T* x = h + (size_t)b * d;
  for (int c = threadIdx.x * PER; c < d; c += (NWARP * 32) * PER)
    *reinterpret_cast<uint4*>(sh_h + c) = __ldg(reinterpret_cast<const uint4*>(x + c));
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  __syncthreads();
  if (k < K) {
    const int pair = b * K + k;
    const int v = idx[pair];
    const bool ok = v >= 0 && v < vocab;
    const float acc = ok ? warp_row_dot<T>(W, v, d, sh_h, lane) : 0.f;
    if (lane == 0) logits[pair] = ok ? acc : __int_as_float(0x7FC00000);
  }
  if (!probs) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&tickets[b], (uint32_t)n_here) + (uint32_t)n_here == (uint32_t)K;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // softmax over the row's K logits (written by other blocks: read through L2), by one warp
  if (warp == 0) warp_softmax_l2(logits + (size_t)b * K, K, probs + (size_t)b * K);
  if (threadIdx.x == 0) tickets[b] = 0u;
}

// ------------------------------------------------------------------------------------------------
// Cluster variant for small batches with K <= CL_MAX_K: one thread-block cluster of up to 8 CTAs
// per row; warp w of cluster CTA c scores candidates c*NWARP + w, c*NWARP + w + CTAs*NWARP, ...
// Each warp also stores its logit into the leader CTA's shared memory (distributed shared
// memory); after a cluster barrier one warp of the leader computes the row's softmax from there,
// without the global ticket and the L2 round trips of the ticket scheme.  Every CTA passes both cluster
// barriers (no early exit), so the barriers always complete.
constexpr int CL_MAX_K = 128;
constexpr int CL_MAX_CTAS = 8;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// Stores v at the same shared-memory offset as `local` in cluster CTA `rank`.
__device__ __forceinline__ void st_cluster_f32(float* local, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(sm100::smem_u32(local)), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

template <typename T, int NWARP>
__global__ void __launch_bounds__(NWARP * 32) k_rescore_cl(const T* __restrict__ h, const T* __restrict__ W,
                                                        const int32_t* __restrict__ idx, int d, int vocab, int K,
                                                        float* __restrict__ logits, float* __restrict__ probs) {
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* sh_h = reinterpret_cast<T*>(smem_raw);
  __shared__ float s_z[CL_MAX_K];  // leader CTA: the row's logits
  const uint32_t crank = cluster_ctarank(), csize = cluster_nctarank();
  const int b = (int)(blockIdx.x / csize);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // phase 1 of the cluster barrier: this CTA is running (its shared memory may be written)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  const T* x = h + (size_t)b * d;
  for (int c = threadIdx.x * PER; c < d; c += (NWARP * 32) * PER)
    *reinterpret_cast<uint4*>(sh_h + c) = __ldg(reinterpret_cast<const uint4*>(x + c));
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  __syncthreads();
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA of the cluster is running
  for (int k = (int)crank * NWARP + warp; k < K; k += (int)csize * NWARP) {
    const int pair = b * K + k;
    const int v = idx[pair];
    const bool ok = v >= 0 && v < vocab;
    const float acc = ok ? warp_row_dot<T>(W, v, d, sh_h, lane) : 0.f;
    const float z = ok ? acc : __int_as_float(0x7FC00000);
    if (lane == 0) {
      logits[pair] = z;
      st_cluster_f32(&s_z[k], 0, z);
    }
  }
  // phase 2: the leader sees every logit of the row
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
  if (crank != 0 || !probs || warp != 0) return;
  warp_softmax(s_z, K, probs + (size_t)b * K);
}

template <typename T, int NWARP>
cudaError_t launch_cl(const Ctx& c, const T* h, const T* W, const int32_t* idx, int B, int d, int vocab, int K,
                      float* logits, float* probs) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore_cl<T, NWARP>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  const int ctas = min(CL_MAX_CTAS, (K + NWARP - 1) / NWARP);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)ctas;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ctas));
  cfg.blockDim = dim3(NWARP * 32);
  cfg.dynamicSmemBytes = (size_t)d * sizeof(T);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_before("rescore_cluster", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore_cl<T, NWARP>, h, W, idx, d, vocab, K, logits, probs);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Smallest warp count per CTA with at most one candidate per warp on a full cluster.
template <typename T>
cudaError_t run_cl(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                   float* logits, float* probs) {
  const T* hh = static_cast<const T*>(h);
  const T* ww = static_cast<const T*>(W);
  if (K <= 2 * CL_MAX_CTAS) return launch_cl<T, 2>(c, hh, ww, idx, B, d, vocab, K, logits, probs);
  if (K <= 4 * CL_MAX_CTAS) return launch_cl<T, 4>(c, hh, ww, idx, B, d, vocab, K, logits, probs);
  if (K <= 8 * CL_MAX_CTAS) return launch_cl<T, 8>(c, hh, ww, idx, B, d, vocab, K, logits, probs);
  return launch_cl<T, 16>(c, hh, ww, idx, B, d, vocab, K, logits, probs);
}

// ------------------------------------------------------------------------------------------------
// Ring variant for larger batches.  Block (c, b) scores a share of row b's candidates:
// - bucket mode (bw > 0, when the gathered rows exceed what L2 keeps): the vocabulary is cut into
//   buckets of bw consecutive ids and the share is the candidates whose ids fall in bucket c.
//   Blocks are numbered bucket by bucket, so the blocks running at any time gather W rows from one
//   or two buckets: a W row that several rows of the batch selected is read from HBM by the first
//   of them and found in L2 by the others.  Warp 0 lists the bucket's candidates;
// - chunk mode (bw = 0): the share is candidates [RING_CHUNK c, RING_CHUNK (c + 1)).
// h[b] is bulk-copied into shared memory once (before waiting on the previous kernel).  Each of
// the NW warps gathers the W rows of its part of the share itself, one at a time, with a 1-D bulk
// copy (cp.async.bulk) into a slot of its own.  The copy engine serves one issuing thread at about
// 45 GB/s, so every warp issues; with small blocks, several of them per SM, the copies of one
// block run while another starts.  An id outside [0, vocab) belongs to bucket 0 and is never
// dereferenced.

constexpr int RING_WARPS_BUCKET = 4;   // warps per block in bucket mode (four blocks per SM)
constexpr int RING_WARPS_CHUNK = 8;    // warps per block in chunk mode (two blocks per SM)
constexpr int RING_CHUNK = 32;         // candidates per block in chunk mode
constexpr int RING_BUCKET_PAIRS = 32;  // candidates per block on average in bucket mode
constexpr int RING_SORT = 64;          // bucket lists up to this long are put in id order
constexpr int RING_MAX_K = 4096;       // the bucket's list holds up to a whole row
constexpr uint64_t RING_WAIT_NS = 2000000000ull;

inline size_t ring_smem(int K, int d, int elem, int nw) {
  const size_t row = (size_t)d * elem;
  return 128 + align_up(row, 128) + (size_t)nw * row + (size_t)K * sizeof(int2);
}

template <typename T, int NW>
__global__ void __launch_bounds__(NW * 32)
    k_rescore_ring(const T* __restrict__ h, const T* __restrict__ W, const int32_t* __restrict__ idx, int B, int d,
                   int vocab, int K, int bw, float* __restrict__ logits, float* __restrict__ probs,
                   uint32_t* __restrict__ tickets, int* __restrict__ status) {
  using namespace sm100;
  constexpr int RING_WARPS = NW, RING_THREADS = NW * 32, RING_WSLOTS = 1;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t h_full, full[RING_WARPS][RING_WSLOTS];
  __shared__ int s_last, s_n;
  __shared__ volatile int s_fail;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                         ~static_cast<uintptr_t>(127));
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const T* hs = reinterpret_cast<const T*>(base);
  unsigned char* ring = base + align_up(row_bytes, 128);
  int2* list = reinterpret_cast<int2*>(ring + (size_t)RING_WARPS * RING_WSLOTS * row_bytes);  // (k, id)
  const int c = blockIdx.x / B, b = blockIdx.x % B;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the next kernel may launch as these blocks start (every library kernel launched with
  // programmatic dependent launch waits for this grid before it touches what it touches)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {
    s_fail = 0;
    mbar_init(&h_full, 1);
    for (int w = 0; w < RING_WARPS; ++w)
      for (int s = 0; s < RING_WSLOTS; ++s) mbar_init(&full[w][s], 1);
    fence_barrier_init();
    // h does not depend on the previous kernel
    mbar_arrive_expect_tx(&h_full, row_bytes);
    bulk_load(base, h + (size_t)b * d, row_bytes, &h_full);
  }
  if (bw > 0 && warp == 0) {
    // the row's candidates in bucket c, in candidate order
    asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
    const int32_t* ib = idx + (size_t)b * K;
    int cnt = 0;
    for (int k0 = 0; k0 < K; k0 += 8 * 32) {
      int vv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * 32 + lane;
        vv[u] = k < K ? ib[k] : 0;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int k = k0 + u * 32 + lane;
        const int v = vv[u];
        const bool in = k < K && ((v >= 0 && v < vocab) ? v / bw : 0) == c;
        const uint32_t m = __ballot_sync(0xFFFFFFFFu, in);
        if (in) list[cnt + __popc(m & ((1u << lane) - 1u))] = make_int2(k, v);
        cnt += __popc(m);
      }
    }
    if (cnt <= RING_SORT) {
      // a short list goes into id order (ranked by counting; the keys are distinct), so that the
      // blocks sweep their buckets from low to high ids at about the same pace
      __syncwarp();
      auto key = [&](int i) {
        return i < cnt ? (long long)list[i].y * 4294967296LL + (long long)(uint32_t)list[i].x : LLONG_MAX;
      };
      const long long k0 = key(lane), k1 = key(lane + 32);
      const int2 e0 = lane < cnt ? list[lane] : make_int2(0, 0);
      const int2 e1 = lane + 32 < cnt ? list[lane + 32] : make_int2(0, 0);
      int r0 = 0, r1 = 0;
      for (int q = 0; q < 32; ++q) {
        const long long a = __shfl_sync(0xFFFFFFFFu, k0, q), a1 = __shfl_sync(0xFFFFFFFFu, k1, q);
        r0 += (a < k0) + (a1 < k0);
        r1 += (a < k1) + (a1 < k1);
      }
      __syncwarp();
      if (lane < cnt) list[r0] = e0;
      if (lane + 32 < cnt) list[r1] = e1;
    }
    if (lane == 0) s_n = cnt;
  }
  __syncthreads();
  if (bw == 0) {
    // chunk mode: each warp stages the ids of its own candidates
    asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
    const int n_chunk = min(RING_CHUNK, K - c * RING_CHUNK);
    const int i = warp + lane * RING_WARPS;
    if (i < n_chunk) {
      const int k = c * RING_CHUNK + i;
      list[i] = make_int2(k, idx[(size_t)b * K + k]);
    }
    __syncwarp();
  }
  const int n_here = bw > 0 ? s_n : min(RING_CHUNK, K - c * RING_CHUNK);
  // this warp's candidates: entries warp, warp + RING_WARPS, ... of the share
  const int n_mine = n_here > warp ? (n_here - 1 - warp) / RING_WARPS + 1 : 0;
  unsigned char* mine = ring + (size_t)warp * RING_WSLOTS * row_bytes;
  auto entry = [&](int j) { return list[warp + j * RING_WARPS]; };  // (k, id) of the warp's j-th candidate
  auto issue = [&](int j) {  // lane 0: the copy of the warp's j-th candidate into slot j % RING_WSLOTS
    const int2 kv = entry(j);
    uint64_t* bar = &full[warp][j % RING_WSLOTS];
    if (kv.y >= 0 && kv.y < vocab) {
      mbar_arrive_expect_tx(bar, row_bytes);
      bulk_load(mine + (size_t)(j % RING_WSLOTS) * row_bytes, W + (size_t)kv.y * d, row_bytes, bar);
    } else {
      mbar_arrive(bar);
    }
  };
  int issued = 0, consumed = 0;  // lane 0's counts
  if (lane == 0)
    for (; issued < RING_WSLOTS && issued < n_mine; ++issued) issue(issued);
  bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&h_full, 0, RING_WAIT_NS));
  if (!ok && lane == 0) {
    atomicOr(status, 1 << DH_ERR_TIMEOUT);
    s_fail = 1;
  }
  for (int j = 0; ok && j < n_mine; ++j) {
    const int s = j % RING_WSLOTS;
    if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[warp][s], (uint32_t)(j / RING_WSLOTS) & 1u, RING_WAIT_NS))) {
      if (lane == 0) {
        atomicOr(status, 1 << DH_ERR_TIMEOUT);
        s_fail = 1;
      }
      ok = false;
      break;
    }
    consumed = j + 1;
    const int2 kv = entry(j);
    const bool valid = kv.y >= 0 && kv.y < vocab;
    float acc = 0.f;
    if (valid) {
      const T* wr = reinterpret_cast<const T*>(mine + (size_t)s * row_bytes);
      for (int e = lane * Elem<T>::PER16; e < d; e += 32 * Elem<T>::PER16)
        acc = Elem<T>::dot16(*reinterpret_cast<const uint4*>(hs + e), *reinterpret_cast<const uint4*>(wr + e), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    __syncwarp();  // every lane has read slot s
    if (lane == 0) {
      logits[(size_t)b * K + kv.x] = valid ? acc : __int_as_float(0x7FC00000);
      if (issued < n_mine) {
        fence_proxy_async_smem();
        issue(issued);
        ++issued;
      }
    }
  }
  if (!ok && lane == 0)  // let this warp's copies in flight land before the block exits
    for (int j = consumed; j < issued; ++j)
      mbar_wait(&full[warp][j % RING_WSLOTS], (uint32_t)(j / RING_WSLOTS) & 1u, RING_WAIT_NS);
  __syncthreads();
  if (s_fail) return;
  // (a block with no candidates takes no ticket: the row's count may already have been reset)
  if (!probs || n_here == 0) return;
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&tickets[b], (uint32_t)n_here) + (uint32_t)n_here == (uint32_t)K;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // softmax over the row's K logits (written by other blocks: read through L2), by one warp
  if (warp == 0) warp_softmax_l2(logits + (size_t)b * K, K, probs + (size_t)b * K);
  if (threadIdx.x == 0) tickets[b] = 0u;
}

template <typename T, int NW>
cudaError_t launch_ring(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                        int nbk, int bw, float* logits, float* probs, uint32_t* tickets, int* status) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore_ring<T, NW>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * nbk));
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = ring_smem(K, d, (int)sizeof(T), NW);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore_ring", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore_ring<T, NW>, static_cast<const T*>(h), static_cast<const T*>(W), idx, B, d,
                         vocab, K, bw, logits, probs, tickets, status);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t run_ring(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                     float* logits, float* probs, uint32_t* tickets, int* status, bool force_buckets) {
  // bucket mode once the gathered rows are larger than L2 (or when asked for); chunk mode below
  if (force_buckets || (double)B * K * d * sizeof(T) > (double)c.l2_bytes) {
    const int nbk0 = std::max(1, std::min(K / RING_BUCKET_PAIRS, vocab));
    const int bw = (vocab + nbk0 - 1) / nbk0;
    return launch_ring<T, RING_WARPS_BUCKET>(c, h, W, idx, B, d, vocab, K, (vocab + bw - 1) / bw, bw, logits, probs,
                                             tickets, status);
  }
  return launch_ring<T, RING_WARPS_CHUNK>(c, h, W, idx, B, d, vocab, K, (K + RING_CHUNK - 1) / RING_CHUNK, 0, logits,
                                          probs, tickets, status);
}

// Sweep variant for large batches: block j owns SW_ROWS batch rows, keeps their h rows in shared
// memory, and orders its SW_ROWS x K (row, candidate) pairs by vocabulary bucket (ids >> SW_SHIFT,
// a counting sort); a producer thread then streams the pairs' W rows through a ring of bulk-copy
// slots in that order while the consumer warps take the slots in turn.  Every block walks the
// vocabulary from low to high ids at the same pace, so a W row that several rows of the batch
// share is requested by their blocks within a few buckets of each other: HBM delivers it once and
// L2 serves the rest (the B x K candidates of a batch hold each distinct row about 1.5 times at
// batch 512).  A block owns its rows' K logits, so it computes their softmax itself at the end.
// Per-candidate dot products have the order of the other rescoring kernels (bit-identical logits).
constexpr int SW_CONSUMERS = 16;
constexpr int SW_THREADS = (SW_CONSUMERS + 1) * 32;
// One slot per consumer warp: warp w takes items w, w + SW_SLOTS, ..., all in slot w, so the slot's
// mbarrier phases advance one round per item of that warp.  (With fewer slots than consumers a warp
// could wait for round r + 2 of a slot still in round r, and an mbarrier's parity cannot tell the
// two apart; a fresh mbarrier also reports its odd phase complete, which a warp starting at round
// 1 would take as data.)
constexpr int SW_SLOTS = SW_CONSUMERS;
static_assert(SW_SLOTS == SW_CONSUMERS, "each consumer warp owns one ring slot");
constexpr int SW_ROWS_MAX = 4;
constexpr int SW_SHIFT = 11;  // bucket = 2048 ids

// Rows per block: enough that the grid fits the SMs in one wave (one block per SM).
inline int sweep_rows(int B, int num_sms) { return std::min(SW_ROWS_MAX, std::max(1, (B + num_sms - 1) / num_sms)); }

__host__ __device__ inline size_t sweep_smem(int rows, int d, int elem, int K, int n_buckets) {
  return 128 + align_up((size_t)rows * d * elem, 128) + (size_t)SW_SLOTS * d * elem +
         align_up((size_t)rows * K * 8, 16) + (size_t)n_buckets * 4;
}

template <typename T>
__global__ void __launch_bounds__(SW_THREADS, 1)
    k_rescore_sweep(const T* __restrict__ h, const T* __restrict__ W, const int32_t* __restrict__ idx, int B, int d,
                    int vocab, int K, int rows, int n_buckets, float* __restrict__ logits, float* __restrict__ probs,
                    int* __restrict__ status) {
  using namespace sm100;
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t h_full, full[SW_SLOTS], empty[SW_SLOTS];
  __shared__ int slot_pair[SW_SLOTS], slot_ok[SW_SLOTS];
  __shared__ volatile int s_fail;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                         ~static_cast<uintptr_t>(127));
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const int b0 = blockIdx.x * rows;
  const int nrows = min(rows, B - b0);
  const int n_pairs = nrows * K;
  const T* hs = reinterpret_cast<const T*>(base);
  unsigned char* ring = base + align_up((size_t)rows * row_bytes, 128);
  int2* order = reinterpret_cast<int2*>(ring + (size_t)SW_SLOTS * row_bytes);  // (pair, id) by bucket
  uint32_t* bucket = reinterpret_cast<uint32_t*>(reinterpret_cast<unsigned char*>(order) +
                                                 align_up((size_t)rows * K * 8, 16));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_fail = 0;
    mbar_init(&h_full, 1);
    for (int s = 0; s < SW_SLOTS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
    // the block's h rows do not depend on the previous kernel
    mbar_arrive_expect_tx(&h_full, (uint32_t)nrows * row_bytes);
    for (int r = 0; r < nrows; ++r) bulk_load(base + (size_t)r * row_bytes, h + (size_t)(b0 + r) * d, row_bytes, &h_full);
  }
  for (int z = threadIdx.x; z < n_buckets; z += SW_THREADS) bucket[z] = 0u;
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  // counting sort of the pairs by bucket: counts, exclusive prefix (one warp), scatter
  const int32_t* ib = idx + (size_t)b0 * K;
  for (int q = threadIdx.x; q < n_pairs; q += SW_THREADS) {
    const int v = ib[q];
    atomicAdd(&bucket[(v >= 0 && v < vocab) ? (v >> SW_SHIFT) : 0], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    uint32_t run = 0u;
    for (int z0 = 0; z0 < n_buckets; z0 += 32) {
      const int z = z0 + lane;
      const uint32_t cnt = z < n_buckets ? bucket[z] : 0u;
      uint32_t incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      if (z < n_buckets) bucket[z] = run + incl - cnt;
      run += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
  }
  __syncthreads();
  for (int q = threadIdx.x; q < n_pairs; q += SW_THREADS) {
    const int v = ib[q];
    order[atomicAdd(&bucket[(v >= 0 && v < vocab) ? (v >> SW_SHIFT) : 0], 1u)] = make_int2(q, v);
  }
  __syncthreads();
  if (warp == SW_CONSUMERS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      for (int i = 0; i < n_pairs && !s_fail; ++i) {
        const int s = i % SW_SLOTS;
        if (!mbar_wait(&empty[s], ((uint32_t)(i / SW_SLOTS) & 1u) ^ 1u, RING_WAIT_NS)) {
          s_fail = 1;
          atomicOr(status, 1 << DH_ERR_TIMEOUT);
          break;
        }
        const int2 qv = order[i];  // shared memory: the issue loop never waits on a global load
        const int q = qv.x, v = qv.y;
        const bool ok = v >= 0 && v < vocab;
        slot_pair[s] = q;
        slot_ok[s] = ok;
        if (ok) {
          mbar_arrive_expect_tx(&full[s], row_bytes);
          bulk_load(ring + (size_t)s * row_bytes, W + (size_t)v * d, row_bytes, &full[s]);
        } else {
          mbar_arrive(&full[s]);
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const bool h_ok = __all_sync(0xFFFFFFFFu, mbar_wait(&h_full, 0, RING_WAIT_NS));
    if (!h_ok) {
      if (lane == 0) atomicOr(status, 1 << DH_ERR_TIMEOUT);
      s_fail = 1;
    }
    for (int i = warp; h_ok && i < n_pairs; i += SW_CONSUMERS) {
      const int s = i % SW_SLOTS;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (uint32_t)(i / SW_SLOTS) & 1u, RING_WAIT_NS))) {
        if (lane == 0) atomicOr(status, 1 << DH_ERR_TIMEOUT);
        s_fail = 1;
        break;
      }
      const int q = slot_pair[s];
      const bool ok = slot_ok[s] != 0;
      const T* hr = hs + (size_t)(q / K) * d;
      float acc = 0.f;
      if (ok) {
        const T* wr = reinterpret_cast<const T*>(ring + (size_t)s * row_bytes);
        for (int c = lane * PER; c < d; c += 32 * PER)
          acc = Elem<T>::dot16(*reinterpret_cast<const uint4*>(hr + c), *reinterpret_cast<const uint4*>(wr + c), acc);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      __syncwarp();
      if (lane == 0) {
        logits[(size_t)b0 * K + q] = ok ? acc : __int_as_float(0x7FC00000);
        mbar_arrive(&empty[s]);  // the slot is free once the warp has read it
      }
    }
  }
  __syncthreads();
  if (s_fail) {
    // let every copy issued into this block's shared memory land before it exits
    if (threadIdx.x == 0) {
      mbar_wait(&h_full, 0, RING_WAIT_NS);
      for (int s = 0; s < SW_SLOTS && s < n_pairs; ++s) {
        const int last = s + ((n_pairs - 1 - s) / SW_SLOTS) * SW_SLOTS;
        mbar_wait(&full[s], (uint32_t)(last / SW_SLOTS) & 1u, RING_WAIT_NS);
      }
    }
    __syncthreads();
    return;
  }
  // the softmax of each owned row, one warp per row (the logits were written by this block)
  if (probs && warp < nrows) warp_softmax_l2(logits + (size_t)(b0 + warp) * K, K, probs + (size_t)(b0 + warp) * K);
}

template <typename T>
cudaError_t run_sweep(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                      float* logits, float* probs, int* status) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore_sweep<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  const int rows = sweep_rows(B, c.num_sms);
  const int n_buckets = ((vocab - 1) >> SW_SHIFT) + 1;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((B + rows - 1) / rows));
  cfg.blockDim = dim3(SW_THREADS);
  cfg.dynamicSmemBytes = sweep_smem(rows, d, (int)sizeof(T), K, n_buckets);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore_sweep", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore_sweep<T>, static_cast<const T*>(h), static_cast<const T*>(W), idx, B, d,
                         vocab, K, rows, n_buckets, logits, probs, status);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                int K, float* logits, float* probs, uint32_t* tickets) {
  // K <= CL_MAX_K: the cluster kernel (the DH_FORCE_RESCORE=ticket switch selects the ticket kernel)
  if (K <= CL_MAX_K && tuning().rescore != Tuning::RESCORE_TICKET)
    return run_cl<T>(c, h, W, idx, B, d, vocab, K, logits, probs);
  // Small problems use 2-warp blocks so that more SMs pull W rows; larger ones 8-warp blocks.
  const int nw = (long long)B * K <= 512 ? 2 : WARPS;
  static unsigned long long smem_done2 = 0, smem_done8 = 0;
  cudaError_t e = nw == 2 ? allow_max_smem(k_rescore<T, 2>, c.device, &smem_done2)
                          : allow_max_smem(k_rescore<T, WARPS>, c.device, &smem_done8);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the blocks may start while the stage-1 kernel drains; they
  // stage h and then wait (griddepcontrol.wait) for its results.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ((K + nw - 1) / nw)));
  cfg.blockDim = dim3(nw * 32);
  cfg.dynamicSmemBytes = (size_t)d * sizeof(T);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore", c.stream);
  e = nw == 2 ? cudaLaunchKernelEx(&cfg, k_rescore<T, 2>, static_cast<const T*>(h), static_cast<const T*>(W), idx, d,
                                   vocab, K, logits, probs, tickets)
              : cudaLaunchKernelEx(&cfg, k_rescore<T, WARPS>, static_cast<const T*>(h), static_cast<const T*>(W), idx, d,
                                   vocab, K, logits, probs, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool rescore_supported(int d) { return d <= MAX_D_SMEM; }

bool rescore_sweep_supported(int B, int K, int d, int vocab, int dtype, int num_sms) {
  const int elem = dtype == DH_BF16 ? 2 : 4;
  const int rows = sweep_rows(B, num_sms);
  return sweep_smem(rows, d, elem, K, ((vocab - 1) >> SW_SHIFT) + 1) <= 220 * 1024;
}

cudaError_t launch_rescore_sweep(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                 int vocab, int K, int dtype, float* logits, float* probs, int* status) {
  if (dtype == DH_BF16) return run_sweep<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, status);
  return run_sweep<float>(c, h, W, idx, B, d, vocab, K, logits, probs, status);
}

// The ring needs up to RING_WARPS_CHUNK + 1 rows of shared memory and the share's list (K
// entries): at K = 256 up to d = 11256 bf16 or 5628 fp32.
bool rescore_ring_fits(int K, int d, int dtype) {
  const int elem = dtype == DH_BF16 ? 2 : 4;
  return K <= RING_MAX_K && ring_smem(K, d, elem, std::max(RING_WARPS_CHUNK, RING_WARPS_BUCKET)) <= 200 * 1024;
}

// The ring variant from this many (row, candidate) pairs on: below it, one warp per pair with all
// of a row's loads in flight has the lower latency.
bool rescore_ring_used(int B, int K, int d, int dtype) {
  return (long long)B * K >= 2048 && rescore_ring_fits(K, d, dtype);
}

cudaError_t launch_rescore_ring(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets,
                                int* status, bool force_buckets) {
  if (dtype == DH_BF16)
    return run_ring<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, status, force_buckets);
  return run_ring<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, status, force_buckets);
}

// The deduplicated path holds a W row in registers (MAXW 16-byte vectors per lane).
cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                           int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
  return run<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
}

}  // namespace dh
