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
#include "dh_internal.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

constexpr int WARPS = 8;          // candidates per block (one warp each)
constexpr int THREADS = WARPS * 32;
constexpr int MAXW = 20;          // 16-byte W vectors per lane in flight (d = 5120 bf16 in one batch)
constexpr int MAX_D_SMEM = 8192;  // h row staged in shared memory (bf16: 16 KB, fp32: 32 KB)

// Block (b, kb) scores candidates kb*8 .. kb*8+7 of row b.  The block stages h[b] in shared
// memory (before waiting on the previous kernel: h does not depend on it), then each warp streams
// its W row with MAXW 16-byte loads per lane in flight and reduces with shuffles.  With probs
// requested, the block adds its candidate count to the row's ticket; the block completing the row
// computes the softmax and resets the ticket.
template <typename T>
__global__ void __launch_bounds__(THREADS) k_rescore(const T* __restrict__ h, const T* __restrict__ W,
                                                     const int32_t* __restrict__ idx, int d, int vocab, int K,
                                                     float* __restrict__ logits, float* __restrict__ probs,
                                                     uint32_t* __restrict__ tickets) {
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T* sh_h = reinterpret_cast<T*>(smem_raw);
  __shared__ float red[WARPS];
  __shared__ float s_bcast;
  __shared__ int s_last;
  const int kblocks = (K + WARPS - 1) / WARPS;
  const int b = blockIdx.x / kblocks, kb = blockIdx.x % kblocks;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int k = kb * WARPS + warp;
  const int n_here = min(WARPS, K - kb * WARPS);
  const T* x = h + (size_t)b * d;
  for (int c = threadIdx.x * PER; c < d; c += THREADS * PER)
    *reinterpret_cast<uint4*>(sh_h + c) = __ldg(reinterpret_cast<const uint4*>(x + c));
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  __syncthreads();
  if (k < K) {
    const int pair = b * K + k;
    const int v = idx[pair];
    const bool ok = v >= 0 && v < vocab;
    float acc = 0.f;
    if (ok) {
      const T* w = W + (size_t)v * d;
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
            Elem<T>::unpack(*reinterpret_cast<const uint4*>(sh_h + c), xf);
#pragma unroll
            for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
          }
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
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
  // softmax over the row's K logits (written by other blocks: read through L2)
  const float* z = logits + (size_t)b * K;
  float m = -INFINITY;
  for (int i = threadIdx.x; i < K; i += THREADS) m = fmaxf(m, __ldcg(z + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = red[0];
    for (int i = 1; i < WARPS; ++i) mm = fmaxf(mm, red[i]);
    s_bcast = mm;
  }
  __syncthreads();
  m = s_bcast;
  float ssum = 0.f;
  for (int i = threadIdx.x; i < K; i += THREADS) ssum += expf(__ldcg(z + i) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  __syncthreads();
  if (lane == 0) red[warp] = ssum;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int i = 0; i < WARPS; ++i) tot += red[i];
    s_bcast = 1.f / tot;
    tickets[b] = 0u;
  }
  __syncthreads();
  const float inv = s_bcast;
  for (int i = threadIdx.x; i < K; i += THREADS) probs[(size_t)b * K + i] = expf(__ldcg(z + i) - m) * inv;
}

// ------------------------------------------------------------------------------------------------
// Reordered rescoring for large batches: at B = 512, K = 256 the 131072 (row, candidate) pairs
// name about 88K distinct W rows, so fetching each distinct row from HBM once saves a third of the
// traffic.
//   k_link:    one thread per pair pushes the pair onto a per-W-row list (atomic exchange on
//              head[v]); the first pair of a row appends v to the list of distinct rows;
//              out-of-range ids go on one more list.
//   k_flatten: one thread per list lays its pairs out contiguously in a processing order.
//   k_rescore_stream (below) then scores the pairs in that order.
// Lists and counters live in the workspace and are left empty for the next call.

struct UniqState {
  uint32_t nuniq, done, bad_head, cursor;
};

__global__ void k_link(const int32_t* __restrict__ idx, int BK, int vocab, uint32_t* __restrict__ head,
                       uint32_t* __restrict__ next, uint32_t* __restrict__ uniq, UniqState* __restrict__ st) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx comes from the previous kernel
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= BK) return;
  const int v = idx[p];
  if (v < 0 || v >= vocab) {
    next[p] = atomicExch(&st->bad_head, (uint32_t)p + 1u);
    return;
  }
  const uint32_t old = atomicExch(&head[v], (uint32_t)p + 1u);
  next[p] = old;
  if (old == 0u) uniq[atomicAdd(&st->nuniq, 1u)] = (uint32_t)v;
}

// softmax of row b (K logits, written by other warps: read through L2) by one warp
__device__ void warp_softmax(const float* __restrict__ logits, float* __restrict__ probs, int b, int K) {
  const int lane = threadIdx.x & 31;
  const float* z = logits + (size_t)b * K;
  float m = -INFINITY;
  for (int i = lane; i < K; i += 32) m = fmaxf(m, __ldcg(z + i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float ssum = 0.f;
  for (int i = lane; i < K; i += 32) ssum += expf(__ldcg(z + i) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  const float inv = 1.f / ssum;
  for (int i = lane; i < K; i += 32) probs[(size_t)b * K + i] = expf(__ldcg(z + i) - m) * inv;
}

// lane 0 counts one finished pair of row b; returns (to all lanes) whether the row is complete
__device__ __forceinline__ bool finish_pair(uint32_t* tickets, int b, int K, bool with_probs) {
  if (!with_probs) return false;
  uint32_t last = 0;
  if ((threadIdx.x & 31) == 0) {
    __threadfence();
    last = atomicAdd(&tickets[b], 1u) == (uint32_t)(K - 1);
    if (last) __threadfence();
  }
  return __shfl_sync(0xFFFFFFFFu, last, 0) != 0;
}

// ------------------------------------------------------------------------------------------------
// Streaming rescoring for larger batches: one persistent block per SM walks a contiguous range of
// the pair list (in the given order, or row-major).  A ring of slots in shared memory holds, per
// pair, the W row and the h row, filled by 1-D bulk copies (cp.async.bulk) so that about 200 KB
// per SM stays in flight regardless of the compute warps' latency.  Warp 8 produces: its lanes
// resolve 32 pairs' (row, id) at a time, lane 0 issues the copies; warps 0-7 consume the slots in
// turn, reduce, write the logit and count it on the row's ticket.  When the pairs are ordered by
// W row (k_link + k_flatten), repeated rows are fetched back to back and served by L2, so HBM
// sees each distinct row about once.

constexpr int ST_CONSUMERS = 8;
constexpr int ST_THREADS = (ST_CONSUMERS + 1) * 32;
constexpr int ST_MAX_SLOTS = 16;
constexpr uint64_t ST_WAIT_NS = 2000000000ull;

// thread per distinct row: lay its pairs out contiguously in `order`; the extra thread u == nuniq
// appends the out-of-range pairs.  The lists are emptied for the next call.
__global__ void k_flatten(int BK, uint32_t* __restrict__ head, const uint32_t* __restrict__ next,
                          const uint32_t* __restrict__ uniq, UniqState* __restrict__ st, uint32_t* __restrict__ order) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  const uint32_t nuniq = __ldcg(&st->nuniq);
  if (u > nuniq || (int)u > BK) return;
  uint32_t* hp = (u == nuniq) ? &st->bad_head : head + __ldcg(uniq + u);
  uint32_t len = 0;
  for (uint32_t q = __ldcg(hp); q != 0u; q = __ldcg(next + q - 1)) ++len;
  if (len == 0) return;
  uint32_t off = atomicAdd(&st->cursor, len);
  for (uint32_t q = __ldcg(hp); q != 0u; q = __ldcg(next + q - 1)) order[off++] = q - 1;
  *hp = 0u;
}

template <typename T>
__global__ void __launch_bounds__(ST_THREADS, 1)
    k_rescore_stream(const T* __restrict__ h, const T* __restrict__ W, const int32_t* __restrict__ idx,
                     const uint32_t* __restrict__ order, int BK, int d, int vocab, int K, float* __restrict__ logits,
                     float* __restrict__ probs, uint32_t* __restrict__ tickets, UniqState* __restrict__ st,
                     int* __restrict__ status, int nslot) {
  using namespace sm100;
  constexpr int PER = Elem<T>::PER16;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[ST_MAX_SLOTS], empty[ST_MAX_SLOTS];
  __shared__ int slot_pair[ST_MAX_SLOTS], slot_valid[ST_MAX_SLOTS];
  __shared__ volatile int s_fail;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                         ~static_cast<uintptr_t>(127));
  const uint32_t row_bytes = (uint32_t)d * sizeof(T);
  const uint32_t slot_bytes = 2 * row_bytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int i0 = (int)((long long)BK * c / G), i1 = (int)((long long)BK * (c + 1) / G);
  const bool with_probs = probs != nullptr;
  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < nslot; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    fence_barrier_init();
  }
  __syncthreads();
  asm volatile("griddepcontrol.wait;" ::: "memory");  // idx / order come from earlier kernels

  if (warp == ST_CONSUMERS) {
    // ------------------------------------------------------------ producer warp
    for (int ib = i0; ib < i1 && !s_fail; ib += 32) {
      const int i = ib + lane;
      int pair = -1, v = -1;
      if (i < i1) {
        pair = order ? (int)__ldcg(order + i) : i;
        v = __ldg(idx + pair);
      }
      const int n = min(32, i1 - ib);
      for (int j = 0; j < n; ++j) {
        const int pj = __shfl_sync(0xFFFFFFFFu, pair, j);
        const int vj = __shfl_sync(0xFFFFFFFFu, v, j);
        if (lane == 0) {
          const int k = ib + j - i0;
          const int s = k % nslot;
          if (!mbar_wait(&empty[s], ((uint32_t)(k / nslot) & 1u) ^ 1u, ST_WAIT_NS)) {
            s_fail = 1;
            atomicOr(status, 1 << DH_ERR_TIMEOUT);
          } else {
            const bool ok = vj >= 0 && vj < vocab;
            slot_pair[s] = pj;
            slot_valid[s] = ok;
            unsigned char* dst = base + (size_t)s * slot_bytes;
            if (ok) {
              mbar_arrive_expect_tx(&full[s], slot_bytes);
              bulk_load(dst, W + (size_t)vj * d, row_bytes, &full[s]);
              bulk_load(dst + row_bytes, h + (size_t)(pj / K) * d, row_bytes, &full[s]);
            } else {
              mbar_arrive(&full[s]);
            }
          }
        }
        if (__shfl_sync(0xFFFFFFFFu, (int)s_fail, 0)) break;
      }
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    for (int k = warp; k < i1 - i0; k += ST_CONSUMERS) {
      const int s = k % nslot;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (uint32_t)(k / nslot) & 1u, ST_WAIT_NS))) {
        if (lane == 0) atomicOr(status, 1 << DH_ERR_TIMEOUT);
        s_fail = 1;
        break;
      }
      const int pair = slot_pair[s];
      const bool ok = slot_valid[s] != 0;
      float acc = 0.f;
      if (ok) {
        const T* wr = reinterpret_cast<const T*>(base + (size_t)s * slot_bytes);
        const T* hr = reinterpret_cast<const T*>(base + (size_t)s * slot_bytes + row_bytes);
        for (int cidx = lane * PER; cidx < d; cidx += 32 * PER) {
          float wf[PER], xf[PER];
          Elem<T>::unpack(*reinterpret_cast<const uint4*>(wr + cidx), wf);
          Elem<T>::unpack(*reinterpret_cast<const uint4*>(hr + cidx), xf);
#pragma unroll
          for (int e = 0; e < PER; ++e) acc = fmaf(xf[e], wf[e], acc);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      __syncwarp();
      if (lane == 0) {
        logits[pair] = ok ? acc : __int_as_float(0x7FC00000);
        mbar_arrive(&empty[s]);  // the slot is free once the warp has read it
      }
      const int b = pair / K;
      if (finish_pair(tickets, b, K, with_probs)) {
        warp_softmax(logits, probs, b, K);
        if (lane == 0) tickets[b] = 0u;
      }
    }
  }
  __syncthreads();
  // after a failed wait, let every copy issued into the ring land before the block exits
  if (threadIdx.x == 0 && s_fail) {
    const int n = i1 - i0;
    for (int s = 0; s < nslot && s < n; ++s) {
      const int last = s + ((n - 1 - s) / nslot) * nslot;  // the last item mapped to slot s
      mbar_wait(&full[s], (uint32_t)(last / nslot) & 1u, ST_WAIT_NS);
    }
  }
  // the last block out leaves the shared counters at zero for the next call
  if (threadIdx.x == 0 && st) {
    __threadfence();
    if (atomicAdd(&st->done, 1u) == (uint32_t)(G - 1)) {
      st->nuniq = 0u;
      st->cursor = 0u;
      st->done = 0u;
      __threadfence();
    }
  }
}

template <typename T>
cudaError_t launch_stream(const Ctx& c, const void* h, const void* W, const int32_t* idx, const uint32_t* order,
                          int B, int d, int vocab, int K, float* logits, float* probs, uint32_t* tickets,
                          UniqState* st, int* status) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore_stream<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  const size_t slot_bytes = 2 * (size_t)d * sizeof(T);
  const int avail = max_dynamic_smem(k_rescore_stream<T>, c.device) - 128;
  const int nslot = min(ST_MAX_SLOTS, (int)(avail / slot_bytes));
  if (nslot < 2) return cudaErrorInvalidConfiguration;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c.num_sms);
  cfg.blockDim = dim3(ST_THREADS);
  cfg.dynamicSmemBytes = 128 + (size_t)nslot * slot_bytes;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore_stream", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore_stream<T>, static_cast<const T*>(h), static_cast<const T*>(W), idx, order,
                         B * K, d, vocab, K, logits, probs, tickets, st, status, nslot);
  prof_after(c.stream);
  return e;
}

template <typename T>
cudaError_t run_uniq(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                     float* logits, float* probs, uint32_t* tickets, UniqState* st, uint32_t* head, uint32_t* next,
                     uint32_t* uniq, uint32_t* order, int* status) {
  const int BK = B * K;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((BK + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore_link", c.stream);
  cudaError_t e = cudaLaunchKernelEx(&cfg, k_link, idx, BK, vocab, head, next, uniq, st);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)((BK + 1 + 255) / 256));
  prof_before("rescore_flatten", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_flatten, BK, head, (const uint32_t*)next, (const uint32_t*)uniq, st, order);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return launch_stream<T>(c, h, W, idx, order, B, d, vocab, K, logits, probs, tickets, st, status);
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                int K, float* logits, float* probs, uint32_t* tickets) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_rescore<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the blocks may start while the stage-1 kernel drains; they
  // stage h and then wait (griddepcontrol.wait) for its results.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * ((K + WARPS - 1) / WARPS)));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = (size_t)d * sizeof(T);
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("rescore", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_rescore<T>, static_cast<const T*>(h), static_cast<const T*>(W), idx, d, vocab, K,
                         logits, probs, tickets);
  prof_after(c.stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

bool rescore_supported(int d) { return d <= MAX_D_SMEM; }

// The deduplicated path holds a W row in registers (MAXW 16-byte vectors per lane).
// The streaming kernels need the pair lists, distinct-row list and processing order in the
// workspace from this many pairs on.
bool rescore_uniq_used(int B, int d, int K, int dtype) {
  (void)dtype;
  return (long long)B * K >= 2048 && d <= MAX_D_SMEM;
}

cudaError_t launch_rescore_stream(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                  int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets,
                                  int* status) {
  if (dtype == DH_BF16)
    return launch_stream<__nv_bfloat16>(c, h, W, idx, nullptr, B, d, vocab, K, logits, probs, tickets, nullptr,
                                        status);
  return launch_stream<float>(c, h, W, idx, nullptr, B, d, vocab, K, logits, probs, tickets, nullptr, status);
}

size_t rescore_uniq_bytes(int B, int vocab, int K) {
  return align_up(sizeof(UniqState), 256) + align_up((size_t)vocab * 4, 256) + 3 * align_up((size_t)B * K * 4, 256);
}

cudaError_t launch_rescore_uniq(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets,
                                void* area, int* status) {
  char* a = static_cast<char*>(area);
  UniqState* st = reinterpret_cast<UniqState*>(a);
  a += align_up(sizeof(UniqState), 256);
  uint32_t* head = reinterpret_cast<uint32_t*>(a);
  a += align_up((size_t)vocab * 4, 256);
  uint32_t* next = reinterpret_cast<uint32_t*>(a);
  a += align_up((size_t)B * K * 4, 256);
  uint32_t* uniq = reinterpret_cast<uint32_t*>(a);
  a += align_up((size_t)B * K * 4, 256);
  uint32_t* order = reinterpret_cast<uint32_t*>(a);
  if (dtype == DH_BF16)
    return run_uniq<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, st, head, next, uniq, order,
                                   status);
  return run_uniq<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets, st, head, next, uniq, order, status);
}

cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                           int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
  return run<float>(c, h, W, idx, B, d, vocab, K, logits, probs, tickets);
}

}  // namespace dh
