// Stage 1 for small batches (B <= 8) in one cooperative launch: projection, vocabulary-wide
// low-rank scores with group summaries, and the exact top-K, with V streamed by TMA from the first
// instruction on.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the low-rank head scores the whole vocabulary to retrieve K candidates, then the full-rank head
// scores them.  At batch 1 the whole call moves about 40 MB (V dominates), so its cost is HBM time
// plus every serial dependency: h U must finish before t V, and the global top-K before rescoring.
// Running the steps in one resident grid removes the kernel boundaries between them.
//
// One block per SM (grid = SM count), 16 warps.  Each warp owns one or more groups of 64
// vocabulary ids and three 4 KB TMA stages of V (64 ids x 32 bf16 rows, or 16 fp32 rows).
//   P0  each warp issues the TMA loads of its first three stages (V does not depend on t).
//   P1  block c computes the partial products of h with the d-slice c of U for every (row, column)
//       and writes them to the workspace; grid barrier.
//   P2  every block sums the partials of every t element in the same fixed order (so all blocks
//       hold bit-identical t), rounds to the activation dtype and keeps t in shared memory;
//       block 0 also writes t for the selection's re-scoring step.
//   P3  each warp streams its groups: lane i scores ids 2i and 2i+1 of the group for all rows,
//       then a shuffle butterfly folds the 64 scores into the group record.  grid barrier.
//   P4  block b (< B) selects row b exactly from its records (select.cuh), reusing the V staging
//       buffers as scratch.
// Grid barriers are sense-reversing counters in the workspace; every wait (barrier or TMA) gives
// up after two seconds, raises DH_ERR_TIMEOUT in the status word, and the block drains its own
// outstanding copies before it exits.
#include "grid_sync.cuh"
#include "select.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

using namespace sm100;

constexpr int SB_THREADS = 512;
constexpr int SB_WARPS = SB_THREADS / 32;
constexpr int NS = 3;              // TMA stages per warp
constexpr int STAGE_BYTES = 4096;  // one box of 64 ids x (4096 / (64 * sizeof(T))) rows
constexpr int MAX_B = 8;
constexpr int MAX_BR = 2048;  // B * r values of t kept in shared memory
constexpr int CH = 40;        // projection rows per batch of loads in flight
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr size_t STAGE_REGION = (size_t)SB_WARPS * NS * STAGE_BYTES;

struct SbParams {
  const void* h;
  const void* U;
  const void* V;
  int B, d, r, vocab, K, n_groups;
  float* partial;  // [B*r][gridDim.x]
  void* t_out;     // [B][r] in the activation dtype
  GroupRec* recs;  // [B][n_groups]
  int32_t* idx_out;
  float* score_out;
  GridBar* bar;
  int* status;
};

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <typename T>
__global__ void __launch_bounds__(SB_THREADS, 1)
    k_small_b(const __grid_constant__ CUtensorMap tmV, SbParams p) {
  constexpr int ROWS = STAGE_BYTES / (GROUP * (int)sizeof(T));  // V rows per stage
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[SB_WARPS][NS];
  __shared__ float st[MAX_BR];       // t as fp32, [B][r]
  __shared__ float sh_h[MAX_B * CH];  // the block's slice of h
  __shared__ volatile int s_fail;

  unsigned char* stages = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int B = p.B, r = p.r, BR = p.B * p.r;
  const int spg = r / ROWS;  // stages per group

  // this block's groups, and this warp's share of them
  const int g0 = (int)((long long)p.n_groups * c / G), g1 = (int)((long long)p.n_groups * (c + 1) / G);
  const int my_groups = (g1 - g0 > warp) ? (g1 - g0 - warp + SB_WARPS - 1) / SB_WARPS : 0;
  const int total_stages = my_groups * spg;

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int w = 0; w < SB_WARPS; ++w)
      for (int s = 0; s < NS; ++s) mbar_init(&full[w][s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  unsigned char* wstage = stages + (size_t)warp * NS * STAGE_BYTES;
  int issued = 0;    // stages this warp has asked TMA for (meaningful in lane 0)
  int consumed = 0;  // stages this warp has waited for and read
  auto issue = [&](int q) {  // stage q of this warp into slot q % NS (lane 0 only)
    const int g = g0 + warp + (q / spg) * SB_WARPS;
    const int row0 = (q % spg) * ROWS;
    uint64_t* bar = &full[warp][q % NS];
    mbar_arrive_expect_tx(bar, STAGE_BYTES);
    tma_load_2d(wstage + (q % NS) * STAGE_BYTES, &tmV, g * GROUP, row0, bar);
    issued = q + 1;
  };

  // ---------------------------------------------------------------- P0: V prefetch
  if (lane == 0) {
    prefetch_tmap(&tmV);
    for (int q = 0; q < NS && q < total_stages; ++q) issue(q);
  }

  // ---------------------------------------------------------------- P1: projection partials
  {
    const T* h = static_cast<const T*>(p.h);
    const T* U = static_cast<const T*>(p.U);
    const int i0 = (int)((long long)p.d * c / G), i1 = (int)((long long)p.d * (c + 1) / G);
    const int npairs = r / 2;
    for (int base = i0; base < i1; base += CH) {
      const int n = min(CH, i1 - base);
      __syncthreads();
      for (int e = threadIdx.x; e < B * n; e += blockDim.x) {
        const int b = e / n, i = e - b * n;
        sh_h[b * CH + i] = Elem<T>::to_f(h[(size_t)b * p.d + base + i]);
      }
      __syncthreads();
      for (int w = threadIdx.x; w < npairs * B; w += blockDim.x) {
        const int b = w / npairs, jp = w - b * npairs;
        const T* up = U + (size_t)base * r + 2 * jp;
        float u[CH][2];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          if (i < n) {
            u[i][0] = Elem<T>::to_f(up[(size_t)i * r]);
            u[i][1] = Elem<T>::to_f(up[(size_t)i * r + 1]);
          }
        }
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          if (i < n) {
            const float hv = sh_h[b * CH + i];
            a0 = fmaf(hv, u[i][0], a0);
            a1 = fmaf(hv, u[i][1], a1);
          }
        }
        // several load batches of the same slice accumulate in place
        float* o = p.partial + (size_t)(b * r + 2 * jp) * G + c;
        if (base == i0) {
          o[0] = a0;
          o[G] = a1;
        } else {
          o[0] += a0;
          o[G] += a1;
        }
      }
    }
  }
  if (!grid_sync(p.bar, gridDim.x, WAIT_NS, p.status, &s_fail)) goto drain;

  // ---------------------------------------------------------------- P2: t, identical in every block
  {
    int L = 1;  // lanes per output (power of two, <= 32)
    while (L < 32 && L * 2 * BR <= SB_THREADS) L *= 2;
    const int per_pass = SB_THREADS / L;
    const int sub = lane % L;
    for (int e0 = 0; e0 < BR; e0 += per_pass) {
      const int e = e0 + (int)threadIdx.x / L;
      float acc = 0.f;
      if (e < BR) {
        const float* src = p.partial + (size_t)e * G;
        for (int k0 = sub; k0 < G; k0 += 16 * L) {
          float v[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) v[q] = (k0 + q * L < G) ? __ldcg(src + k0 + q * L) : 0.f;
#pragma unroll
          for (int q = 0; q < 16; ++q) acc += v[q];
        }
      }
      for (int o = L / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
      if (sub == 0 && e < BR) {
        const T tv = Elem<T>::from_f(acc);
        st[e] = Elem<T>::to_f(tv);
        if (c == 0) static_cast<T*>(p.t_out)[e] = tv;
      }
    }
  }
  __syncthreads();

  // ---------------------------------------------------------------- P3: stream V, group records
  {
    for (int k = 0; k < my_groups; ++k) {
      const int g = g0 + warp + k * SB_WARPS;
      float acc[MAX_B][2];
#pragma unroll
      for (int b = 0; b < MAX_B; ++b) acc[b][0] = acc[b][1] = 0.f;
      for (int rb = 0; rb < spg; ++rb) {
        const int q = k * spg + rb;
        // the outcome is made warp-uniform so that the lanes never split around __syncwarp
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[warp][q % NS], (uint32_t)(q / NS) & 1u, WAIT_NS))) {
          if (lane == 0) atomicOr(p.status, 1 << DH_ERR_TIMEOUT);
          s_fail = 1;
          goto drain;
        }
        consumed = q + 1;
        const unsigned char* tile = wstage + (q % NS) * STAGE_BYTES;
        const int j0 = rb * ROWS;
#pragma unroll 8
        for (int j = 0; j < ROWS; ++j) {
          float v0, v1;
          if (sizeof(T) == 2) {
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(tile + j * 128 + lane * 4);
            v0 = __uint_as_float(w2 << 16);
            v1 = __uint_as_float(w2 & 0xFFFF0000u);
          } else {
            const float2 f2 = *reinterpret_cast<const float2*>(tile + j * 256 + lane * 8);
            v0 = f2.x;
            v1 = f2.y;
          }
#pragma unroll
          for (int b = 0; b < MAX_B; ++b) {
            if (b < B) {
              const float tb = st[b * r + j0 + j];
              acc[b][0] = fmaf(tb, v0, acc[b][0]);
              acc[b][1] = fmaf(tb, v1, acc[b][1]);
            }
          }
        }
        __syncwarp();
        if (lane == 0 && q + NS < total_stages) {
          fence_proxy_async_smem();
          issue(q + NS);
        }
      }
      const uint32_t id0 = (uint32_t)(g * GROUP + 2 * lane);
#pragma unroll
      for (int b = 0; b < MAX_B; ++b) {
        if (b < B) {
          Top2 sm;
          sm.init();
          if ((int)id0 < p.vocab) sm.push(acc[b][0], id0);
          if ((int)id0 + 1 < p.vocab) sm.push(acc[b][1], id0 + 1);
#pragma unroll
          for (int x = 1; x < 32; x <<= 1) sm.merge_shfl(0xFFFFFFFFu, x);
          if (lane == 0) p.recs[(size_t)b * p.n_groups + g] = sm.record((uint32_t)(g * GROUP));
        }
      }
    }
  }
  if (!grid_sync(p.bar, gridDim.x, WAIT_NS, p.status, &s_fail)) goto drain;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---------------------------------------------------------------- P4: exact top-K of row c
  if (c < B) {
    const T* tr = static_cast<const T*>(p.t_out) + (size_t)c * r;
    sel::select_row<T>(stages, p.recs + (size_t)c * p.n_groups, tr, static_cast<const T*>(p.V), r, p.vocab,
                       p.K, p.idx_out + (size_t)c * p.K, p.score_out + (size_t)c * p.K);
  }
  return;

drain:
  // a failed wait: let every copy this warp issued and did not read land before the block exits
  if (lane == 0)
    for (int q = consumed; q < issued; ++q) mbar_wait(&full[warp][q % NS], (uint32_t)(q / NS) & 1u, WAIT_NS);
  __syncwarp();
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

template <typename T>
cudaError_t run(const Ctx& c, const SbParams& p0) {
  constexpr int ROWS = STAGE_BYTES / (GROUP * (int)sizeof(T));
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_small_b<T>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  const size_t smem = STAGE_REGION + 1024;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_small_b<T>, SB_THREADS, smem);
  if (e != cudaSuccess) return note_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor(k_small_b)");
  const int G = min(c.num_sms * max(per_sm, 0), 1024);
  if (G < 1) return note_error(cudaErrorInvalidConfiguration, "k_small_b: no resident block fits");

  EncodeTiledFn fn = encode_fn();
  if (!fn) return note_error(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  CUtensorMap tmV;
  cuuint64_t dims[2] = {(cuuint64_t)p0.vocab, (cuuint64_t)p0.r};
  cuuint64_t strides[1] = {(cuuint64_t)p0.vocab * sizeof(T)};
  cuuint32_t box[2] = {(cuuint32_t)GROUP, (cuuint32_t)ROWS};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&tmV, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(p0.V), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(V, small batch)");

  SbParams p = p0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3(SB_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("small_b", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_small_b<T>, tmV, p);
  prof_after(c.stream);
  if (e != cudaSuccess) return note_error(e, "cudaLaunchKernelEx(k_small_b)");
  return note_error(cudaGetLastError(), "k_small_b launch");
}

}  // namespace

bool small_b_supported(int B, int r, int dtype) {
  const int rows = STAGE_BYTES / (GROUP * (dtype == DH_BF16 ? 2 : 4));
  return B >= 1 && B <= MAX_B && B * r <= MAX_BR && r % rows == 0 && r % 2 == 0;
}

size_t small_b_partial_floats(int B, int r) { return (size_t)1024 * B * r; }

cudaError_t launch_small_b(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r,
                           int vocab, int K, int dtype, float* partial, void* t_out, GroupRec* recs,
                           int32_t* idx_out, float* score_out, void* bar, int* status) {
  SbParams p;
  p.h = h;
  p.U = U;
  p.V = V;
  p.B = B;
  p.d = d;
  p.r = r;
  p.vocab = vocab;
  p.K = K;
  p.n_groups = (vocab + GROUP - 1) / GROUP;
  p.partial = partial;
  p.t_out = t_out;
  p.recs = recs;
  p.idx_out = idx_out;
  p.score_out = score_out;
  p.bar = static_cast<GridBar*>(bar);
  p.status = status;
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, p);
  return run<float>(c, p);
}

}  // namespace dh
