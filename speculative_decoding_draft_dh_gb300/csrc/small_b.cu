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
// One block per SM (grid = SM count), 16 warps.  Each block owns a contiguous run of 256-id
// tiles and streams them in sets of four: a stage is four TMA boxes of 256 ids x 16 bf16 rows (8
// fp32 rows) = 32 KB, i.e. 2 KB contiguous per V row, with six stages in flight.
//   P0  thread 0 issues the TMA loads of the first six stages (V does not depend on t).
//   P1  block c computes the partial products of h with the d-slice c of U for every (row, column)
//       and writes them to the workspace; grid barrier.
//   P2  every block sums the partials of every t element in the same fixed order (so all blocks
//       hold bit-identical t), rounds to the activation dtype and keeps t in shared memory;
//       block 0 also writes t for the selection's re-scoring step.
//   P3  warp w scores the 64-id group w of the current set: lane i accumulates ids 2i and 2i+1
//       for all rows over the stages; after the last band a shuffle butterfly folds the 64
//       scores into the group record.  A block barrier per stage frees its slot for the next
//       TMA load.  grid barrier.
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
constexpr int TILE = 256;            // vocabulary ids per TMA box
constexpr int SET_TILES = 4;         // tiles streamed together (16 warps x 64 ids)
constexpr int NS = 6;                // stages in flight
constexpr int STAGE_BYTES = 32768;   // SET_TILES boxes of 256 ids x (32 KB / 4 / 256 / sizeof(T)) rows
constexpr int MAX_B = 8;
constexpr int MAX_BR = 2048;  // B * r values of t kept in shared memory
constexpr int CH = 40;        // projection rows per batch of loads in flight
constexpr int RED = 48;       // partial sums per lane in flight in the t reduction
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr size_t STAGE_REGION = (size_t)NS * STAGE_BYTES;

struct SbParams {
  const void* h;
  const void* U;
  const void* V;
  int B, d, r, vocab, K, n_groups, n_tiles;
  float* partial;  // [B*r][gridDim.x]
  void* t_out;     // [B][r] in the activation dtype
  GroupRec* recs;  // [B][n_groups]
  int32_t* idx_out;
  float* score_out;
  GridBar* bar;
  int* status;
};

// Two adjacent values of row-major storage as floats (4-byte load for bf16, 8-byte for fp32).
template <typename T>
__device__ __forceinline__ void load_pair(const T* p, float& a, float& b);
template <>
__device__ __forceinline__ void load_pair<__nv_bfloat16>(const __nv_bfloat16* p, float& a, float& b) {
  const uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
  a = __uint_as_float(w << 16);
  b = __uint_as_float(w & 0xFFFF0000u);
}
template <>
__device__ __forceinline__ void load_pair<float>(const float* p, float& a, float& b) {
  const float2 f = __ldg(reinterpret_cast<const float2*>(p));
  a = f.x;
  b = f.y;
}

template <typename T>
__global__ void __launch_bounds__(SB_THREADS, 1)
    k_small_b(const __grid_constant__ CUtensorMap tmV, SbParams p) {
  constexpr int RB = STAGE_BYTES / (SET_TILES * TILE * (int)sizeof(T));  // V rows per stage
  constexpr int ROW_BYTES = TILE * (int)sizeof(T);                        // one box row
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[NS];
  __shared__ float st[MAX_BR];        // t as fp32, [B][r]
  __shared__ float sh_h[MAX_B * CH];  // the block's slice of h
  __shared__ volatile int s_fail;

  unsigned char* stages = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int B = p.B, r = p.r, BR = p.B * p.r;
  const int bands = r / RB;  // stages per tile set

  // this block's 256-id tiles, streamed in sets of up to four
  const int t0 = (int)((long long)p.n_tiles * c / G), t1 = (int)((long long)p.n_tiles * (c + 1) / G);
  const int n_sets = (t1 - t0 + SET_TILES - 1) / SET_TILES;
  const int total_stages = n_sets * bands;

  if (threadIdx.x == 0) {
    s_fail = 0;
    for (int s = 0; s < NS; ++s) mbar_init(&full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  int issued = 0;    // stages asked of TMA (thread 0)
  int consumed = 0;  // stages read by the block
  auto issue = [&](int q) {  // stage q into slot q % NS (thread 0 only)
    const int set = q / bands, band = q % bands;
    const int tile = t0 + set * SET_TILES;
    const int nt = min(SET_TILES, t1 - tile);
    uint64_t* bar = &full[q % NS];
    mbar_arrive_expect_tx(bar, (uint32_t)(nt * TILE * RB * sizeof(T)));
    for (int k = 0; k < nt; ++k)
      tma_load_2d(stages + (size_t)(q % NS) * STAGE_BYTES + (size_t)k * RB * ROW_BYTES, &tmV, (tile + k) * TILE,
                  band * RB, bar);
    issued = q + 1;
  };

  // ---------------------------------------------------------------- P0: V prefetch
  if (threadIdx.x == 0) {
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
        for (int i = 0; i < CH; ++i)
          if (i < n) load_pair<T>(up + (size_t)i * r, u[i][0], u[i][1]);
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
        for (int k0 = sub; k0 < G; k0 += RED * L) {
          float v[RED];
#pragma unroll
          for (int q = 0; q < RED; ++q) v[q] = (k0 + q * L < G) ? __ldcg(src + k0 + q * L) : 0.f;
#pragma unroll
          for (int q = 0; q < RED; ++q) acc += v[q];
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
    // warp w scores group (w % 4) of tile (w / 4) of the current set; lane i owns ids 2i, 2i+1
    const int k_tile = warp / 4, g_in_tile = warp % 4;
    float acc[MAX_B][2];
#pragma unroll
    for (int b = 0; b < MAX_B; ++b) acc[b][0] = acc[b][1] = 0.f;
    for (int q = 0; q < total_stages; ++q) {
      const int set = q / bands, band = q % bands;
      const int tile = t0 + set * SET_TILES + k_tile;
      const bool mine = tile < t1;
      // the outcome is made warp-uniform so that the lanes never split around the barriers
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&full[q % NS], (uint32_t)(q / NS) & 1u, WAIT_NS))) {
        if (lane == 0) atomicOr(p.status, 1 << DH_ERR_TIMEOUT);
        s_fail = 1;
      }
      __syncthreads();
      if (s_fail) goto drain;
      consumed = q + 1;
      if (mine) {
        const unsigned char* box = stages + (size_t)(q % NS) * STAGE_BYTES + (size_t)k_tile * RB * ROW_BYTES +
                                   (size_t)(g_in_tile * GROUP + 2 * lane) * sizeof(T);
        const int j0 = band * RB;
#pragma unroll
        for (int j = 0; j < RB; ++j) {
          float v0, v1;
          if (sizeof(T) == 2) {
            const uint32_t w2 = *reinterpret_cast<const uint32_t*>(box + j * ROW_BYTES);
            v0 = __uint_as_float(w2 << 16);
            v1 = __uint_as_float(w2 & 0xFFFF0000u);
          } else {
            const float2 f2 = *reinterpret_cast<const float2*>(box + j * ROW_BYTES);
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
      }
      __syncthreads();  // every warp is done with slot q % NS
      if (threadIdx.x == 0 && q + NS < total_stages) {
        fence_proxy_async_smem();
        issue(q + NS);
      }
      if (band == bands - 1) {
        if (mine) {
          const int g = tile * (TILE / GROUP) + g_in_tile;
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
              if (lane == 0 && g < p.n_groups) p.recs[(size_t)b * p.n_groups + g] = sm.record((uint32_t)(g * GROUP));
            }
          }
        }
#pragma unroll
        for (int b = 0; b < MAX_B; ++b) acc[b][0] = acc[b][1] = 0.f;
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
  // a failed wait: let every copy the block issued and did not read land before it exits
  if (threadIdx.x == 0)
    for (int q = consumed; q < issued; ++q) mbar_wait(&full[q % NS], (uint32_t)(q / NS) & 1u, WAIT_NS);
  __syncthreads();
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
  constexpr int RB = STAGE_BYTES / (SET_TILES * TILE * (int)sizeof(T));
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
  cuuint32_t box[2] = {(cuuint32_t)TILE, (cuuint32_t)RB};
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
  const int rows = STAGE_BYTES / (SET_TILES * TILE * (dtype == DH_BF16 ? 2 : 4));
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
  p.n_tiles = (vocab + TILE - 1) / TILE;
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
