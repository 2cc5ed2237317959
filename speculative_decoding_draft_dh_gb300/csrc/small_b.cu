// Stage 1 for small batches (B <= 8): two kernels chained by programmatic dependent launch, so
// that V streams from HBM while the projection that it will be multiplied with is still being
// computed.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the low-rank head scores the whole vocabulary to retrieve K candidates, then the full-rank head
// scores them.  At batch 1 the whole call moves about 40 MB (V dominates), so its cost is HBM time
// plus every serial dependency: h U must finish before t V, and the global top-K before rescoring.
//
// k_proj_small (grid: two blocks per SM, each a slice of d): waits for the previous kernel (h may
//   come from it), loads its slice of U (and h), signals its dependents may launch, multiplies, and
//   adds its partial t into one of eight 64-bit fixed-point accumulator copies (scale 2^32) with
//   integer atomics, which are exact and order independent, so t is deterministic.  There is no
//   final pass: the readers of t sum the copies themselves (acc_to_t).
// k_scores_lsu (default; r a multiple of 64; one 4-warp block per 256-id tile, all blocks resident):
//   before waiting for the projection, each warp puts up to 32 of its V rows on chip, 16 in
//   registers and 16 bulk-copied into shared memory (cp.async.bulk on an mbarrier), so at r = 128
//   the whole of V is in flight while t is computed.  After the wait it derives t from the
//   accumulators, multiplies, adds the four warps' partial sums in a fixed order and folds each
//   group of 64 ids into its record.  Rows beyond 32 per warp stream through registers.
// k_scores_small (TMA variant for other r; one block per SM, 16 warps): issues the TMA loads of its
//   first six 32 KB stages of V before waiting for the projection, then streams its run of 256-id
//   tiles in sets of four: a stage is four boxes of 256 ids x 16 bf16 rows (8 fp32 rows), 2 KB
//   contiguous per V row.  Warp w folds the 64 scores of group w of the set into its record; a
//   block barrier per stage frees the stage's slot for the next TMA load.
// k_select (select.cu) then picks the exact top-K per row from the records, deriving t from the
// accumulators for its refinement step, and clears the accumulators for the next call.
// Every TMA or bulk-copy wait gives up after two seconds and raises DH_ERR_TIMEOUT in the status
// word.
#include <cstdlib>
#include <cstring>

#include "select.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

using namespace sm100;

constexpr int SB_THREADS = 512;
constexpr int TILE = 256;           // vocabulary ids per TMA box
constexpr int SET_TILES = 4;        // tiles streamed together (16 warps x 64 ids)
constexpr int NS = 6;               // stages in flight
constexpr int STAGE_BYTES = 32768;  // SET_TILES boxes of 256 ids x (32 KB / 4 / 256 / sizeof(T)) rows
constexpr int MAX_B = 8;
constexpr int MAX_BR = ACC_MAX_BR;  // B * r values of t
constexpr int PJ_THREADS = 256;
constexpr int PJ_GROUPS = 4;        // row groups per block in the projection (reduced in smem)
constexpr int CH = 12;              // projection rows per thread in one batch of loads
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr size_t STAGE_REGION = (size_t)NS * STAGE_BYTES;
constexpr float FIX_SCALE = 4294967296.0f;  // 2^32

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

struct ProjSmall {
  const void* h;
  const void* U;
  int B, d, r;
  unsigned long long* acc;  // [ACC_COPIES][B*r] fixed-point accumulators (zero between calls)
  int* status;              // workspace status word
};

// Fixed-point range: a block's partial v converts to round(v * 2^32) in a signed 64-bit integer,
// so |v| must stay below 2^31; the integer sums are exact (modulo 2^64) as long as every final
// |t| stays below 2^31 too.  Beyond that the conversion saturates: the block raises
// DH_ERR_UNSUPPORTED in the status word and the call's outputs are unspecified.
constexpr float FIX_LIMIT = 2147483648.0f;  // 2^31

// NB = B (1..MAX_B): the accumulators are sized for the batch, so that at batch 1 a projection
// block holds few registers and the scores kernel's blocks, launched early, fit beside it.
template <typename T, int NB>
__global__ void __launch_bounds__(PJ_THREADS) k_proj_small(ProjSmall p) {
  constexpr int PAIRS = PJ_THREADS / PJ_GROUPS;  // column pairs per pass
  __shared__ float red[PJ_GROUPS][NB * 2 * PAIRS];  // per-group partials of this pass, [b][2 * pair]
  const T* h = static_cast<const T*>(p.h);
  const T* U = static_cast<const T*>(p.U);
  const int B = p.B, r = p.r, BR = B * r, npairs = r / 2;
  const int G = gridDim.x, c = blockIdx.x;
  const int i0 = (int)((long long)p.d * c / G), i1 = (int)((long long)p.d * (c + 1) / G);
  const int rows = i1 - i0;
  const int grp = threadIdx.x / PAIRS;  // row group of this thread
  const int lt = threadIdx.x % PAIRS;
  const int per_grp = (rows + PJ_GROUPS - 1) / PJ_GROUPS;
  const int g0 = i0 + grp * per_grp, g1 = min(i1, g0 + per_grp);
  bool triggered = false;
  // launched with programmatic dependent launch: h may come from the kernel before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // each thread owns one column pair for every row of the batch, so U is read once
  for (int jp0 = 0; jp0 < npairs; jp0 += PAIRS) {
    const int jp = jp0 + lt;
    const bool on = jp < npairs;
    float a[NB][2];
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) a[bb][0] = a[bb][1] = 0.f;
    for (int base = g0; base < g1; base += CH) {
      const int n = min(CH, g1 - base);
      float u[CH][2];
      if (on) {
#pragma unroll
        for (int i = 0; i < CH; ++i)
          if (i < n) load_pair<T>(U + (size_t)(base + i) * r + 2 * jp, u[i][0], u[i][1]);
      }
      if (!triggered) {  // U is in flight: the scores kernel may start streaming V
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        triggered = true;
      }
      if (on) {
#pragma unroll
        for (int i = 0; i < CH; ++i) {
          if (i < n) {
#pragma unroll
            for (int bb = 0; bb < NB; ++bb) {
              const float hv = Elem<T>::to_f(h[(size_t)bb * p.d + base + i]);
              a[bb][0] = fmaf(hv, u[i][0], a[bb][0]);
              a[bb][1] = fmaf(hv, u[i][1], a[bb][1]);
            }
          }
        }
      }
    }
    // add the row groups' partials in a fixed order, then one integer atomic per (b, j)
#pragma unroll
    for (int bb = 0; bb < NB; ++bb) {
      red[grp][bb * 2 * PAIRS + 2 * lt] = a[bb][0];
      red[grp][bb * 2 * PAIRS + 2 * lt + 1] = a[bb][1];
    }
    __syncthreads();
    for (int q2 = threadIdx.x; q2 < B * 2 * PAIRS; q2 += PJ_THREADS) {
      const int bb = q2 / (2 * PAIRS), jj = 2 * jp0 + (q2 % (2 * PAIRS));
      if (jj < r) {
        float v = 0.f;
#pragma unroll
        for (int q = 0; q < PJ_GROUPS; ++q) v += red[q][q2];
        if (!(fabsf(v) < FIX_LIMIT)) atomicOr(p.status, 1 << DH_ERR_UNSUPPORTED);
        const long long fx = __float2ll_rn(v * FIX_SCALE);
        atomicAdd(p.acc + (size_t)(c % ACC_COPIES) * BR + bb * r + jj, (unsigned long long)fx);
      }
    }
    __syncthreads();
  }
  if (!triggered) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Vector form of the projection (r / (16 / sizeof(T)) a power of two up to PV_THREADS): one light
// block of PV_THREADS threads per SM, so that every block of the scores kernel fits beside it
// and issues its V loads as soon as it is launched.  Block c owns a slice of d; thread t loads one
// 16-byte vector (VEC columns) of row (t / tpr) of each pass of rpp rows, all passes in flight at
// once; the rpp row groups' partials are added in a fixed order in shared memory and each (b, j)
// is added once into the fixed-point accumulators.
constexpr int PV_THREADS = 128;
constexpr int PV_LOADS = 8;  // 16-byte loads per thread in flight

bool proj_vec_ok(int r, int elem) {
  const int tpr = r * elem / 16;
  return r * elem % 16 == 0 && tpr >= 1 && tpr <= PV_THREADS && (tpr & (tpr - 1)) == 0;
}

template <typename T, int NB>
__global__ void __launch_bounds__(PV_THREADS) k_proj_vec(ProjSmall p) {
  constexpr int VEC = Elem<T>::PER16;
  extern __shared__ float pv_red[];  // [rpp][NB * r]
  const T* h = static_cast<const T*>(p.h);
  const T* U = static_cast<const T*>(p.U);
  const int r = p.r, BR = p.B * r;
  const int tpr = r / VEC, rpp = PV_THREADS / tpr;
  const int G = gridDim.x, c = blockIdx.x;
  const int i0 = (int)((long long)p.d * c / G), i1 = (int)((long long)p.d * (c + 1) / G);
  const int grp = threadIdx.x / tpr, col = (threadIdx.x % tpr) * VEC;
  float acc[NB][VEC];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[b][e] = 0.f;
  // launched with programmatic dependent launch: h may come from the kernel before this one
  asm volatile("griddepcontrol.wait;" ::: "memory");
  bool triggered = false;
  for (int base = i0; base < i1; base += PV_LOADS * rpp) {
    uint4 u[PV_LOADS];
#pragma unroll
    for (int q = 0; q < PV_LOADS; ++q) {
      const int row = base + q * rpp + grp;
      u[q] = row < i1 ? __ldg(reinterpret_cast<const uint4*>(U + (size_t)row * r + col)) : make_uint4(0, 0, 0, 0);
    }
    if (!triggered) {  // U is in flight: the scores kernel may launch and start streaming V
      asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      triggered = true;
    }
#pragma unroll
    for (int q = 0; q < PV_LOADS; ++q) {
      const int row = base + q * rpp + grp;
      if (row < i1) {
#pragma unroll
        for (int b = 0; b < NB; ++b) Elem<T>::axpy16(Elem<T>::scalar_of(h[(size_t)b * p.d + row]), u[q], acc[b]);
      }
    }
  }
  if (!triggered) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < VEC; ++e) pv_red[(size_t)grp * BR + b * r + col + e] = acc[b][e];
  __syncthreads();
  for (int q = threadIdx.x; q < BR; q += PV_THREADS) {
    float v = 0.f;
    for (int g = 0; g < rpp; ++g) v += pv_red[(size_t)g * BR + q];
    if (!(fabsf(v) < FIX_LIMIT)) atomicOr(p.status, 1 << DH_ERR_UNSUPPORTED);
    atomicAdd(p.acc + (size_t)(c % ACC_COPIES) * BR + q, (unsigned long long)__float2ll_rn(v * FIX_SCALE));
  }
}

struct ScoresSmall {
  const unsigned long long* acc;  // the projection's accumulators: t = acc_to_t(acc, B*r, e)
  int B, r, vocab, n_groups, n_tiles;
  GroupRec* recs;
  uint32_t* gkeys;  // [B][n_groups]: order-preserving key of each group's best score (0: empty group)
  int* status;
};

template <typename T, int NB>
__global__ void __launch_bounds__(SB_THREADS, 1)
    k_scores_small(const __grid_constant__ CUtensorMap tmV, ScoresSmall p) {
  constexpr int RB = STAGE_BYTES / (SET_TILES * TILE * (int)sizeof(T));  // V rows per stage
  constexpr int ROW_BYTES = TILE * (int)sizeof(T);                        // one box row
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t full[NS];
  __shared__ float st[MAX_BR];  // t as fp32, [B][r]
  __shared__ volatile int s_fail;

  unsigned char* stages = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                           ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;
  const int r = p.r, BR = p.B * p.r;
  const int bands = r / RB;  // stages per tile set
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

  // V does not depend on t: start streaming before waiting for the projection
  if (threadIdx.x == 0) {
    prefetch_tmap(&tmV);
    for (int q = 0; q < NS && q < total_stages; ++q) issue(q);
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int e = threadIdx.x; e < BR; e += blockDim.x) st[e] = acc_to_t<T>(p.acc, BR, e);
  __syncthreads();

  {
    // warp w scores group (w % 4) of tile (w / 4) of the current set; lane i owns ids 2i, 2i+1
    const int k_tile = warp / 4, g_in_tile = warp % 4;
    float acc[NB][2];
#pragma unroll
    for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.f;
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
          for (int b = 0; b < NB; ++b) {
            const float tb = st[b * r + j0 + j];
            acc[b][0] = fmaf(tb, v0, acc[b][0]);
            acc[b][1] = fmaf(tb, v1, acc[b][1]);
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
          for (int b = 0; b < NB; ++b) {
            Top2 sm;
            sm.init();
            if ((int)id0 < p.vocab) sm.push(acc[b][0], id0);
            if ((int)id0 + 1 < p.vocab) sm.push(acc[b][1], id0 + 1);
#pragma unroll
            for (int x = 1; x < 32; x <<= 1) sm.merge_shfl(0xFFFFFFFFu, x);
            if (lane == 0 && g < p.n_groups) {
              p.recs[(size_t)b * p.n_groups + g] = sm.record((uint32_t)(g * GROUP));
              p.gkeys[(size_t)b * p.n_groups + g] = sm.i1 == 0xFFFFFFFFu ? 0u : fkey(sm.v1);
            }
          }
        }
#pragma unroll
        for (int b = 0; b < NB; ++b) acc[b][0] = acc[b][1] = 0.f;
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

// LSU variant of the scores kernel: one block per 256-id tile (bf16; 128 ids for fp32), four warps
// splitting the rank dimension (warp w takes rows [w r/4, (w+1) r/4)).  Lane i owns ids
// PER*i .. PER*i + PER-1 of the tile, one 16-byte vector per row.  Before waiting for the
// projection each warp puts its first LSU_BATCH rows into registers and bulk-copies the next
// LSU_SROWS rows (one contiguous segment of the tile per row) into shared memory; rows beyond
// those stream through registers after the wait.  The four warps' partial sums are added in a
// fixed order through shared memory (aliasing the staged rows), then warp g folds group g of the
// tile into its record.
constexpr int LSU_WARPS = 4;
constexpr int LSU_BATCH = 16;  // rows per warp in registers
constexpr int LSU_SROWS = 16;  // rows per warp staged in shared memory
constexpr int LSU_SEG = 512;   // bytes of one row segment of a tile (32 lanes x 16 bytes)

template <typename T, int NB>
__global__ void __launch_bounds__(LSU_WARPS * 32) k_scores_lsu(const T* __restrict__ V, ScoresSmall p) {
  constexpr int PER = Elem<T>::PER16;   // ids per lane (8 bf16 / 4 fp32)
  constexpr int TW = 32 * PER;          // ids per block tile
  static_assert(TW * (int)sizeof(T) == LSU_SEG, "a tile row is one 512-byte segment");
  static_assert(LSU_WARPS * NB * TW * 4 <= LSU_WARPS * LSU_SROWS * LSU_SEG, "partial sums fit the staging area");
  __shared__ __align__(128) unsigned char vs[LSU_WARPS][LSU_SROWS][LSU_SEG];
  __shared__ typename Elem<T>::Scalar st[MAX_BR];  // t, in the form axpy16 takes
  __shared__ uint64_t vbar[LSU_WARPS];
  __shared__ int s_fail;
  float(*part)[NB][TW] = reinterpret_cast<float(*)[NB][TW]>(&vs[0][0][0]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, r = p.r, BR = B * r;
  const int tile0 = blockIdx.x * TW;
  const int c0 = tile0 + lane * PER;
  const bool valid = c0 < p.vocab;  // vocab is a multiple of PER
  const int rq = r / LSU_WARPS;     // rows per warp (r is a multiple of 64 on this path)
  const int j0 = warp * rq;
  const int nreg = min(LSU_BATCH, rq);
  const int nsm = min(LSU_SROWS, rq - nreg);
  const T* vp = V + (valid ? c0 : 0);
  uint4 raw[LSU_BATCH];
#pragma unroll
  for (int q = 0; q < LSU_BATCH; ++q)
    raw[q] = (valid && q < nreg) ? ld_nc_v4(vp + (size_t)(j0 + q) * p.vocab) : make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) s_fail = 0;
  // staged rows: lane 0 of each warp bulk-copies them on the warp's own mbarrier
  const uint32_t seg_bytes = (uint32_t)(min(TW, p.vocab - tile0) * (int)sizeof(T));  // multiple of 16
  if (lane == 0) {
    sm100::mbar_init(&vbar[warp], 1);
    sm100::fence_barrier_init();
    if (nsm > 0) {
      sm100::mbar_arrive_expect_tx(&vbar[warp], (uint32_t)nsm * seg_bytes);
      for (int i = 0; i < nsm; ++i)
        sm100::bulk_load(&vs[warp][i][0], V + (size_t)(j0 + nreg + i) * p.vocab + tile0, seg_bytes, &vbar[warp]);
    }
  }
  __syncwarp();
  // the selection kernel may launch now (it waits for this grid's records itself)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // t comes from the projection kernel
  for (int e = threadIdx.x; e < BR; e += blockDim.x) st[e] = Elem<T>::scalar(acc_to_t<T>(p.acc, BR, e));
  __syncthreads();
  float acc[NB][PER];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[b][e] = 0.f;
  auto fma_row = [&](const uint4& u, int j) {
#pragma unroll
    for (int b = 0; b < NB; ++b) Elem<T>::axpy16(st[b * r + j], u, acc[b]);
  };
#pragma unroll
  for (int q = 0; q < LSU_BATCH; ++q)
    if (q < nreg) fma_row(raw[q], j0 + q);
  bool ok = true;
  if (nsm > 0) {
    // warp-uniform outcome of the bounded wait
    ok = __all_sync(0xFFFFFFFFu, sm100::mbar_wait(&vbar[warp], 0, WAIT_NS));
    if (!ok) {
      if (lane == 0) {
        atomicOr(p.status, 1 << DH_ERR_TIMEOUT);
        s_fail = 1;
        sm100::mbar_wait(&vbar[warp], 0, WAIT_NS);  // let the copies land before the block moves on
      }
      __syncwarp();
    } else if (valid) {
      for (int i = 0; i < nsm; ++i)
        fma_row(*reinterpret_cast<const uint4*>(&vs[warp][i][lane * 16]), j0 + nreg + i);
    }
  }
  for (int jb = nreg + nsm; jb < rq; jb += LSU_BATCH) {
#pragma unroll
    for (int q = 0; q < LSU_BATCH; ++q)
      raw[q] = (valid && jb + q < rq) ? ld_nc_v4(vp + (size_t)(j0 + jb + q) * p.vocab) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int q = 0; q < LSU_BATCH; ++q)
      if (jb + q < rq) fma_row(raw[q], j0 + jb + q);
  }
  __syncthreads();  // every warp is done with the staged rows: the partial sums reuse the area
  const bool write = s_fail == 0;
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int e = 0; e < PER; ++e) part[warp][b][lane * PER + e] = acc[b][e];
  __syncthreads();
  // warp g folds group g (64 ids): lane i takes ids 2i, 2i+1 of the group
  constexpr int GROUPS = TW / GROUP;
  for (int g = warp; g < GROUPS; g += LSU_WARPS) {
    const int col = g * GROUP + 2 * lane;
    const uint32_t id0 = (uint32_t)(tile0 + col);
    const int gg = (int)(id0 / GROUP);
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int w = 0; w < LSU_WARPS; ++w) {
        s0 += part[w][b][col];
        s1 += part[w][b][col + 1];
      }
      Top2 sm;
      sm.init();
      if ((int)id0 < p.vocab) sm.push(s0, id0);
      if ((int)id0 + 1 < p.vocab) sm.push(s1, id0 + 1);
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) sm.merge_shfl(0xFFFFFFFFu, x);
      if (lane == 0 && gg < p.n_groups && write) {
        p.recs[(size_t)b * p.n_groups + gg] = sm.record((uint32_t)gg * GROUP);
        p.gkeys[(size_t)b * p.n_groups + gg] = sm.i1 == 0xFFFFFFFFu ? 0u : fkey(sm.v1);
      }
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename T, int NB>
cudaError_t launch_tma(const Ctx& c, cudaLaunchConfig_t& cfg, const CUtensorMap& tmV, const ScoresSmall& sp) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_scores_small<T, NB>, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  e = carveout_max_shared(reinterpret_cast<const void*>(k_scores_small<T, NB>), c.device);
  if (e != cudaSuccess) return e;
  return cudaLaunchKernelEx(&cfg, k_scores_small<T, NB>, tmV, sp);
}

template <typename T>
cudaError_t run(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r, int vocab,
                unsigned long long* acc, GroupRec* recs, uint32_t* gkeys, int* status) {
  constexpr int RB = STAGE_BYTES / (SET_TILES * TILE * (int)sizeof(T));
  cudaError_t e = cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;

  ProjSmall pp;
  pp.h = h;
  pp.U = U;
  pp.B = B;
  pp.d = d;
  pp.r = r;
  pp.acc = acc;
  pp.status = status;
  const bool lsu = r % (LSU_WARPS * 16) == 0 && !tuning().scores_tma;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("proj_small", c.stream);
  if (proj_vec_ok(r, (int)sizeof(T))) {
    // one block per SM: room for four blocks of the scores kernel beside it
    const int rpp = PV_THREADS / (r / Elem<T>::PER16);
    cfg.gridDim = dim3((unsigned)max(1, min(c.num_sms, d / rpp)));
    cfg.blockDim = dim3(PV_THREADS);
    cfg.dynamicSmemBytes = (size_t)rpp * B * r * sizeof(float);
    switch (B) {
#define DH_PV_CASE(n)                                                                    \
  case n:                                                                                \
    e = carveout_max_shared(reinterpret_cast<const void*>(k_proj_vec<T, n>), c.device); \
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_proj_vec<T, n>, pp);           \
    break;
      DH_PV_CASE(1) DH_PV_CASE(2) DH_PV_CASE(3) DH_PV_CASE(4) DH_PV_CASE(5) DH_PV_CASE(6) DH_PV_CASE(7) DH_PV_CASE(8)
#undef DH_PV_CASE
      default: e = cudaErrorInvalidValue;
    }
  } else {
    // three blocks per SM: more row slices keep more of U in flight (batch 1, µs per call: 21.5
    // with one block per SM, 19.4 with two, 19.05 with three, 19.2 with four)
    cfg.gridDim = dim3((unsigned)max(1, min(3 * c.num_sms, d / 4)));
    cfg.blockDim = dim3(PJ_THREADS);
    switch (B) {
#define DH_PJ_CASE(n)                                                                      \
  case n:                                                                                  \
    e = carveout_max_shared(reinterpret_cast<const void*>(k_proj_small<T, n>), c.device); \
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_proj_small<T, n>, pp);           \
    break;
      DH_PJ_CASE(1) DH_PJ_CASE(2) DH_PJ_CASE(3) DH_PJ_CASE(4) DH_PJ_CASE(5) DH_PJ_CASE(6) DH_PJ_CASE(7) DH_PJ_CASE(8)
#undef DH_PJ_CASE
      default: e = cudaErrorInvalidValue;
    }
  }
  prof_after(c.stream);
  if (e != cudaSuccess) return note_error(e, "cudaLaunchKernelEx(k_proj_small)");

  ScoresSmall sp;
  sp.acc = acc;
  sp.B = B;
  sp.r = r;
  sp.vocab = vocab;
  sp.n_groups = (vocab + GROUP - 1) / GROUP;
  sp.n_tiles = (vocab + TILE - 1) / TILE;
  sp.recs = recs;
  sp.gkeys = gkeys;
  sp.status = status;
  if (lsu) {
    constexpr int TW = 32 * Elem<T>::PER16;
    cfg.gridDim = dim3((unsigned)((vocab + TW - 1) / TW));
    cfg.blockDim = dim3(LSU_WARPS * 32);
    cfg.dynamicSmemBytes = 0;
    prof_before("scores_lsu", c.stream);
    switch (B) {
#define DH_LSU_CASE(n)                                                                     \
  case n:                                                                                  \
    e = carveout_max_shared(reinterpret_cast<const void*>(k_scores_lsu<T, n>), c.device); \
    if (e == cudaSuccess) e = cudaLaunchKernelEx(&cfg, k_scores_lsu<T, n>, static_cast<const T*>(V), sp); \
    break;
      DH_LSU_CASE(1) DH_LSU_CASE(2) DH_LSU_CASE(3) DH_LSU_CASE(4) DH_LSU_CASE(5) DH_LSU_CASE(6) DH_LSU_CASE(7)
      DH_LSU_CASE(8)
#undef DH_LSU_CASE
      default: e = cudaErrorInvalidValue;
    }
    prof_after(c.stream);
    if (e != cudaSuccess) return note_error(e, "cudaLaunchKernelEx(k_scores_lsu)");
    return note_error(cudaGetLastError(), "small-batch stage 1 launch");
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return note_error(cudaErrorNotSupported, "cuTensorMapEncodeTiled entry point");
  CUtensorMap tmV;
  cuuint64_t dims[2] = {(cuuint64_t)vocab, (cuuint64_t)r};
  cuuint64_t strides[1] = {(cuuint64_t)vocab * sizeof(T)};
  cuuint32_t box[2] = {(cuuint32_t)TILE, (cuuint32_t)RB};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&tmV, sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(V), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(V, small batch)");

  cfg.gridDim = dim3((unsigned)c.num_sms);
  cfg.blockDim = dim3(SB_THREADS);
  cfg.dynamicSmemBytes = STAGE_REGION + 1024;
  prof_before("scores_small", c.stream);
  switch (B) {
#define DH_TMA_CASE(n) case n: e = launch_tma<T, n>(c, cfg, tmV, sp); break;
    DH_TMA_CASE(1) DH_TMA_CASE(2) DH_TMA_CASE(3) DH_TMA_CASE(4) DH_TMA_CASE(5) DH_TMA_CASE(6) DH_TMA_CASE(7)
    DH_TMA_CASE(8)
#undef DH_TMA_CASE
    default: e = cudaErrorInvalidValue;
  }
  prof_after(c.stream);
  if (e != cudaSuccess) return note_error(e, "cudaLaunchKernelEx(k_scores_small)");
  return note_error(cudaGetLastError(), "small-batch stage 1 launch");
}

}  // namespace

bool small_b_supported(int B, int r, int dtype) {
  const int rows = STAGE_BYTES / (SET_TILES * TILE * (dtype == DH_BF16 ? 2 : 4));
  return B >= 1 && B <= MAX_B && B * r <= MAX_BR && r % rows == 0 && r % 2 == 0;
}

cudaError_t launch_small_b(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r,
                           int vocab, int dtype, unsigned long long* acc, GroupRec* recs, uint32_t* gkeys,
                           int* status) {
  if (dtype == DH_BF16) return run<__nv_bfloat16>(c, h, U, V, B, d, r, vocab, acc, recs, gkeys, status);
  return run<float>(c, h, U, V, B, d, r, vocab, acc, recs, gkeys, status);
}

}  // namespace dh
