// Stage 1b (tensor-core path, bf16, B >= a few rows): S = T V on tcgen05 with the accumulator in
// TMEM and a fused epilogue that folds every group of 64 vocabulary ids into a GroupRec, so the
// B x vocab score matrix never reaches memory.
//
// EAGLE-4 summary page, section "Retrieve vocabulary candidates cheaply, then score them exactly":
// the low-rank head scores the whole vocabulary to retrieve candidates.  At high load the product
// T [B x r] V [r x vocab] is a dense contraction (B*r flop per V byte), so it runs on the tensor
// cores; the selection that follows is shared with the CUDA-core path.
//
// One CTA per SM owns a 128-row tile of T (kept resident in shared memory, r/64 TMA boxes of
// 128 x 64 bf16 with 128-byte swizzle) and a contiguous range of 256-wide vocabulary tiles.
// Warp roles:
//   warp 0     TMA producer: streams V in stages of 64 (K) x 256 (N) bf16 (four 64 x 64 boxes).
//   warp 1     TMEM allocator and MMA issuer: per vocabulary tile, r/16 tcgen05.mma
//              (M=128, N=256, K=16, A K-major, B N-major) into one of two TMEM accumulators.
//   warps 2-9  epilogue: tcgen05.ld 32x32b (thread = row); two warps per TMEM lane quarter, each
//              owning two of the tile's four 64-id groups; branch-free per-group top-two + third
//              score; one 16-byte record store per (row, group).
// With at most 64 rows of T (one row tile), the A tile holds 2 or 4 copies of T's rows, so the
// MMA computes every score 2 or 4 times over the lane quarters.  A warp can read only its own lane
// quarter of TMEM, so with one copy all of a small batch's folding would fall on the two warps of
// one quarter; with copies, each copy folds a different share of the tile's groups and the two
// warps of a quarter take alternate tiles.  The tensor cores have time to spare at these sizes;
// the epilogue does not.
// Every mbarrier wait gives up after two seconds and raises DH_ERR_TIMEOUT in the status word;
// the CTA then drains its outstanding copies and MMAs (again with bounded waits) and frees TMEM.
#include "dh_internal.cuh"
#include "sm100.cuh"

namespace dh {
namespace {

using namespace sm100;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int A_CHUNK_BYTES = BM * BK * 2;  // 16 KB: 128 rows x 128 bytes
constexpr int B_BOX_BYTES = BK * 64 * 2;    // 8 KB: 64 K-rows x 64 ids
constexpr int B_STAGE_BYTES = 4 * B_BOX_BYTES;
constexpr int THREADS = 320;         // producer, MMA issuer, 8 epilogue warps
constexpr int EPI_WARPS = 8;
constexpr uint32_t TMEM_COLS = 512;  // two 128 x 256 fp32 accumulators
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int MAX_STAGES = 8;
// V stages issued before the wait for the projection: the copies of all the ring's stages from
// every CTA at once kept the producer from reaching the wait (and T's load) for up to 3.5 µs;
// two stages measured best (8 rows: 25.6 against 26.5 µs per call; 64 rows: 56.6 against 57.2).
constexpr int PRE_STAGES = 2;

struct MmaParams {
  int B, r, vocab, n_groups, n_tiles, n_split, stages;
  int rep;  // copies of T's rows in the 128-row A tile (1, 2 or 4; see the epilogue)
  GroupRec* recs;
  uint32_t* gkeys;  // [B][n_groups] each group's best key for the fused head's fast selection, or null
  int* status;
};

__device__ __forceinline__ void raise_timeout(volatile int* s_abort, int* status) {
  *s_abort = 1;
  atomicOr(status, 1 << DH_ERR_TIMEOUT);
}

__global__ void __launch_bounds__(THREADS, 1)
    k_lowrank_mma(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, MmaParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[2 + 2 * MAX_STAGES + 4];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_abort;

  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int nkc = p.r / BK;
  unsigned char* sA = base;
  unsigned char* sB = sA + nkc * A_CHUNK_BYTES;
  uint64_t* a_full = &bars[0];
  uint64_t* drain = &bars[1];
  uint64_t* b_full = &bars[2];
  uint64_t* b_empty = &bars[2 + MAX_STAGES];
  uint64_t* acc_full = &bars[2 + 2 * MAX_STAGES];
  uint64_t* acc_empty = &bars[2 + 2 * MAX_STAGES + 2];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m = blockIdx.x / p.n_split, part = blockIdx.x % p.n_split;
  const int nt0 = (int)((long long)p.n_tiles * part / p.n_split);
  const int nt1 = (int)((long long)p.n_tiles * (part + 1) / p.n_split);
  const int ntiles = nt1 - nt0;
  const int stages = p.stages;

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(a_full, 1);
    mbar_init(drain, 1);
    for (int s = 0; s < stages; ++s) {
      mbar_init(&b_full[s], 1);
      mbar_init(&b_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], p.rep == 1 ? EPI_WARPS : EPI_WARPS / 2);  // the warps that take the tile
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // the selection kernel may launch now; it waits (griddepcontrol.wait) for this grid's records
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      // V does not depend on the projection: its first PRE_STAGES stages are issued before waiting
      // for the previous kernel (programmatic dependent launch), T (the A operand) after it.
      bool a_issued = false;
      auto issue_a = [&]() {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        mbar_arrive_expect_tx(a_full, (uint32_t)(nkc * A_CHUNK_BYTES));
        // rep copies of T's first BM / rep rows, one per BM / rep smem rows (128 bytes per row)
        const int rows_rep = BM / p.rep;
        for (int kc = 0; kc < nkc; ++kc)
          for (int q = 0; q < p.rep; ++q)
            tma_load_2d(sA + kc * A_CHUNK_BYTES + q * rows_rep * 128, &tmA, kc * BK, m * BM, a_full);
        a_issued = true;
      };
      uint32_t issued_parity = 0;  // bit s: parity of the last load issued into stage s
      uint32_t issued_mask = 0;
      int s = 0, n_issued = 0;
      uint32_t ph = 0;
      for (int t = 0; t < ntiles && !s_abort; ++t) {
        const int n0 = (nt0 + t) * BN;
        for (int kc = 0; kc < nkc; ++kc) {
          if (!a_issued && n_issued == min(stages, PRE_STAGES)) issue_a();
          ++n_issued;
          if (!mbar_wait(&b_empty[s], ph ^ 1u, WAIT_NS)) { raise_timeout(&s_abort, p.status); break; }
          mbar_arrive_expect_tx(&b_full[s], B_STAGE_BYTES);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            tma_load_2d(sB + s * B_STAGE_BYTES + q * B_BOX_BYTES, &tmB, n0 + q * 64, kc * BK, &b_full[s]);
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
      }
      if (!a_issued) issue_a();
      // every copy this CTA issued must land before the CTA can exit
      mbar_wait(a_full, 0, WAIT_NS);
      for (int q = 0; q < stages; ++q)
        if ((issued_mask >> q) & 1u) mbar_wait(&b_full[q], (issued_parity >> q) & 1u, WAIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, 0, 1);
      bool ok = mbar_wait(a_full, 0, WAIT_NS);
      if (!ok) raise_timeout(&s_abort, p.status);
      tc_fence_after();
      int s = 0;
      uint32_t ph = 0;
      for (int t = 0; t < ntiles && ok && !s_abort; ++t) {
        const int buf = t & 1;
        const uint32_t acc_ph = (uint32_t)(t >> 1) & 1u;
        if (!mbar_wait(&acc_empty[buf], acc_ph ^ 1u, WAIT_NS)) { raise_timeout(&s_abort, p.status); break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(buf * BN);
        for (int kc = 0; kc < nkc; ++kc) {
          if (!mbar_wait(&b_full[s], ph, WAIT_NS)) { raise_timeout(&s_abort, p.status); ok = false; break; }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + kc * A_CHUNK_BYTES);
          const uint32_t b_base = smem_u32(sB + s * B_STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // A: K-major, 128-byte rows, 8-row groups 1 KB apart; +32 bytes per K step of 16.
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
            // B: N-major, 64-id (128-byte) atoms 8 KB apart, 8-row K groups 1 KB apart.
            const uint64_t bd = smem_desc_sw128(b_base + kk * 2048, B_BOX_BYTES, 1024);
            mma_f16(d_tmem, ad, bd, idesc, (kc | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&b_empty[s]);
          if (++s == stages) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&acc_full[buf]);
      }
      // all MMAs issued by this thread complete before TMEM is released
      mma_commit(drain);
      mbar_wait(drain, 0, WAIT_NS);
    }
  } else {
    // -------------------------------------------------------------- epilogue (warps 2-9)
    const int q = warp & 3;             // TMEM lanes [32q, 32q + 32) are accessible to this warp
    const int half = (warp - 2) >> 2;
    // rep = 1: every tile, groups 2*half and 2*half + 1.  rep > 1 (one row tile holding rep copies
    // of T's rows): the lane quarters of copy c take groups [c*4/rep, (c+1)*4/rep) and the two
    // halves take alternate tiles, so each warp folds 4/rep times fewer scores per tile.
    const int rows_rep = BM / p.rep;
    const int copy = (q * 32) / rows_rep;
    const int row = m * BM + (q * 32) % rows_rep + lane;
    const int n_g = p.rep == 1 ? 2 : 4 / p.rep;
    const int g_first = p.rep == 1 ? 2 * half : copy * n_g;
    const int t_first = p.rep == 1 ? 0 : half, t_step = p.rep == 1 ? 1 : 2;
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    for (int t = t_first; t < ntiles; t += t_step) {
      const int buf = t & 1;
      const uint32_t acc_ph = (uint32_t)(t >> 1) & 1u;
      // warp-uniform outcome: the TMEM loads below are .sync.aligned and need the whole warp
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&acc_full[buf], acc_ph, WAIT_NS))) {
        raise_timeout(&s_abort, p.status);
        break;
      }
      tc_fence_after();
      const int n0 = (nt0 + t) * BN;
#pragma unroll 1
      for (int gg = 0; gg < n_g; ++gg) {
        const int g = g_first + gg;
        const int gc0 = n0 + g * GROUP;
        Top2 sm;
        sm.init();
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          float v[32];
          tmem_ld_32x32b_x32(lane_addr + (uint32_t)(buf * BN + g * GROUP + h2 * 32), v);
          if (gc0 + GROUP <= p.vocab) {
#pragma unroll
            for (int i = 0; i < 32; ++i) sm.push(v[i], (uint32_t)(gc0 + h2 * 32 + i));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (gc0 + h2 * 32 + i < p.vocab) sm.push(v[i], (uint32_t)(gc0 + h2 * 32 + i));
          }
        }
        if (row < p.B && gc0 < p.vocab) {
          p.recs[(size_t)row * p.n_groups + gc0 / GROUP] = sm.record((uint32_t)gc0);
          if (p.gkeys) p.gkeys[(size_t)row * p.n_groups + gc0 / GROUP] = sm.i1 == 0xFFFFFFFFu ? 0u : fkey(sm.v1);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// ------------------------------------------------------------------------------------------------
// Stage 1a on the tensor cores (bf16, larger batches): partial[s] = h[:, K-slice s] U[K-slice s, :]
// for a split-K grid of (row tile, column tile, slice) blocks; k_proj_reduce_mma then sums the
// slices in a fixed order and rounds t to bf16.  A = h (K-major, streamed), B = U (N-major).
// Warp roles as in k_lowrank_mma; one accumulator of 128 x BN fp32 in TMEM per block.

struct ProjParams {
  int B, d, r, BN, n_ntiles, splits;
  float* partial;  // [splits][B][r]
  int* status;
};

__global__ void __launch_bounds__(THREADS, 1)
    k_proj_mma(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmU, ProjParams p) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bars[2 * MAX_STAGES + 2];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_abort;
  unsigned char* base = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                         ~static_cast<uintptr_t>(1023));
  const int nb = p.BN / 64;                        // 64-id boxes of U per stage
  const int stage_bytes = A_CHUNK_BYTES + nb * B_BOX_BYTES;
  uint64_t* full = &bars[0];
  uint64_t* empty = &bars[MAX_STAGES];
  uint64_t* acc_full = &bars[2 * MAX_STAGES];
  uint64_t* drain = &bars[2 * MAX_STAGES + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_per_split = gridDim.x / p.splits;
  const int split = blockIdx.x / tiles_per_split;
  const int tile = blockIdx.x % tiles_per_split;
  const int m = tile / p.n_ntiles, n = tile % p.n_ntiles;
  const int nkc_all = p.d / BK;
  const int kc0 = (int)((long long)nkc_all * split / p.splits);
  const int kc1 = (int)((long long)nkc_all * (split + 1) / p.splits);
  const int nkc = kc1 - kc0;
  const int stages = min(MAX_STAGES, (int)(200 * 1024 / stage_bytes));
  uint32_t tmem_cols = 32;  // TMEM allocations are powers of two >= 32 columns
  while (tmem_cols < (uint32_t)p.BN) tmem_cols <<= 1;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_slot, tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  // launched with programmatic dependent launch: h may come from the kernel before this one, which
  // may also still read the workspace, so nothing is loaded or stored before the wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // the reduce kernel may launch now; it waits (griddepcontrol.wait) for the partial sums
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmH);
      prefetch_tmap(&tmU);
      uint32_t issued_parity = 0, issued_mask = 0, ph = 0;
      int s = 0;
      for (int kc = kc0; kc < kc1 && !s_abort; ++kc) {
        if (!mbar_wait(&empty[s], ph ^ 1u, WAIT_NS)) { raise_timeout(&s_abort, p.status); break; }
        unsigned char* st = base + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
        tma_load_2d(st, &tmH, kc * BK, m * BM, &full[s]);
        for (int q = 0; q < nb; ++q)
          tma_load_2d(st + A_CHUNK_BYTES + q * B_BOX_BYTES, &tmU, n * p.BN + q * 64, kc * BK, &full[s]);
        issued_mask |= 1u << s;
        issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
      for (int q = 0; q < stages; ++q)
        if ((issued_mask >> q) & 1u) mbar_wait(&full[q], (issued_parity >> q) & 1u, WAIT_NS);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, p.BN, 0, 1);
      int s = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int kc = 0; kc < nkc && !s_abort; ++kc) {
        if (!mbar_wait(&full[s], ph, WAIT_NS)) { raise_timeout(&s_abort, p.status); ok = false; break; }
        tc_fence_after();
        const uint32_t a_base = smem_u32(base + (size_t)s * stage_bytes);
        const uint32_t b_base = a_base + A_CHUNK_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = smem_desc_sw128(a_base + kk * 32, 16, 1024);
          const uint64_t bd = smem_desc_sw128(b_base + kk * 2048, B_BOX_BYTES, 1024);
          mma_f16(tmem, ad, bd, idesc, (kc | kk) != 0 ? 1u : 0u);
        }
        mma_commit(&empty[s]);
        if (++s == stages) { s = 0; ph ^= 1u; }
      }
      if (ok) mma_commit(acc_full);
      mma_commit(drain);
      mbar_wait(drain, 0, WAIT_NS);
    }
  } else if (warp < 6) {  // warps 2-5 cover the four TMEM lane quarters
    const int q = warp & 3;
    const int row = m * BM + q * 32 + lane;
    if (__all_sync(0xFFFFFFFFu, mbar_wait(acc_full, 0, WAIT_NS))) {
      tc_fence_after();
      const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
      float* out = p.partial + ((size_t)split * p.B + row) * p.r + (size_t)n * p.BN;
      for (int c0 = 0; c0 < p.BN; c0 += 32) {
        float v[32];
        tmem_ld_32x32b_x32(lane_addr + (uint32_t)c0, v);
        if (row < p.B) {
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(out + c0 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
        }
      }
    } else {
      raise_timeout(&s_abort, p.status);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// t[e] = bf16(sum over s of partial[s][e]), slices in ascending order (deterministic).  Each
// thread owns four consecutive outputs (B*r is a multiple of 64) and keeps 8 slices in flight.
// Launched with programmatic dependent launch.  The scores kernel (which sets up, prefetches V and
// then waits for t itself) is released before the wait for the projection's partial sums when
// early is set, else after it.  Early release hides the scores kernel's set-up behind a long
// projection (r = 256, B = 64: 58.1 against 58.9 µs per step) but lets its V prefetch compete with
// a short one (r = 128, B = 8: 32.4 against 31.9 µs).
__global__ void k_proj_reduce_mma(const float* __restrict__ partial, int BR, int splits, int early,
                                  __nv_bfloat16* __restrict__ t) {
  if (early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!early) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int e = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (e >= BR) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < splits; s0 += 8) {
    float4 v[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (s0 + q < splits) v[q] = __ldcg(reinterpret_cast<const float4*>(partial + (size_t)(s0 + q) * BR + e));
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      if (s0 + q < splits) {
        acc.x += v[q].x;
        acc.y += v[q].y;
        acc.z += v[q].z;
        acc.w += v[q].w;
      }
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  *reinterpret_cast<__nv_bfloat162*>(t + e) = lo;
  *reinterpret_cast<__nv_bfloat162*>(t + e + 2) = hi;
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

// 2-D bf16 tensor map over a row-major [rows x cols] matrix, box [box_rows x box_cols], 128B swizzle.
bool make_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mma_path_supported(int B, int r, int dtype) {
  return dtype == DH_BF16 && B >= 1 && r % BK == 0 && r >= BK && r <= 512;
}

bool proj_mma_supported(int B, int d, int r, int dtype) {
  return mma_path_supported(B, r, dtype) && d % BK == 0 && (r <= 256 || r % 256 == 0);
}

// Split-K slices of the tensor-core projection: enough blocks to cover the SMs but at least four
// 64-wide K chunks per slice (the reduction reads every slice).  num_sms = 256 bounds the
// workspace independently of the device.
int proj_mma_splits(int B, int d, int r, int num_sms) {
  const int m_tiles = (B + BM - 1) / BM;
  const int n_tiles = (r + 255) / 256;
  return max(1, min(d / (4 * BK), num_sms / (m_tiles * n_tiles)));
}

cudaError_t launch_proj_mma(const Ctx& c, const void* h, const void* U, int B, int d, int r, float* partial,
                            int max_splits, void* t, int* status) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_proj_mma, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  ProjParams p;
  p.B = B;
  p.d = d;
  p.r = r;
  p.BN = r <= 256 ? r : 256;
  p.n_ntiles = r / p.BN;
  p.splits = min(max_splits, proj_mma_splits(B, d, r, c.num_sms));
  p.partial = partial;
  p.status = status;
  const int stage_bytes = A_CHUNK_BYTES + (p.BN / 64) * B_BOX_BYTES;
  const int stages = min(MAX_STAGES, 200 * 1024 / stage_bytes);
  const size_t smem = 1024 + (size_t)stages * stage_bytes;
  CUtensorMap tmH, tmU;
  if (!make_map(&tmH, h, (uint64_t)d, (uint64_t)B, BK, BM)) return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(h)");
  if (!make_map(&tmU, U, (uint64_t)r, (uint64_t)d, 64, BK)) return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(U)");
  const int m_tiles = (B + BM - 1) / BM;
  const int grid = p.splits * m_tiles * p.n_ntiles;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  {  // programmatic dependent launch: the set-up overlaps the previous kernel's tail
    cudaLaunchConfig_t pc = {};
    pc.gridDim = dim3((unsigned)grid);
    pc.blockDim = dim3(THREADS);
    pc.dynamicSmemBytes = smem;
    pc.stream = c.stream;
    pc.attrs = attr;
    pc.numAttrs = 1;
    prof_before("proj_mma", c.stream);
    e = cudaLaunchKernelEx(&pc, k_proj_mma, tmH, tmU, p);
    prof_after(c.stream);
  }
  if (e != cudaSuccess) return note_error(e, "launch k_proj_mma");
  const int BR = B * r;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((BR / 4 + 255) / 256));
  cfg.blockDim = dim3(256);
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("proj_reduce_mma", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_proj_reduce_mma, static_cast<const float*>(partial), BR, p.splits, r >= 256 ? 1 : 0,
                         static_cast<__nv_bfloat16*>(t));
  prof_after(c.stream);
  if (e != cudaSuccess) return note_error(e, "launch k_proj_reduce_mma");
  return note_error(cudaGetLastError(), "launch k_proj_reduce_mma");
}

cudaError_t launch_lowrank_mma(const Ctx& c, const void* t, const void* V, int B, int r, int vocab,
                               GroupRec* recs, uint32_t* gkeys, int* status) {
  static unsigned long long smem_done = 0;
  cudaError_t e = allow_max_smem(k_lowrank_mma, c.device, &smem_done);
  if (e != cudaSuccess) return e;
  const int nkc = r / BK;
  // dynamic: 1 KB alignment slack + resident A + B stages
  const int avail = max_dynamic_smem(k_lowrank_mma, c.device) - 1024 - nkc * A_CHUNK_BYTES;
  const int stages = min(MAX_STAGES, avail / B_STAGE_BYTES);
  if (stages < 2) return note_error(cudaErrorInvalidConfiguration, "lowrank_mma: shared memory for 2 stages");
  const size_t smem = 1024 + (size_t)nkc * A_CHUNK_BYTES + (size_t)stages * B_STAGE_BYTES;

  const int num_m = (B + BM - 1) / BM;
  // one row tile: replicate T's rows over the lane quarters (see the epilogue)
  const int rep = num_m == 1 && B <= BM / 4 ? 4 : (num_m == 1 && B <= BM / 2 ? 2 : 1);
  CUtensorMap tmA, tmB;
  if (!make_map(&tmA, t, (uint64_t)r, (uint64_t)B, BK, BM / rep))
    return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(T)");
  if (!make_map(&tmB, V, (uint64_t)vocab, (uint64_t)r, 64, BK))
    return note_error(cudaErrorInvalidValue, "cuTensorMapEncodeTiled(V)");

  MmaParams p;
  p.B = B;
  p.r = r;
  p.vocab = vocab;
  p.n_groups = (vocab + GROUP - 1) / GROUP;
  p.n_tiles = (vocab + BN - 1) / BN;
  p.n_split = max(1, min(p.n_tiles, c.num_sms / num_m));
  p.rep = rep;
  p.stages = stages;
  p.recs = recs;
  p.gkeys = gkeys;
  p.status = status;
  // programmatic dependent launch: set-up and the first V stages overlap the projection's tail
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(num_m * p.n_split));
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before("lowrank_mma", c.stream);
  e = cudaLaunchKernelEx(&cfg, k_lowrank_mma, tmA, tmB, p);
  prof_after(c.stream);
  if (e != cudaSuccess) return note_error(e, "launch k_lowrank_mma");
  return note_error(cudaGetLastError(), "launch k_lowrank_mma");
}

}  // namespace dh
