// Internal declarations shared by the CUDA translation units of libdh (not part of the ABI).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dh.h"

namespace dh {

// Every workspace starts with a 256-byte header whose first word collects device-side status bits
// (1 << dh_status) raised by bounded waits; dh_workspace_status reads and clears it.
constexpr size_t WS_HEADER = 256;
// Fixed-point accumulators of the small-batch projection (8 copies of B * r <= 2048 int64), right
// after the header in the stage-1 workspace.
constexpr size_t WS_FIX_BYTES = 8 * 2048 * 8;

// The small-batch projection's accumulator: ACC_COPIES copies of B*r (at most 2048) signed 64-bit
// fixed-point values with scale 2^32 (projection block c adds into copy c mod ACC_COPIES, which
// keeps the same-address atomics per element low).
constexpr int ACC_COPIES = 8;
constexpr int ACC_MAX_BR = 2048;
static_assert(WS_FIX_BYTES >= (size_t)ACC_COPIES * ACC_MAX_BR * 8, "accumulator fits the fixed region");

// Vocabulary columns summarised together by the stage-1 kernels.  Every group of GROUP consecutive
// ids yields one GroupRec: its two best (score, id) pairs in (score desc, id asc) order and the
// third-best score.  The selection step works from these records; the full score row never
// reaches memory.
constexpr int GROUP = 64;
constexpr uint32_t NO_OFFSET = 0xFFu;

struct __align__(16) GroupRec {
  float m1, m2, m3;  // best, second and third score in the group (-inf when absent)
  uint32_t offs;     // offset in group of the best (bits 0-7) and the second (bits 8-15); 0xFF = absent
};

// ------------------------------------------------------------------ numeric helpers

// Order-preserving map of a float onto uint32 (larger float -> larger key).  -0 is folded onto
// +0 so that keys agree with float equality.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// (a_val, a_id) ranks before (b_val, b_id) in (score desc, id asc) order.
__device__ __forceinline__ bool ranks_before(float av, uint32_t ai, float bv, uint32_t bi) {
  return av > bv || (av == bv && ai < bi);
}

// Running summary of a stream of (score, id) pairs: the top two pairs and the third score.
struct Top2 {
  float v1, v2, v3;
  uint32_t i1, i2;
  __device__ __forceinline__ void init() {
    v1 = v2 = v3 = -INFINITY;
    i1 = i2 = 0xFFFFFFFFu;
  }
  // Pairs must arrive in increasing id order for ties to keep the lower id.  Branch-free, so the
  // lanes of a warp never diverge on their data: the three values by a min/max insertion network,
  // the two ids by two compares.  A NaN x changes nothing: it fails both compares, the inner
  // minima propagate it and the outer maxima then keep the stored values.
  __device__ __forceinline__ static float min_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
  }
  __device__ __forceinline__ void push(float x, uint32_t id) {
    const bool c1 = x > v1, c2 = x > v2;
    v3 = fmaxf(v3, min_nan(v2, x));
    v2 = fmaxf(v2, min_nan(v1, x));
    i2 = c1 ? i1 : (c2 ? id : i2);
    v1 = fmaxf(v1, x);
    i1 = c1 ? id : i1;
  }
  // Merge with another summary of a disjoint set of ids.
  __device__ __forceinline__ void merge(float bv1, uint32_t bi1, float bv2, uint32_t bi2, float bv3) {
    // the four known pairs sorted by (score desc, id asc): a1 >= a2 and b1 >= b2 already hold
    float w1, w2, x3;
    uint32_t j1, j2;
    if (ranks_before(v1, i1, bv1, bi1)) {
      w1 = v1; j1 = i1;
      if (ranks_before(v2, i2, bv1, bi1)) { w2 = v2; j2 = i2; x3 = fmaxf(v3, bv1); }
      else { w2 = bv1; j2 = bi1; x3 = fmaxf(v2, bv2); }
    } else {
      w1 = bv1; j1 = bi1;
      if (ranks_before(v1, i1, bv2, bi2)) { w2 = v1; j2 = i1; x3 = fmaxf(v2, bv2); }
      else { w2 = bv2; j2 = bi2; x3 = fmaxf(v1, bv3); }
    }
    x3 = fmaxf(x3, fmaxf(v3, bv3));
    v1 = w1; i1 = j1; v2 = w2; i2 = j2; v3 = x3;
  }
  __device__ __forceinline__ void merge_shfl(unsigned mask, int lane_xor) {
    float bv1 = __shfl_xor_sync(mask, v1, lane_xor);
    float bv2 = __shfl_xor_sync(mask, v2, lane_xor);
    float bv3 = __shfl_xor_sync(mask, v3, lane_xor);
    uint32_t bi1 = __shfl_xor_sync(mask, i1, lane_xor);
    uint32_t bi2 = __shfl_xor_sync(mask, i2, lane_xor);
    merge(bv1, bi1, bv2, bi2, bv3);
  }
  // Record for the group starting at id g0.
  __device__ __forceinline__ GroupRec record(uint32_t g0) const {
    GroupRec r;
    r.m1 = v1; r.m2 = v2; r.m3 = v3;
    uint32_t o1 = (i1 == 0xFFFFFFFFu) ? NO_OFFSET : (i1 - g0);
    uint32_t o2 = (i2 == 0xFFFFFFFFu) ? NO_OFFSET : (i2 - g0);
    r.offs = o1 | (o2 << 8);
    return r;
  }
};

// fp32 fused multiply-add of two bf16 inputs, taken from the low (or high) halves of 32-bit words.
// The mixed-precision form (bf16 inputs, fp32 addend and result) widens both inputs exactly and
// rounds once, so it returns fmaf(float(a), float(b), c) bit for bit, without separate widening
// instructions.
__device__ __forceinline__ float fma_bf16_lo(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fma_bf16_hi(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\tmov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 %0, ah, bh, %3;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

// Per-dtype element access.  For the dot products:
// - dot16(x, w, acc): acc = fma(x[e], w[e], acc) for e = 0, 1, ... over the elements of two
//   16-byte vectors, one fp32 rounding per step (the order every rescoring kernel shares);
// - Scalar: a scalar operand in the form axpy16 takes (fp32; for bf16 the value's bits in both
//   halves of a word), from scalar(v) of a value v that the dtype represents exactly;
// - axpy16(t, w, acc): acc[e] = fma(t, w[e], acc[e]) for each element of one 16-byte vector.
template <typename T> struct Elem;
template <> struct Elem<float> {
  static constexpr int PER16 = 4;  // elements per 16-byte vector
  using Scalar = float;
  __device__ __forceinline__ static void unpack(const uint4& u, float* out) {
    out[0] = __uint_as_float(u.x); out[1] = __uint_as_float(u.y);
    out[2] = __uint_as_float(u.z); out[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ static float to_f(float x) { return x; }
  __device__ __forceinline__ static float from_f(float x) { return x; }
  __device__ __forceinline__ static float dot16(const uint4& x, const uint4& w, float acc) {
    acc = fmaf(__uint_as_float(x.x), __uint_as_float(w.x), acc);
    acc = fmaf(__uint_as_float(x.y), __uint_as_float(w.y), acc);
    acc = fmaf(__uint_as_float(x.z), __uint_as_float(w.z), acc);
    return fmaf(__uint_as_float(x.w), __uint_as_float(w.w), acc);
  }
  __device__ __forceinline__ static Scalar scalar(float v) { return v; }
  __device__ __forceinline__ static Scalar scalar_of(float x) { return x; }
  __device__ __forceinline__ static void axpy16(Scalar t, const uint4& w, float* acc) {
    acc[0] = fmaf(t, __uint_as_float(w.x), acc[0]);
    acc[1] = fmaf(t, __uint_as_float(w.y), acc[1]);
    acc[2] = fmaf(t, __uint_as_float(w.z), acc[2]);
    acc[3] = fmaf(t, __uint_as_float(w.w), acc[3]);
  }
};
template <> struct Elem<__nv_bfloat16> {
  static constexpr int PER16 = 8;
  using Scalar = uint32_t;
  __device__ __forceinline__ static void unpack(const uint4& u, float* out) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      out[2 * q] = __uint_as_float(w[q] << 16);
      out[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ __forceinline__ static __nv_bfloat16 from_f(float x) { return __float2bfloat16_rn(x); }
  __device__ __forceinline__ static float dot16(const uint4& x, const uint4& w, float acc) {
    acc = fma_bf16_lo(x.x, w.x, acc);
    acc = fma_bf16_hi(x.x, w.x, acc);
    acc = fma_bf16_lo(x.y, w.y, acc);
    acc = fma_bf16_hi(x.y, w.y, acc);
    acc = fma_bf16_lo(x.z, w.z, acc);
    acc = fma_bf16_hi(x.z, w.z, acc);
    acc = fma_bf16_lo(x.w, w.w, acc);
    return fma_bf16_hi(x.w, w.w, acc);
  }
  // v must be a bf16 value (its low 16 bits are zero)
  __device__ __forceinline__ static Scalar scalar(float v) {
    const uint32_t u = __float_as_uint(v) >> 16;
    return u | (u << 16);
  }
  __device__ __forceinline__ static Scalar scalar_of(__nv_bfloat16 x) {
    const uint32_t u = __bfloat16_as_ushort(x);
    return u | (u << 16);
  }
  __device__ __forceinline__ static void axpy16(Scalar t, const uint4& w, float* acc) {
    acc[0] = fma_bf16_lo(t, w.x, acc[0]);
    acc[1] = fma_bf16_hi(t, w.x, acc[1]);
    acc[2] = fma_bf16_lo(t, w.y, acc[2]);
    acc[3] = fma_bf16_hi(t, w.y, acc[3]);
    acc[4] = fma_bf16_lo(t, w.z, acc[4]);
    acc[5] = fma_bf16_hi(t, w.z, acc[5]);
    acc[6] = fma_bf16_lo(t, w.w, acc[6]);
    acc[7] = fma_bf16_hi(t, w.w, acc[7]);
  }
};

// Softmax over z[0..K) by one warp (lane i takes elements i, i + 32, ...; max and sum by xor
// shuffles, so every lane gets the same values): out[k] = exp(z[k] - max) / sum.  For the small
// K of the cluster kernels this avoids a block barrier per reduction.
// Every kernel that computes probabilities uses this one order, so that all stage-2 paths agree
// bit for bit.  With L2 set, z is global memory written by other blocks and is read through L2.
template <bool L2>
__device__ __forceinline__ void warp_softmax_impl(const float* z, int K, float* out) {
  const int lane = threadIdx.x & 31;
  auto ld = [&](int i) { return L2 ? __ldcg(z + i) : z[i]; };
  float m = -INFINITY;
  for (int i = lane; i < K; i += 32) m = fmaxf(m, ld(i));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  float ssum = 0.f;
  for (int i = lane; i < K; i += 32) ssum += expf(ld(i) - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, o);
  const float inv = 1.f / ssum;
  for (int i = lane; i < K; i += 32) out[i] = expf(ld(i) - m) * inv;
}
__device__ __forceinline__ void warp_softmax(const float* z, int K, float* out) { warp_softmax_impl<false>(z, K, out); }
__device__ __forceinline__ void warp_softmax_l2(const float* z, int K, float* out) { warp_softmax_impl<true>(z, K, out); }

// Element e of t from the fixed-point accumulator copies (copy q at acc + q*BR), rounded to the
// activation dtype.  The integer sum is exact and order independent, so every reader derives the
// same t.  Read through L2 (the copies were written by atomics).
template <typename T>
__device__ __forceinline__ float acc_to_t(const unsigned long long* acc, int BR, int e) {
  long long fx = 0;
#pragma unroll
  for (int q = 0; q < ACC_COPIES; ++q) fx += (long long)__ldcg(acc + (size_t)q * BR + e);
  return Elem<T>::to_f(Elem<T>::from_f((float)((double)fx * (1.0 / 4294967296.0))));
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// ------------------------------------------------------------------ host side

// Test and tuning switches (tuning.cu): read from the environment once per process, changed only by
// dh_set_tuning.  They select kernels; results do not depend on them.
struct Tuning {
  enum Path { PATH_AUTO, PATH_GEMV, PATH_MMA, PATH_FUSED };
  enum Rescore { RESCORE_AUTO, RESCORE_DIRECT, RESCORE_RING, RESCORE_TICKET, RESCORE_SWEEP, RESCORE_BUCKET };
  Path force_path = PATH_AUTO;      // stage-1 path, when the forced one supports the shape
  bool head_split = false;          // dh_draft_head: the two calls' kernels, not the cluster head
  bool head_cluster = false;        // dh_draft_head: the cluster head wherever it fits, whatever K
  int head_ctas_max = 16;           // largest cluster of the fused head (16, 8 or 4)
  Rescore rescore = RESCORE_AUTO;   // stage-2 kernel choice
  bool scores_tma = false;          // small-batch scores: the TMA variant for every rank
  bool head_select_radix = false;   // fused head: the cooperative radix selection, not the fast one
};
const Tuning& tuning();

struct Ctx {
  int device;
  int num_sms;
  long long l2_bytes;
  cudaStream_t stream;
};

bool get_ctx(void* stream, Ctx* ctx);

// Kernel-launch bookkeeping for dh_prof_*: call before and after a launch.
void prof_before(const char* name, cudaStream_t s);
void prof_after(cudaStream_t s);

// Launchers (one per translation unit).  All return cudaError_t of the launch.
cudaError_t launch_proj(const Ctx& c, const void* h, const void* U, int B, int d, int r, int dtype,
                        float* partial, int nsplit, void* t_out);
int proj_splits(const Ctx& c, int B, int d, int r);

bool mma_path_supported(int B, int r, int dtype);
bool small_b_supported(int B, int r, int dtype);
bool proj_mma_supported(int B, int d, int r, int dtype);
int proj_mma_splits(int B, int d, int r, int num_sms);
cudaError_t launch_proj_mma(const Ctx& c, const void* h, const void* U, int B, int d, int r, float* partial,
                            int max_splits, void* t, int* status);
// Small-batch stage 1: the projection leaves t in the fixed-point accumulators `acc` (ACC_COPIES
// copies of B*r values, zero between calls); the scores kernel and the selection read t from there
// and the selection clears them.
// gkeys [B][n_groups]: each group's best score as an order-preserving key (0: empty group).
cudaError_t launch_small_b(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r,
                           int vocab, int dtype, unsigned long long* acc, GroupRec* recs, uint32_t* gkeys,
                           int* status);
// gkeys (may be null): as for the small-batch path, each group's best key (0: empty group).
cudaError_t launch_lowrank_mma(const Ctx& c, const void* t, const void* V, int B, int r, int vocab,
                               GroupRec* recs, uint32_t* gkeys, int* status);

cudaError_t launch_scores_summary(const Ctx& c, const void* t, const void* V, int B, int r, int vocab,
                                  int dtype, GroupRec* recs);

// t: [B][r] in the activation dtype, or nullptr with acc set (small-batch path: t is derived from
// the projection's fixed-point accumulators, which the selection then clears).
cudaError_t launch_select(const Ctx& c, const GroupRec* recs, const void* t, unsigned long long* acc,
                          const void* V, int B, int r, int vocab, int K, int dtype, int32_t* idx_out,
                          float* score_out, uint32_t* tickets = nullptr);

// Small batches: selection and rescoring in one thread-block cluster per row (head_cl.cu).
bool head_cluster_supported(int B, int d, int vocab, int K, int dtype);
// Cluster size (16, 8 or 4 CTAs) with which the fused head runs all B rows in one wave on this
// device, or 0 when it cannot (or when the two kernels are faster for B rows of K candidates).
int head_cluster_ctas(const Ctx& c, int B, int K, int d, int vocab, int dtype);
// Fused selection and rescoring with clusters of `ctas` CTAs: t from the small-batch accumulators
// (acc) or, with acc null, from t [B][r] in the activation dtype.
// gkeys: the groups' best keys from the small-batch scores kernel (the fast selection), or null
// (the cooperative radix selection).
cudaError_t launch_head_cluster(const Ctx& c, int ctas, const GroupRec* recs, const uint32_t* gkeys,
                                unsigned long long* acc, const void* t, const void* V, const void* h, const void* W,
                                int B, int d, int r, int vocab, int K, int dtype, int32_t* idx_out, float* score_out,
                                float* logits, float* probs, int* status);

cudaError_t launch_expand(const Ctx& c, const float* probs, const int32_t* idx, const float* parent_prob, int B,
                          int K, int w, float min_benefit, int32_t* child_token, float* child_prob,
                          int32_t* n_keep);

bool rescore_supported(int d);
// Large batches: the vocabulary-sweep rescoring (W rows shared by rows of the batch read once).
bool rescore_sweep_supported(int B, int K, int d, int vocab, int dtype, int num_sms);
cudaError_t launch_rescore_sweep(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                 int vocab, int K, int dtype, float* logits, float* probs, int* status);
bool rescore_ring_used(int B, int K, int d, int dtype);
bool rescore_ring_fits(int K, int d, int dtype);
cudaError_t launch_rescore_ring(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d,
                                int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets,
                                int* status, bool force_buckets = false);
cudaError_t launch_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B,
                           int d, int vocab, int K, int dtype, float* logits, float* probs, uint32_t* tickets);

// Vocabulary-sharded head (shard.cu).
cudaError_t launch_add_offset(const Ctx& c, int32_t* idx, long long n, int offset);
cudaError_t launch_merge_topk(const Ctx& c, const int32_t* idx_parts, const float* score_parts, int P, int B, int K,
                              int32_t* idx_out, float* score_out);
cudaError_t launch_localize(const Ctx& c, const int32_t* idx, long long n, int offset, int vocab_shard,
                            int32_t* local);
cudaError_t launch_shard_stats(const Ctx& c, const int32_t* local, int B, int K, float* logits, float* stats);
cudaError_t launch_combine_softmax(const Ctx& c, const float* logits_parts, const float* stats_parts, int P, int B,
                                   int K, float* logits_out, float* probs_out);

// Sizing the next draft level (sizing.cu).
size_t size_level_smem(int F, int Wc, int wmax);
cudaError_t launch_size_level(const Ctx& c, const float* child_prob, const int32_t* child_token,
                              const int32_t* n_valid, int R, int F, int Wc, const float* cost,
                              const int32_t* bin_batch, int n_bins, int wmax, int batch, float theta,
                              int32_t* width, int32_t* sel_parent, int32_t* sel_token, float* sel_prob);

// Chain verification at positive temperature (verify.cu).  seg_stats: B*(L+1)*verify_segments(vocab,
// dtype) float2.
int verify_segments(int vocab, int dtype);
cudaError_t launch_verify(const Ctx& c, const void* logits, int dtype, int B, int L, int vocab, int K,
                          const int32_t* cand_idx, const float* cand_prob, const int32_t* draft, const float* u_accept,
                          const float* u_sample, float temperature, int32_t* n_accept, int32_t* token,
                          float2* seg_stats);

cudaError_t launch_tree(const Ctx& c, const void* logits, const int32_t* parent, const int32_t* token,
                        int B, int N, int vocab, int dtype, int32_t* argmax_ws, int32_t* argmax_out,
                        int32_t* path, int32_t* len, int32_t* bonus, int32_t* err);

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Records the failing CUDA call of the current thread for dh_last_error(); returns e.
cudaError_t note_error(cudaError_t e, const char* where);

// Sets a kernel's preferred shared-memory carveout to the largest, once per (kernel, device).
// Blocks of kernels with different carveouts cannot share an SM (the SM is reconfigured only when
// empty), so the kernels of one pipeline that are meant to overlap through programmatic dependent
// launch all take the same one.
cudaError_t carveout_max_shared(const void* kernel, int device);

// Raises a kernel's dynamic shared memory limit to the device maximum minus its static shared
// memory, once per device (a plain attribute call, so it is also safe during stream capture).
template <class Kernel>
cudaError_t allow_max_smem(Kernel kernel, int device, unsigned long long* done_mask) {
  if (device < 64 && ((*done_mask >> device) & 1ull)) return cudaSuccess;
  int maxopt = 0;
  cudaError_t e = cudaDeviceGetAttribute(&maxopt, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  if (e != cudaSuccess) return note_error(e, "cudaDeviceGetAttribute(MaxSharedMemoryPerBlockOptin)");
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kernel);
  if (e != cudaSuccess) return note_error(e, "cudaFuncGetAttributes");
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           maxopt - (int)fa.sharedSizeBytes);
  if (e != cudaSuccess) return note_error(e, "cudaFuncSetAttribute(MaxDynamicSharedMemorySize)");
  if (device < 64) *done_mask |= 1ull << device;
  return e;
}

// Dynamic shared memory available to `kernel` on `device` (opt-in maximum minus static usage).
template <class Kernel>
int max_dynamic_smem(Kernel kernel, int device) {
  int maxopt = 0;
  cudaFuncAttributes fa;
  if (cudaDeviceGetAttribute(&maxopt, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) return 0;
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return 0;
  return maxopt - (int)fa.sharedSizeBytes;
}

}  // namespace dh
