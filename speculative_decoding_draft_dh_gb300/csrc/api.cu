// C ABI of libdh: argument validation, workspace layout and kernel sequencing (see include/dh.h).
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "dh_internal.cuh"

namespace dh {

namespace {

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
long long g_l2[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
bool valid_dtype(int dt) { return dt == DH_F32 || dt == DH_BF16; }
int elem_bytes(int dt) { return dt == DH_BF16 ? 2 : 4; }
// row length in elements whose byte size is a multiple of 16
bool row16(long long n, int dt) { return (n * elem_bytes(dt)) % 16 == 0; }

// ---- workspace layouts (all offsets 256-byte aligned)

struct TopkLayout {
  size_t fix, t, partial, recs, gkeys, total;
  int nsplit;
};

TopkLayout topk_layout(int B, int d, int r, int vocab) {
  TopkLayout L;
  Ctx dummy{0, 0, 0, nullptr};
  L.nsplit = proj_splits(dummy, B, d, r);
  const size_t n_groups = (size_t)(vocab + GROUP - 1) / GROUP;
  // state that must be zero between calls sits at fixed offsets, so that a call with other
  // arguments never finds another call's data there: the small-batch projection accumulator
  size_t off = WS_HEADER;
  L.fix = off;
  off = align_up(off + WS_FIX_BYTES, 256);
  L.t = off;
  off = align_up(off + (size_t)B * r * 4, 256);
  L.partial = off;
  size_t partial_floats = (size_t)L.nsplit * B * r;
  // tensor-core projection: split-K slices for up to 256 SMs
  partial_floats = std::max(partial_floats, (size_t)proj_mma_splits(B, d, r, 256) * B * r);
  off = align_up(off + partial_floats * 4, 256);
  L.recs = off;
  off = align_up(off + (size_t)B * n_groups * sizeof(GroupRec), 256);
  L.gkeys = off;
  off = align_up(off + (size_t)B * n_groups * sizeof(uint32_t), 256);
  L.total = off;
  return L;
}

// Largest batch for the small-batch pipeline when the tensor-core path also applies (measured on
// the batch-1 shapes through dh_draft_head in CUDA graphs, us per call, small-batch against
// tensor-core path: 20.0 / 25.5 at B = 3, 22.7 / 26.5 at B = 4, 37.1 / 26.5 at B = 5, 43.6 / 27.1
// at B = 8; from five rows the scores kernel's registers no longer let four blocks share an SM).
constexpr int SMALL_MAX_B = 4;

enum Path { PATH_GEMV, PATH_MMA, PATH_FUSED };

// Stage-1 path: the small-batch pipeline (projection + scores kernels) up to SMALL_MAX_B rows where
// the tensor-core path applies and up to 8 rows otherwise, the tensor-core kernels for larger bf16
// batches, the multi-kernel CUDA-core path for the rest.  The DH_FORCE_PATH switch (gemv, mma or
// fused) overrides the choice when the forced path supports the shape (tests and tuning).
Path choose_path(int B, int r, int dtype) {
  const Tuning::Path f = tuning().force_path;
  if (f == Tuning::PATH_GEMV) return PATH_GEMV;
  if (f == Tuning::PATH_MMA && mma_path_supported(B, r, dtype)) return PATH_MMA;
  if (f == Tuning::PATH_FUSED && small_b_supported(B, r, dtype)) return PATH_FUSED;
  // from SMALL_MAX_B rows on, the tensor-core path is faster where it applies (bf16)
  if (small_b_supported(B, r, dtype) && !(B > SMALL_MAX_B && mma_path_supported(B, r, dtype))) return PATH_FUSED;
  if (mma_path_supported(B, r, dtype) && B > SMALL_MAX_B) return PATH_MMA;
  return PATH_GEMV;
}

// ---- profiling

struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::atomic<bool> g_prof{false};
std::vector<ProfRec> g_prof_recs;

}  // namespace

namespace {
thread_local char g_last_error[256] = "";
}

cudaError_t note_error(cudaError_t e, const char* where) {
  if (e != cudaSuccess) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s (%s)", where, cudaGetErrorName(e),
                  cudaGetErrorString(e));
  }
  return e;
}

bool get_ctx(void* stream, Ctx* ctx) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  ctx->device = dev;
  ctx->stream = static_cast<cudaStream_t>(stream);
  if (dev < kMaxDevices && g_sms[dev] > 0) {
    ctx->num_sms = g_sms[dev];
    ctx->l2_bytes = g_l2[dev];
    return true;
  }
  int sms = 0, l2 = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) return false;
  if (dev < kMaxDevices) {
    g_l2[dev] = l2;
    g_sms[dev] = sms;
  }
  ctx->num_sms = sms;
  ctx->l2_bytes = l2;
  return true;
}

void prof_before(const char* name, cudaStream_t s) {
  if (!g_prof) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  ProfRec r{name, nullptr, nullptr};
  if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return;
  cudaEventRecord(r.a, s);
  g_prof_recs.push_back(r);
}

void prof_after(cudaStream_t s) {
  if (!g_prof) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_recs.empty()) cudaEventRecord(g_prof_recs.back().b, s);
}

cudaError_t carveout_max_shared(const void* kernel, int device) {
  static std::mutex mu;
  static std::vector<std::pair<const void*, int>> done;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& d : done)
    if (d.first == kernel && d.second == device) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return note_error(e, "cudaFuncSetAttribute(PreferredSharedMemoryCarveout)");
  done.emplace_back(kernel, device);
  return cudaSuccess;
}

}  // namespace dh

using namespace dh;

extern "C" {

const char* dh_status_string(int status) {
  switch (status) {
    case DH_OK: return "ok";
    case DH_ERR_INVALID_ARG: return "invalid argument";
    case DH_ERR_UNSUPPORTED: return "unsupported alignment, dtype or size";
    case DH_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case DH_ERR_CUDA: return "CUDA error";
    case DH_ERR_TIMEOUT: return "device-side wait timed out";
    case DH_ERR_BAD_INPUT: return "bad input data";
    default: return "unknown status";
  }
}

int dh_version(void) { return 100; }

const char* dh_last_error(void) { return g_last_error; }

// ------------------------------------------------------------------ stage 1

namespace {

// Where stage 1 leaves t for the selection: in the small-batch projection's accumulators (acc) or
// in the activation dtype (t); and the group records.
struct Stage1 {
  const void* t;
  unsigned long long* acc;
  GroupRec* recs;
  const uint32_t* gkeys;  // the groups' best keys (small-batch path, or tensor-core path when asked), else null
};

// Stage 1 up to the group records: projection and scores with group summaries.  want_keys: the
// tensor-core path writes the groups' best keys too (for the fused head's fast selection); the
// small-batch path always does.
int run_records(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r, int vocab,
                int dtype, char* ws, const TopkLayout& L, Stage1* out, bool want_keys = false) {
  void* t = ws + L.t;
  float* partial = reinterpret_cast<float*>(ws + L.partial);
  GroupRec* recs = reinterpret_cast<GroupRec*>(ws + L.recs);
  out->recs = recs;
  out->gkeys = nullptr;
  const Path path = choose_path(B, r, dtype);
  if (path == PATH_FUSED) {
    unsigned long long* acc = reinterpret_cast<unsigned long long*>(ws + L.fix);
    uint32_t* gkeys = reinterpret_cast<uint32_t*>(ws + L.gkeys);
    if (launch_small_b(c, h, U, V, B, d, r, vocab, dtype, acc, recs, gkeys, reinterpret_cast<int*>(ws)) !=
        cudaSuccess)
      return DH_ERR_CUDA;
    out->t = nullptr;
    out->acc = acc;
    out->gkeys = gkeys;
    return DH_OK;
  }
  if (path == PATH_MMA && proj_mma_supported(B, d, r, dtype)) {
    if (launch_proj_mma(c, h, U, B, d, r, partial, proj_mma_splits(B, d, r, 256), t, reinterpret_cast<int*>(ws)) !=
        cudaSuccess)
      return DH_ERR_CUDA;
  } else if (note_error(launch_proj(c, h, U, B, d, r, dtype, partial, L.nsplit, t), "projection") != cudaSuccess) {
    return DH_ERR_CUDA;
  }
  if (path == PATH_MMA) {
    uint32_t* gkeys = want_keys ? reinterpret_cast<uint32_t*>(ws + L.gkeys) : nullptr;
    if (launch_lowrank_mma(c, t, V, B, r, vocab, recs, gkeys, reinterpret_cast<int*>(ws)) != cudaSuccess)
      return DH_ERR_CUDA;
    out->gkeys = gkeys;
  } else if (note_error(launch_scores_summary(c, t, V, B, r, vocab, dtype, recs), "scores") != cudaSuccess) {
    return DH_ERR_CUDA;
  }
  out->t = t;
  out->acc = nullptr;
  return DH_OK;
}

// The selection after the records, one block per row.  tickets (may be null): the rescoring's
// per-row tickets, which the selection clears for the rescoring that follows in the same call.
int run_select(const Ctx& c, const Stage1& s1, const void* V, int B, int r, int vocab, int K, int dtype,
               int32_t* idx_out, float* score_out, uint32_t* tickets = nullptr) {
  if (note_error(launch_select(c, s1.recs, s1.t, s1.acc, V, B, r, vocab, K, dtype, idx_out, score_out, tickets),
                 "select") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// Stage 1 after validation: projection, scores with group summaries, selection.
int run_topk(const Ctx& c, const void* h, const void* U, const void* V, int B, int d, int r, int vocab, int K,
             int dtype, int32_t* idx_out, float* score_out, char* ws, const TopkLayout& L) {
  Stage1 s1;
  const int st = run_records(c, h, U, V, B, d, r, vocab, dtype, ws, L, &s1);
  if (st != DH_OK) return st;
  return run_select(c, s1, V, B, r, vocab, K, dtype, idx_out, score_out);
}

// Stage 2 after validation: the ring kernel from 2048 pairs, the direct kernels below.  The
// DH_FORCE_RESCORE switch (direct, ring or sweep) overrides the choice by batch size (tests and
// tuning); the vocabulary sweep runs only when asked for.
int run_rescore(const Ctx& c, const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                int dtype, float* logits_out, float* probs_out, uint32_t* tickets, int* status) {
  const Tuning::Rescore f = tuning().rescore;
  const bool sweep = f == Tuning::RESCORE_SWEEP && rescore_sweep_supported(B, K, d, vocab, dtype, c.num_sms);
  if (sweep)
    return note_error(launch_rescore_sweep(c, h, W, idx, B, d, vocab, K, dtype, logits_out, probs_out, status),
                      "rescore (sweep)") == cudaSuccess
               ? DH_OK
               : DH_ERR_CUDA;
  const bool ring_ok = rescore_ring_fits(K, d, dtype);  // shape fits the ring's shared memory
  bool ring = ring_ok && rescore_ring_used(B, K, d, dtype);
  if (f == Tuning::RESCORE_DIRECT || f == Tuning::RESCORE_TICKET) ring = false;
  if (f == Tuning::RESCORE_RING || f == Tuning::RESCORE_BUCKET) ring = ring_ok;
  const cudaError_t e =
      ring ? note_error(launch_rescore_ring(c, h, W, idx, B, d, vocab, K, dtype, logits_out, probs_out, tickets,
                                            status, f == Tuning::RESCORE_BUCKET),
                        "rescore (ring)")
           : note_error(launch_rescore(c, h, W, idx, B, d, vocab, K, dtype, logits_out, probs_out, tickets), "rescore");
  return e == cudaSuccess ? DH_OK : DH_ERR_CUDA;
}

}  // namespace

size_t dh_lowrank_topk_workspace(int B, int d, int r, int vocab, int /*K*/, int /*dtype*/) {
  if (B <= 0 || d <= 0 || r <= 0 || vocab <= 0) return 0;
  return topk_layout(B, d, r, vocab).total;
}

int dh_lowrank_topk(const void* h, const void* U, const void* V, int B, int d, int r, int vocab, int K,
                    int dtype, int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                    void* stream) {
  if (B < 0 || d <= 0 || r <= 0 || vocab <= 0) return DH_ERR_INVALID_ARG;
  if (K < 1 || K > vocab || K > DH_MAX_K) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!h || !U || !V || !idx_out || !score_out) return DH_ERR_INVALID_ARG;
  if (r > DH_MAX_RANK || vocab > DH_MAX_VOCAB) return DH_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(U) || !aligned16(V)) return DH_ERR_UNSUPPORTED;
  if (!row16(d, dtype) || !row16(r, dtype) || !row16(vocab, dtype)) return DH_ERR_UNSUPPORTED;
  const TopkLayout L = topk_layout(B, d, r, vocab);
  if (!workspace || !aligned256(workspace) || ws_bytes < L.total) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  return run_topk(c, h, U, V, B, d, r, vocab, K, dtype, idx_out, score_out, static_cast<char*>(workspace), L);
}

// ------------------------------------------------------------------ stage 2

size_t dh_exact_rescore_workspace(int B, int, int, int K, int) {
  if (B <= 0 || K <= 0) return 0;
  return WS_HEADER + align_up((size_t)B * sizeof(uint32_t), 256);
}

int dh_exact_rescore(const void* h, const void* W, const int32_t* idx, int B, int d, int vocab, int K,
                     int dtype, float* logits_out, float* probs_out, void* workspace, size_t ws_bytes,
                     void* stream) {
  if (B < 0 || d <= 0 || vocab <= 0 || K < 1 || K > DH_MAX_K) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!h || !W || !idx || !logits_out) return DH_ERR_INVALID_ARG;
  if (vocab > DH_MAX_VOCAB) return DH_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(W) || !row16(d, dtype)) return DH_ERR_UNSUPPORTED;
  if ((long long)B * K > 0x7FFFFFFFLL || !rescore_supported(d)) return DH_ERR_UNSUPPORTED;
  const size_t need = dh_exact_rescore_workspace(B, d, vocab, K, dtype);
  if (!workspace || !aligned256(workspace) || ws_bytes < need) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  uint32_t* tickets = reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + WS_HEADER);
  return run_rescore(c, h, W, idx, B, d, vocab, K, dtype, logits_out, probs_out, tickets,
                     static_cast<int*>(workspace));
}

// ------------------------------------------------------------------ both stages

namespace {
// Both stages' workspaces: stage 1's layout, then the rescoring tickets.
size_t head_rescore_offset(int B, int d, int r, int vocab) { return align_up(topk_layout(B, d, r, vocab).total, 256); }
}  // namespace

size_t dh_draft_head_workspace(int B, int d, int r, int vocab, int K, int /*dtype*/) {
  if (B <= 0 || d <= 0 || r <= 0 || vocab <= 0 || K <= 0) return 0;
  return head_rescore_offset(B, d, r, vocab) + align_up((size_t)B * sizeof(uint32_t), 256);
}

int dh_draft_head(const void* h, const void* U, const void* V, const void* W, int B, int d, int r, int vocab,
                  int K, int dtype, int32_t* idx_out, float* score_out, float* logits_out, float* probs_out,
                  void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || d <= 0 || r <= 0 || vocab <= 0) return DH_ERR_INVALID_ARG;
  if (K < 1 || K > vocab || K > DH_MAX_K) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!h || !U || !V || !W || !idx_out || !score_out || !logits_out) return DH_ERR_INVALID_ARG;
  if (r > DH_MAX_RANK || vocab > DH_MAX_VOCAB) return DH_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(U) || !aligned16(V) || !aligned16(W)) return DH_ERR_UNSUPPORTED;
  if (!row16(d, dtype) || !row16(r, dtype) || !row16(vocab, dtype)) return DH_ERR_UNSUPPORTED;
  if ((long long)B * K > 0x7FFFFFFFLL || !rescore_supported(d)) return DH_ERR_UNSUPPORTED;
  const TopkLayout L = topk_layout(B, d, r, vocab);
  const size_t roff = head_rescore_offset(B, d, r, vocab);
  if (!workspace || !aligned256(workspace) || ws_bytes < dh_draft_head_workspace(B, d, r, vocab, K, dtype))
    return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  // Batches whose rows the fused cluster head takes in one wave: the stage-1 kernels, then
  // selection and rescoring in one cluster kernel; larger batches (or the DH_FORCE_HEAD=split
  // switch): the selection and rescoring kernels.
  const bool split = tuning().head_split;
  const int ctas = split || !head_cluster_supported(B, d, vocab, K, dtype) ? 0
                                                                          : head_cluster_ctas(c, B, K, d, vocab, dtype);
  const bool fast = ctas && !tuning().head_select_radix;
  Stage1 s1;
  const int st = run_records(c, h, U, V, B, d, r, vocab, dtype, ws, L, &s1, fast);
  if (st != DH_OK) return st;
  if (ctas) {
    if (note_error(launch_head_cluster(c, ctas, s1.recs, fast ? s1.gkeys : nullptr, s1.acc, s1.t, V, h, W, B, d, r,
                                       vocab, K, dtype, idx_out, score_out, logits_out, probs_out,
                                       reinterpret_cast<int*>(ws)),
                   "selection and rescoring (cluster)") != cudaSuccess)
      return DH_ERR_CUDA;
    return DH_OK;
  }
  // the rescoring's tickets sit after stage 1's layout, which depends on the shape: the selection
  // clears them for this call
  const int ss =
      run_select(c, s1, V, B, r, vocab, K, dtype, idx_out, score_out, reinterpret_cast<uint32_t*>(ws + roff));
  if (ss != DH_OK) return ss;
  return run_rescore(c, h, W, idx_out, B, d, vocab, K, dtype, logits_out, probs_out,
                     reinterpret_cast<uint32_t*>(ws + roff), reinterpret_cast<int*>(ws));
}

// ------------------------------------------------------------------ expanding frontier nodes

int dh_expand_children(const float* probs, const int32_t* idx, const float* parent_prob, int B, int K, int w,
                       float min_benefit, int32_t* child_token, float* child_prob, int32_t* n_keep, void* stream) {
  if (B < 0 || K < 1 || K > DH_MAX_K || w < 1 || w > K) return DH_ERR_INVALID_ARG;
  if (B == 0) return DH_OK;
  if (!probs || !idx || !child_token || !child_prob) return DH_ERR_INVALID_ARG;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  if (note_error(launch_expand(c, probs, idx, parent_prob, B, K, w, min_benefit, child_token, child_prob, n_keep),
                 "expand") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// ------------------------------------------------------------------ vocabulary-sharded head

int dh_lowrank_topk_shard(const void* h, const void* U, const void* V_shard, int B, int d, int r, int vocab_shard,
                          int vocab_offset, int K, int dtype, int32_t* idx_out, float* score_out, void* workspace,
                          size_t ws_bytes, void* stream) {
  if (vocab_offset < 0 || (long long)vocab_offset + vocab_shard > DH_MAX_VOCAB) return DH_ERR_INVALID_ARG;
  const int st = dh_lowrank_topk(h, U, V_shard, B, d, r, vocab_shard, K, dtype, idx_out, score_out, workspace,
                                 ws_bytes, stream);
  if (st != DH_OK || B == 0 || vocab_offset == 0) return st;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  if (note_error(launch_add_offset(c, idx_out, (long long)B * K, vocab_offset), "shard id offset") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

int dh_merge_topk(const int32_t* idx_parts, const float* score_parts, int P, int B, int K, int32_t* idx_out,
                  float* score_out, void* stream) {
  if (P < 1 || B < 0 || K < 1 || K > DH_MAX_K) return DH_ERR_INVALID_ARG;
  if ((long long)P * K > DH_MAX_MERGE_ENTRIES) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!idx_parts || !score_parts || !idx_out || !score_out) return DH_ERR_INVALID_ARG;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  if (note_error(launch_merge_topk(c, idx_parts, score_parts, P, B, K, idx_out, score_out), "merge top-K") !=
      cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

size_t dh_exact_rescore_shard_workspace(int B, int d, int vocab_shard, int K, int dtype) {
  if (B <= 0 || K <= 0) return 0;
  return align_up(dh_exact_rescore_workspace(B, d, vocab_shard, K, dtype), 256) +
         align_up((size_t)B * K * sizeof(int32_t), 256);
}

int dh_exact_rescore_shard(const void* h, const void* W_shard, const int32_t* idx, int B, int d, int vocab_shard,
                           int vocab_offset, int K, int dtype, float* logits_out, float* stats_out, void* workspace,
                           size_t ws_bytes, void* stream) {
  if (B < 0 || d <= 0 || vocab_shard <= 0 || K < 1 || K > DH_MAX_K || vocab_offset < 0) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!h || !W_shard || !idx || !logits_out || !stats_out) return DH_ERR_INVALID_ARG;
  if (vocab_shard > DH_MAX_VOCAB) return DH_ERR_UNSUPPORTED;
  if (!aligned16(h) || !aligned16(W_shard) || !row16(d, dtype)) return DH_ERR_UNSUPPORTED;
  if ((long long)B * K > 0x7FFFFFFFLL || !rescore_supported(d)) return DH_ERR_UNSUPPORTED;
  const size_t rs = align_up(dh_exact_rescore_workspace(B, d, vocab_shard, K, dtype), 256);
  if (!workspace || !aligned256(workspace) || ws_bytes < dh_exact_rescore_shard_workspace(B, d, vocab_shard, K, dtype))
    return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  int32_t* local = reinterpret_cast<int32_t*>(ws + rs);
  if (note_error(launch_localize(c, idx, (long long)B * K, vocab_offset, vocab_shard, local), "shard localize") !=
      cudaSuccess)
    return DH_ERR_CUDA;
  // ids owned by another shard are -1 here: the rescoring leaves their logits NaN, unread rows
  const int st = run_rescore(c, h, W_shard, local, B, d, vocab_shard, K, dtype, logits_out, nullptr,
                             reinterpret_cast<uint32_t*>(ws + WS_HEADER), reinterpret_cast<int*>(ws));
  if (st != DH_OK) return st;
  if (note_error(launch_shard_stats(c, local, B, K, logits_out, stats_out), "shard softmax statistics") !=
      cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

int dh_combine_softmax(const float* logits_parts, const float* stats_parts, int P, int B, int K, float* logits_out,
                       float* probs_out, void* stream) {
  if (P < 1 || B < 0 || K < 1 || K > DH_MAX_K) return DH_ERR_INVALID_ARG;
  if (B == 0) return DH_OK;
  if (!logits_parts || !stats_parts || !logits_out) return DH_ERR_INVALID_ARG;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  if (note_error(launch_combine_softmax(c, logits_parts, stats_parts, P, B, K, logits_out, probs_out),
                 "combine softmax") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// ------------------------------------------------------------------ sizing the next level

int dh_size_level(const float* child_prob, const int32_t* child_token, const int32_t* n_valid, int R, int F, int Wc,
                  const float* cost, const int32_t* bin_batch, int n_bins, int wmax, int batch, float theta,
                  int32_t* width_out, int32_t* sel_parent, int32_t* sel_token, float* sel_prob, void* stream) {
  if (R < 0 || F < 1 || Wc < 1 || n_bins < 1 || wmax < 1 || batch < 0) return DH_ERR_INVALID_ARG;
  if (theta != theta) return DH_ERR_INVALID_ARG;
  if ((long long)F * Wc > DH_MAX_LEVEL_CHILDREN || wmax > DH_MAX_K) return DH_ERR_UNSUPPORTED;
  if (R == 0) return DH_OK;
  if (!child_prob || !child_token || !cost || !bin_batch || !width_out || !sel_parent || !sel_token || !sel_prob)
    return DH_ERR_INVALID_ARG;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  if (note_error(launch_size_level(c, child_prob, child_token, n_valid, R, F, Wc, cost, bin_batch, n_bins, wmax, batch,
                                   theta, width_out, sel_parent, sel_token, sel_prob),
                 "size level") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// ------------------------------------------------------------------ tree acceptance

size_t dh_tree_accept_workspace(int B, int N, int /*vocab*/) {
  if (B <= 0 || N <= 0) return 0;
  return WS_HEADER + align_up((size_t)B * N * sizeof(int32_t), 256);
}

int dh_tree_accept(const void* logits, const int32_t* parent, const int32_t* token, int B, int N, int vocab,
                   int dtype, int32_t* argmax_out, int32_t* path_out, int32_t* len_out, int32_t* bonus_out,
                   int32_t* err_out, void* workspace, size_t ws_bytes, void* stream) {
  if (B < 0 || N <= 0 || vocab <= 0) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!logits || !parent || !token || !path_out || !len_out || !bonus_out) return DH_ERR_INVALID_ARG;
  if (N > DH_MAX_TREE_NODES || (long long)B * N > 0x7FFFFFFFLL) return DH_ERR_UNSUPPORTED;
  if (!aligned16(logits) || !row16(vocab, dtype)) return DH_ERR_UNSUPPORTED;
  const size_t need = dh_tree_accept_workspace(B, N, vocab);
  if (!workspace || !aligned256(workspace) || ws_bytes < need) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  int32_t* am_ws = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + WS_HEADER);
  if (note_error(launch_tree(c, logits, parent, token, B, N, vocab, dtype, am_ws, argmax_out, path_out, len_out,
                             bonus_out, err_out),
                 "tree") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// ------------------------------------------------------------------ chain verification

namespace {
constexpr int kVerifyMaxL = 64;
struct VerifyLayout {
  size_t segs, total;
};
VerifyLayout verify_layout(int B, int L, int vocab, int dtype) {
  VerifyLayout v;
  const size_t nrow = (size_t)B * (L + 1);
  v.segs = WS_HEADER;
  v.total = align_up(v.segs + nrow * (size_t)verify_segments(vocab, dtype) * sizeof(float2), 256);
  return v;
}
}  // namespace

size_t dh_verify_chain_workspace(int B, int L, int vocab, int dtype) {
  if (B <= 0 || L < 0 || L > kVerifyMaxL || vocab <= 0 || !valid_dtype(dtype)) return 0;
  return verify_layout(B, L, vocab, dtype).total;
}

int dh_verify_chain(const void* logits, const int32_t* cand_idx, const float* cand_prob, const int32_t* draft_token,
                    const float* u_accept, const float* u_sample, int B, int L, int vocab, int K, int dtype,
                    float temperature, int32_t* n_accept_out, int32_t* token_out, void* workspace, size_t ws_bytes,
                    void* stream) {
  if (B < 0 || L < 0 || vocab <= 0 || K < 0 || K > DH_MAX_K || (L > 0 && K < 1)) return DH_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || !(temperature < INFINITY)) return DH_ERR_INVALID_ARG;
  if (!valid_dtype(dtype)) return DH_ERR_UNSUPPORTED;
  if (B == 0) return DH_OK;
  if (!logits || !u_sample || !n_accept_out || !token_out) return DH_ERR_INVALID_ARG;
  if (L > 0 && (!cand_idx || !cand_prob || !draft_token || !u_accept)) return DH_ERR_INVALID_ARG;
  if (L > kVerifyMaxL || vocab > DH_MAX_VOCAB ||
      (long long)B * (L + 1) * verify_segments(vocab, dtype) > 0x7FFFFFFFLL)
    return DH_ERR_UNSUPPORTED;
  if (!aligned16(logits) || !row16(vocab, dtype)) return DH_ERR_UNSUPPORTED;
  const VerifyLayout Lw = verify_layout(B, L, vocab, dtype);
  if (!workspace || !aligned256(workspace) || ws_bytes < Lw.total) return DH_ERR_WORKSPACE;
  Ctx c;
  if (!get_ctx(stream, &c)) return DH_ERR_CUDA;
  char* ws = static_cast<char*>(workspace);
  if (note_error(launch_verify(c, logits, dtype, B, L, vocab, K, cand_idx, cand_prob, draft_token, u_accept, u_sample,
                               temperature, n_accept_out, token_out, reinterpret_cast<float2*>(ws + Lw.segs)),
                 "verify chain") != cudaSuccess)
    return DH_ERR_CUDA;
  return DH_OK;
}

// ------------------------------------------------------------------ device status

int dh_workspace_status(void* workspace, void* stream, int* status_out) {
  if (!workspace || !status_out || !aligned256(workspace)) return DH_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DH_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), s) != cudaSuccess) return DH_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DH_ERR_CUDA;
  *status_out = v;
  return DH_OK;
}

// ------------------------------------------------------------------ profiling

int dh_prof_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof = on != 0;
  return DH_OK;
}

int dh_prof_read(char* names, int name_len, double* total_ms, int* launches, int max_kernels) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof_recs);
  }
  std::vector<std::string> keys;
  std::vector<double> tot;
  std::vector<int> cnt;
  int rc = 0;
  for (auto& r : recs) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) rc = -1;
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
    size_t k = 0;
    while (k < keys.size() && keys[k] != r.name) ++k;
    if (k == keys.size()) { keys.push_back(r.name); tot.push_back(0.0); cnt.push_back(0); }
    tot[k] += ms;
    cnt[k] += 1;
  }
  if (rc) return -1;
  const int n = (int)keys.size();
  for (int k = 0; k < n && k < max_kernels; ++k) {
    if (names && name_len > 0) {
      std::string s = keys[k].substr(0, (size_t)name_len - 1);
      std::copy(s.begin(), s.end(), names + (size_t)k * name_len);
      names[(size_t)k * name_len + s.size()] = '\0';
    }
    if (total_ms) total_ms[k] = tot[k];
    if (launches) launches[k] = cnt[k];
  }
  return n;
}

}  // extern "C"
