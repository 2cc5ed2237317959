// CPU oracle for the two-stage draft LM head and greedy draft-tree acceptance.
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the CUDA library is
// checked against.  Only the tests, the package smoke check and the benchmark's CPU-baseline leg
// load it; the product path never does.  It shares no code, header, table or helper with the CUDA
// library: it reads the raw input arrays and writes its own outputs.
//
// Arithmetic: every dot product is accumulated in double from the stored (fp32 or bf16) values;
// products of two stored values are exact in double, so only the running sums round.  Steps follow
// the pages' order:
//
//   EAGLE-4 summary page (yuxiaoba.github.io/tech/en/eagle-4), section "Retrieve vocabulary
//   candidates cheaply, then score them exactly": a low-rank head over the full vocabulary
//   retrieves candidates, and the original full-rank head then gives their exact logits.
//     1. t = h U, rounded to the activation dtype (bf16: round to nearest, ties to even).
//     2. s = t V over the whole vocabulary (the factored order (hU)V, which is why the head is
//        cheap; AlphaSignal "EAGLE-4 Triples Qwen3 Inference Speed...", section "Runtime-sized
//        speculation", low-rank candidate head).
//     3. the K candidates: the first K of all v ordered by (s desc, v asc).
//     4. z = h W[idx]^T, the exact full-rank logits of the candidates.
//     5. p = softmax(z) over the K candidates (temperature 1).
//
//   daily.dev "EAGLE-4 speeds up LLM inference with an adaptive speculative decoding drafter",
//   section "How it works": the target checks every drafted token in one pass, matching tokens
//   are kept and the first mismatch is replaced by the target's own token; EAGLE-4 summary page,
//   section "Distribution preservation...": greedy decoding follows the target's choices.
//     6. a[b,n] = argmax_v L[b,n,v] (ties -> lowest v), over the stored values (a NaN ranks
//        below every number; a row of NaN only gives 0);
//        acc[0] = 1, acc[n] = acc[parent[n]] and token[n] == a[b,parent[n]];
//        the deepest accepted node (ties -> lowest node index) ends the accepted path;
//        len = its depth, path = root..node, bonus = a[b,node].
//
//   EAGLE-4 summary page, section "Why a draft tree needs a cost model": products of draft
//   probabilities approximate the benefit of a branch, and a branch is worth computing when its
//   benefit A over its latency cost C passes a threshold (the page's formula itself is lost; this
//   is its plainest reading, with the caller supplying threshold x C); AlphaSignal page, section
//   "Runtime-sized speculation": a top-k of 1 drafts a chain, larger k a tree.
//     7. expanding a frontier node b: its children are its w candidates of highest exact
//        probability p (ties -> lower token id; a NaN probability ranks below every number),
//        child path probability = parent path probability x p (rounded to fp32), and the node
//        keeps its first n_keep children, those whose path probability exceeds min_benefit.
//
//   EAGLE-4 summary page, section "Distribution preservation has algorithmic and implementation
//   conditions": at positive temperature the target verifies the drafted tokens and a rejection
//   correction keeps the target's distribution; each round's depth is fixed before the round.  For
//   a chain of drafted tokens that correction is standard speculative sampling (Leviathan, Kalman
//   and Matias 2023, "Fast Inference from Transformers via Speculative Decoding"; Chen et al. 2023,
//   "Accelerating Large Language Model Decoding with Speculative Sampling"), restated here:
//     8. request b drafted L tokens x_0..x_{L-1}; target logit rows l_0..l_L (row i: the target's
//        next-token logits after the prefix and x_0..x_{i-1}); temperature T > 0:
//          p_i(v) = exp(l_i(v)/T - m_i) / S_i,  m_i = max_v l_i(v)/T,  S_i = sum_v exp(l_i(v)/T - m_i)
//          q_i(v) = the draft's probability of v at position i (listed for K candidate ids, 0 elsewhere)
//        token i is accepted when u_i < p_i(x_i) / q_i(x_i) (always when q_i(x_i) = 0);
//        n = the number of leading accepted tokens;
//        the emitted token y: n < L: y ~ max(0, p_n - q_n) (normalised); n = L: y ~ p_L (bonus);
//        drawn by inverse CDF in vocabulary order with the uniform w_b: y = the smallest v whose
//        running sum of the weights exceeds w_b times their total (a zero total: the weights p_n).
//
//   EAGLE-4 summary page, section "Why a draft tree needs a cost model": latency tables indexed by
//   batch and verification width price another level; products of draft probabilities estimate its
//   benefit A in accepted tokens; each round decides whether to deepen and how wide to go at the
//   current load, by comparing A with its latency cost C against a threshold (the page's formula
//   is lost; this is its plainest per-branch reading).  AlphaSignal page, section "Runtime-sized
//   speculation": depth and branching are chosen for the active batch size.
//     9. sizing the next level of request r: its frontier's candidate children (path probability
//        A, token, parent slot) are ordered by (A desc, parent asc, slot asc; NaN below every
//        number); with the cost row of the current batch (the first bin whose batch bound is at
//        least the batch, else the last), the j-th child (j = 0, 1, ...) is kept while
//          A_j > theta x (cost[j+1] - cost[j])      (fp32: one rounding for the difference, one
//                                                    for the product; the comparison is exact)
//        i.e. while its benefit per unit of its marginal latency passes theta; the first child
//        that fails, or the width limit, ends the level.  width 0 means: do not deepen.
//
// Build: g++ -O2 -std=c++17 -fopenmp -ffp-contract=off -shared -fPIC dh_oracle.cpp
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <utility>
#include <vector>

namespace {

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

// A bf16 value is the upper half of an IEEE-754 binary32 value.
double bf16_value(uint16_t x) {
  uint32_t u = static_cast<uint32_t>(x) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

double stored_value(const void* p, int dtype, size_t i) {
  if (dtype == ORACLE_F32) return static_cast<double>(static_cast<const float*>(p)[i]);
  return bf16_value(static_cast<const uint16_t*>(p)[i]);
}

// Nearest bf16 value to x, ties to the even significand.  bf16 keeps 8 significant bits and the
// exponent range of binary32 (smallest normal 2^-126, subnormal quantum 2^-133).  Scaling by a
// power of two is exact, nearbyint rounds to nearest-even in the default rounding mode.
double round_to_bf16(double x) {
  if (x == 0.0 || !std::isfinite(x)) return x;
  int e = std::ilogb(x);
  if (e < -126) e = -126;
  double q = std::ldexp(x, 7 - e);
  return std::ldexp(std::nearbyint(q), e - 7);
}

double round_to_dtype(double x, int dtype) {
  if (dtype == ORACLE_F32) return static_cast<double>(static_cast<float>(x));
  return round_to_bf16(x);
}

bool valid_dtype(int dtype) { return dtype == ORACLE_F32 || dtype == ORACLE_BF16; }

// Step 1: t[j] = round( sum_i h[b,i] U[i,j] ).
void project_row(const void* h, const void* U, int b, int d, int r, int dtype, double* t) {
  for (int j = 0; j < r; ++j) {
    double acc = 0.0;
    for (int i = 0; i < d; ++i)
      acc += stored_value(h, dtype, (size_t)b * d + i) * stored_value(U, dtype, (size_t)i * r + j);
    t[j] = round_to_dtype(acc, dtype);
  }
}

// Step 2: s[v] = sum_j t[j] V[j,v]; the sum runs over j in ascending order for every v.
void score_row(const double* t, const void* V, int r, int vocab, int dtype, double* s) {
  for (int v = 0; v < vocab; ++v) s[v] = 0.0;
  for (int j = 0; j < r; ++j) {
    const double tj = t[j];
    for (int v = 0; v < vocab; ++v) s[v] += tj * stored_value(V, dtype, (size_t)j * vocab + v);
  }
}

int row_of(const int32_t* rows, int i) { return rows ? rows[i] : i; }

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

// Nearest bf16 (ties to even) of each x, returned as a double.
int oracle_round_bf16(const double* x, int n, double* out) {
  for (int i = 0; i < n; ++i) out[i] = round_to_bf16(x[i]);
  return 0;
}

// Step 1 for the listed rows (rows == nullptr: rows 0..n_rows-1).  t_out: n_rows x r doubles.
int oracle_lowrank_project(const void* h, const void* U, int B, int d, int r, int dtype,
                           const int32_t* rows, int n_rows, double* t_out) {
  if (!valid_dtype(dtype) || B < 0 || d <= 0 || r <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_rows; ++i) project_row(h, U, row_of(rows, i), d, r, dtype, t_out + (size_t)i * r);
  return 0;
}

// Steps 1-2 for the listed rows.  s_out: n_rows x vocab doubles.
int oracle_lowrank_scores(const void* h, const void* U, const void* V, int B, int d, int r, int vocab,
                          int dtype, const int32_t* rows, int n_rows, double* s_out) {
  if (!valid_dtype(dtype) || B < 0 || d <= 0 || r <= 0 || vocab <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_rows; ++i) {
    std::vector<double> t(r);
    project_row(h, U, row_of(rows, i), d, r, dtype, t.data());
    score_row(t.data(), V, r, vocab, dtype, s_out + (size_t)i * vocab);
  }
  return 0;
}

// Steps 1-3 for the listed rows: idx_out / score_out are n_rows x K, ordered by (s desc, v asc).
int oracle_lowrank_topk(const void* h, const void* U, const void* V, int B, int d, int r, int vocab,
                        int K, int dtype, const int32_t* rows, int n_rows, int32_t* idx_out,
                        double* score_out) {
  if (!valid_dtype(dtype) || B < 0 || d <= 0 || r <= 0 || vocab <= 0 || K <= 0 || K > vocab) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_rows; ++i) {
    std::vector<double> t(r), s(vocab);
    project_row(h, U, row_of(rows, i), d, r, dtype, t.data());
    score_row(t.data(), V, r, vocab, dtype, s.data());
    std::vector<std::pair<double, int32_t>> order(vocab);  // (-s, v): ascending = (s desc, v asc)
    for (int v = 0; v < vocab; ++v) order[v] = {-s[v], v};
    std::partial_sort(order.begin(), order.begin() + K, order.end());
    for (int k = 0; k < K; ++k) {
      idx_out[(size_t)i * K + k] = order[k].second;
      score_out[(size_t)i * K + k] = s[order[k].second];
    }
  }
  return 0;
}

// Steps 4-5 for the listed rows: z = h W[idx]^T and p = softmax(z) over the K candidates.
// Returns -2 if an index lies outside [0, vocab).
int oracle_exact_rescore(const void* h, const void* W, const int32_t* idx, int B, int d, int vocab,
                         int K, int dtype, const int32_t* rows, int n_rows, double* logits_out,
                         double* probs_out) {
  if (!valid_dtype(dtype) || B < 0 || d <= 0 || vocab <= 0 || K <= 0) return -1;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : bad)
  for (int i = 0; i < n_rows; ++i) {
    const int b = row_of(rows, i);
    double* z = logits_out + (size_t)i * K;
    for (int k = 0; k < K; ++k) {
      const int32_t v = idx[(size_t)b * K + k];
      if (v < 0 || v >= vocab) { bad += 1; z[k] = NAN; continue; }
      double acc = 0.0;
      for (int c = 0; c < d; ++c)
        acc += stored_value(h, dtype, (size_t)b * d + c) * stored_value(W, dtype, (size_t)v * d + c);
      z[k] = acc;
    }
    if (probs_out) {
      double m = -INFINITY;
      for (int k = 0; k < K; ++k) m = std::max(m, z[k]);
      double sum = 0.0;
      for (int k = 0; k < K; ++k) sum += std::exp(z[k] - m);
      for (int k = 0; k < K; ++k) probs_out[(size_t)i * K + k] = std::exp(z[k] - m) / sum;
    }
  }
  return bad ? -2 : 0;
}

// Step 6 for the listed requests.  logits: B x N x vocab (request-major); outputs per listed
// request i: argmax_out[i*N + n], path_out[i*N + j] (root first, -1 padded), len_out[i],
// bonus_out[i].  A request whose parent array is not a tree rooted at node 0 with parents
// preceding children gets len = -1, bonus = -1 and an all -1 path.
int oracle_tree_accept(const void* logits, const int32_t* parent, const int32_t* token, int B, int N,
                       int vocab, int dtype, const int32_t* reqs, int n_reqs, int32_t* argmax_out,
                       int32_t* path_out, int32_t* len_out, int32_t* bonus_out) {
  if (!valid_dtype(dtype) || B < 0 || N <= 0 || vocab <= 0) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < n_reqs; ++i) {
    const int b = row_of(reqs, i);
    int32_t* a = argmax_out + (size_t)i * N;
    for (int n = 0; n < N; ++n) {
      // NaN ranks below every number: it never becomes the argmax; a row holding only NaN gives 0
      const size_t base = ((size_t)b * N + n) * (size_t)vocab;
      double best = 0.0;
      int32_t arg = -1;
      for (int v = 0; v < vocab; ++v) {
        const double x = stored_value(logits, dtype, base + v);
        if (std::isnan(x)) continue;
        if (arg < 0 || x > best) { best = x; arg = v; }
      }
      a[n] = arg < 0 ? 0 : arg;
    }
    const int32_t* par = parent + (size_t)b * N;
    const int32_t* tok = token + (size_t)b * N;
    int32_t* path = path_out + (size_t)i * N;
    for (int n = 0; n < N; ++n) path[n] = -1;
    bool ok = par[0] == -1;
    for (int n = 1; n < N && ok; ++n) ok = par[n] >= 0 && par[n] < n;
    if (!ok) { len_out[i] = -1; bonus_out[i] = -1; continue; }
    std::vector<int> depth(N, 0);
    std::vector<char> acc(N, 0);
    acc[0] = 1;
    int best = 0;
    for (int n = 1; n < N; ++n) {
      depth[n] = depth[par[n]] + 1;
      acc[n] = acc[par[n]] && tok[n] == a[par[n]];
      if (acc[n] && depth[n] > depth[best]) best = n;  // strict: ties keep the lower node index
    }
    len_out[i] = depth[best];
    bonus_out[i] = a[best];
    for (int n = best, j = depth[best]; n >= 0; n = par[n], --j) path[j] = n;
  }
  return 0;
}

// Step 7 for every row.  probs, idx: B x K (the row's candidates and their exact probabilities);
// parent_prob: B (null = 1); outputs child_token, child_prob: B x w; n_keep: B (may be null).
int oracle_expand_children(const float* probs, const int32_t* idx, const float* parent_prob, int B, int K, int w,
                           float min_benefit, int32_t* child_token, float* child_prob, int32_t* n_keep) {
  if (B < 0 || K <= 0 || w <= 0 || w > K) return -1;
  for (int b = 0; b < B; ++b) {
    const float* p = probs + (size_t)b * K;
    const int32_t* tk = idx + (size_t)b * K;
    // (probability desc, token asc); NaN below every number
    std::vector<int> order(K);
    for (int k = 0; k < K; ++k) order[k] = k;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
      const bool nx = std::isnan(p[x]), ny = std::isnan(p[y]);
      if (nx != ny) return ny;  // the number ranks first
      if (!nx && p[x] != p[y]) return p[x] > p[y];
      return tk[x] < tk[y];
    });
    const double par = parent_prob ? (double)parent_prob[b] : 1.0;
    int keep = 0;
    for (int c = 0; c < w; ++c) {
      const int k = order[c];
      const float a = (float)(par * (double)p[k]);  // the exact product, rounded once to fp32
      child_token[(size_t)b * w + c] = tk[k];
      child_prob[(size_t)b * w + c] = a;
      if (a > min_benefit) ++keep;
    }
    if (n_keep) n_keep[b] = keep;
  }
  return 0;
}

// Step 8 for every request.  logits: B x (L+1) x vocab; cand_idx, cand_prob: B x L x K;
// draft_token, u_accept: B x L; u_sample: B.  Outputs per request: n_accept, token (the emitted
// token).  For comparisons made in other precisions it also reports, with a relative tolerance tol:
// first_close = the first decision i <= n whose |u_i - ratio_i| <= tol * ratio_i (L + 1 if none),
// and [token_lo, token_hi] = the tokens whose cumulative interval meets the target sum +- tol x total.
int oracle_verify_chain(const void* logits, int dtype, int B, int L, int vocab, int K, const int32_t* cand_idx,
                        const float* cand_prob, const int32_t* draft_token, const float* u_accept,
                        const float* u_sample, double temperature, double tol, int32_t* n_accept,
                        int32_t* token, int32_t* first_close, int32_t* token_lo, int32_t* token_hi) {
  if (!valid_dtype(dtype) || B < 0 || L < 0 || vocab <= 0 || K < 0 || !(temperature > 0.0)) return -1;
#pragma omp parallel for schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    const size_t row0 = (size_t)b * (L + 1);
    // p_i(v) for row i of request b, over the whole vocabulary
    auto probs_of_row = [&](int i, std::vector<double>& p) {
      p.assign(vocab, 0.0);
      double m = -INFINITY;
      for (int v = 0; v < vocab; ++v) {
        p[v] = stored_value(logits, dtype, (row0 + i) * (size_t)vocab + v) / temperature;
        m = std::max(m, p[v]);
      }
      double S = 0.0;
      for (int v = 0; v < vocab; ++v) { p[v] = std::exp(p[v] - m); S += p[v]; }
      for (int v = 0; v < vocab; ++v) p[v] /= S;
    };
    // q_i(v): the draft's probability mass at v (summed over the candidate list)
    auto q_of = [&](int i, int v) {
      double q = 0.0;
      for (int k = 0; k < K; ++k)
        if (cand_idx[((size_t)b * L + i) * K + k] == v) q += cand_prob[((size_t)b * L + i) * K + k];
      return q;
    };
    std::vector<double> p;
    int n = 0, close = L + 1;
    for (; n < L; ++n) {
      probs_of_row(n, p);
      const int x = draft_token[(size_t)b * L + n];
      const double px = (x >= 0 && x < vocab) ? p[x] : 0.0;
      const double qx = (x >= 0 && x < vocab) ? q_of(n, x) : 0.0;
      const double u = u_accept[(size_t)b * L + n];
      if (qx <= 0.0) continue;  // ratio +inf: accepted
      const double ratio = px / qx;
      if (close > L && std::fabs(u - ratio) <= tol * ratio) close = n;
      if (!(u < ratio)) break;
    }
    std::vector<double> w(vocab);
    if (n < L) {
      for (int v = 0; v < vocab; ++v) w[v] = p[v];
      for (int k = 0; k < K; ++k) {
        const int v = cand_idx[((size_t)b * L + n) * K + k];
        if (v >= 0 && v < vocab) w[v] -= cand_prob[((size_t)b * L + n) * K + k];
      }
      for (int v = 0; v < vocab; ++v) w[v] = std::max(0.0, w[v]);
    } else {
      probs_of_row(L, p);
      for (int v = 0; v < vocab; ++v) w[v] = p[v];
    }
    double total = 0.0;
    for (int v = 0; v < vocab; ++v) total += w[v];
    if (total <= 0.0) {
      for (int v = 0; v < vocab; ++v) w[v] = p[v];
      total = 0.0;
      for (int v = 0; v < vocab; ++v) total += w[v];
    }
    const double target = (double)u_sample[b] * total, lo = target - tol * total, hi = target + tol * total;
    int y = -1, ylo = -1, yhi = -1, last = 0;
    double c = 0.0;
    for (int v = 0; v < vocab; ++v) {
      if (w[v] > 0.0) last = v;
      c += w[v];
      if (ylo < 0 && c > lo) ylo = v;
      if (y < 0 && c > target) y = v;
      if (yhi < 0 && c > hi) yhi = v;
    }
    if (y < 0) y = last;
    if (ylo < 0) ylo = last;
    if (yhi < 0) yhi = last;
    n_accept[b] = n;
    token[b] = y;
    if (first_close) first_close[b] = close;
    if (token_lo) token_lo[b] = ylo;
    if (token_hi) token_hi[b] = yhi;
  }
  return 0;
}

// Step 9 for every request.  child_prob, child_token: R x F x Wc (per frontier node, its candidate
// children); n_valid: R x F (children valid per node, null = all Wc); cost: n_bins x (wmax + 1)
// latencies in any unit, bin_batch: n_bins batch bounds (ascending); outputs: width R,
// sel_parent / sel_token / sel_prob R x wmax (the kept children in order; -1 / -1 / 0 after width).
int oracle_size_level(const float* child_prob, const int32_t* child_token, const int32_t* n_valid, int R, int F,
                      int Wc, const float* cost, const int32_t* bin_batch, int n_bins, int wmax, int batch, float theta,
                      int32_t* width, int32_t* sel_parent, int32_t* sel_token, float* sel_prob) {
  if (R < 0 || F <= 0 || Wc <= 0 || n_bins <= 0 || wmax <= 0) return -1;
  int bin = n_bins - 1;
  for (int i = 0; i < n_bins; ++i)
    if (batch <= bin_batch[i]) { bin = i; break; }
  const float* c = cost + (size_t)bin * (wmax + 1);
  for (int r = 0; r < R; ++r) {
    struct Child { float a; int f, slot; };
    std::vector<Child> kids;
    for (int f = 0; f < F; ++f) {
      const int nv = n_valid ? std::min(std::max(n_valid[(size_t)r * F + f], 0), Wc) : Wc;
      for (int k = 0; k < nv; ++k) kids.push_back({child_prob[((size_t)r * F + f) * Wc + k], f, k});
    }
    std::stable_sort(kids.begin(), kids.end(), [](const Child& x, const Child& y) {
      const bool nx = std::isnan(x.a), ny = std::isnan(y.a);
      if (nx != ny) return ny;  // the number ranks first
      if (!nx && x.a != y.a) return x.a > y.a;
      if (x.f != y.f) return x.f < y.f;
      return x.slot < y.slot;
    });
    int w = 0;
    while (w < wmax && w < (int)kids.size()) {
      const float dc = c[w + 1] - c[w];
      const float thr = theta * dc;
      if (!(kids[w].a > thr)) break;
      ++w;
    }
    width[r] = w;
    for (int j = 0; j < wmax; ++j) {
      const bool on = j < w;
      sel_parent[(size_t)r * wmax + j] = on ? kids[j].f : -1;
      sel_token[(size_t)r * wmax + j] = on ? child_token[((size_t)r * F + kids[j].f) * Wc + kids[j].slot] : -1;
      sel_prob[(size_t)r * wmax + j] = on ? kids[j].a : 0.0f;
    }
  }
  return 0;
}

}  // extern "C"
