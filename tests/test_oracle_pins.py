"""Pins for the CPU oracle: checks against things other than the oracle itself.

* bf16 rounding against torch's binary32->bf16 conversion and against a brute-force nearest search
  over every finite bf16 value;
* the candidate list against a numpy lexsort of independently computed low-rank scores;
* exact logits against the full-vocabulary head h W^T (brute force);
* K = vocab, where the two-stage head reduces to the full softmax (scipy);
* W = (U V)^T with no noise, where stage 2 reproduces stage 1;
* hand-built trees with hand-derived results (tests/golden/trees.txt);
* random trees against a brute-force acceptance check that walks every node to the root;
* softmax invariants.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from speculative_decoding_draft_dh_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- bf16 rounding

def _all_bf16_positive_finite():
    bits = np.arange(0, 0x7F80, dtype=np.uint32)  # +0 .. largest finite
    return (bits << 16).view(np.float32).astype(np.float64), bits


_BF16_GRID, _BF16_BITS = _all_bf16_positive_finite()


def brute_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 by searching the sorted grid of all positive finite bf16 values; ties go to
    the grid point whose bit pattern is even."""
    out = np.empty_like(x)
    for i, v in enumerate(x.ravel()):
        a = abs(v)
        j = int(np.searchsorted(_BF16_GRID, a))
        cands = [c for c in (j - 1, j) if 0 <= c < len(_BF16_GRID)]
        best = min(cands, key=lambda c: (abs(_BF16_GRID[c] - a), _BF16_BITS[c] & 1))
        out.ravel()[i] = math.copysign(_BF16_GRID[best], v)
    return out


def test_round_bf16_matches_torch_on_binary32_values():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # force a third of them onto exact halfway points between two bf16 values
    bits[::3] = (bits[::3] & 0xFFFF0000) | 0x8000
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3e38)]
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).float().numpy().astype(np.float64)
    got = oracle.round_bf16(x.astype(np.float64))
    np.testing.assert_array_equal(got, want)


def test_round_bf16_matches_brute_force_on_doubles():
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-40, 38, 3000),
                        rng.standard_normal(200) * 1e-39])  # include bf16 subnormals
    np.testing.assert_array_equal(oracle.round_bf16(x), brute_bf16(x))


# ---------------------------------------------------------------- stage 1

MID = inputs.HeadConfig("mid_bf16", 3, 512, 8192, 64, 32, "bf16", 0.1, True)


def _f64(t):
    return t.detach().float().double().numpy()


def _independent_scores(h, U, V, dtype):
    """Low-rank scores computed without the oracle: t rounded by numpy (fp32) or by the brute-force
    bf16 grid search, then a float64 matmul."""
    t = _f64(h) @ _f64(U)
    t = t.astype(np.float32).astype(np.float64) if dtype == "f32" else brute_bf16(t)
    return t @ _f64(V)


@pytest.mark.parametrize("cfg", [inputs.HEAD_CONFIGS["tiny"], MID], ids=["tiny_f32", "mid_bf16"])
def test_topk_matches_lexsort(cfg):
    x = inputs.make_head(cfg, seed=0, with_W=False)
    s = _independent_scores(x["h"], x["U"], x["V"], cfg.dtype)
    idx, sc = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    for b in range(cfg.B):
        order = np.lexsort((np.arange(cfg.vocab), -s[b]))[: cfg.K]
        np.testing.assert_array_equal(idx[b], order)
        np.testing.assert_allclose(sc[b], s[b][order], rtol=1e-12, atol=1e-12)
    full = oracle.lowrank_scores(x["h"], x["U"], x["V"])
    np.testing.assert_allclose(full, s, rtol=1e-12, atol=1e-12)


def test_project_rounds_to_activation_dtype():
    cfg = MID
    x = inputs.make_head(cfg, seed=3, with_W=False)
    t = oracle.lowrank_project(x["h"], x["U"])
    exact = _f64(x["h"]) @ _f64(x["U"])
    np.testing.assert_array_equal(t, brute_bf16(exact))
    # every value is a bf16 value
    np.testing.assert_array_equal(t, torch.from_numpy(t).float().to(torch.bfloat16).double().numpy())


def test_rows_subset_matches_full():
    cfg = inputs.HEAD_CONFIGS["tiny"]
    x = inputs.make_head(cfg, seed=5)
    idx, sc = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    idx2, sc2 = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, rows=[3, 1])
    np.testing.assert_array_equal(idx2, idx[[3, 1]])
    np.testing.assert_array_equal(sc2, sc[[3, 1]])


# ---------------------------------------------------------------- stage 2

@pytest.mark.parametrize("cfg", [inputs.HEAD_CONFIGS["tiny"], MID], ids=["tiny_f32", "mid_bf16"])
def test_exact_logits_match_full_head(cfg):
    x = inputs.make_head(cfg, seed=0)
    idx, _ = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    z, p = oracle.exact_rescore(x["h"], x["W"], idx)
    full = _f64(x["h"]) @ _f64(x["W"]).T  # brute force: the whole full-rank head
    hits = 0
    for b in range(cfg.B):
        np.testing.assert_allclose(z[b], full[b][idx[b]], rtol=1e-9, atol=1e-12)
        top = int(np.argmax(full[b]))
        if top in set(idx[b].tolist()):
            hits += 1
            assert idx[b][int(np.argmax(z[b]))] == top
    assert hits >= 1  # the retrieval finds the full-head argmax on these inputs


def test_K_equals_vocab_reduces_to_full_softmax():
    cfg = inputs.head_config("tiny", K=4096)
    x = inputs.make_head(cfg, seed=0)
    idx, _ = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    z, p = oracle.exact_rescore(x["h"], x["W"], idx)
    full = _f64(x["h"]) @ _f64(x["W"]).T
    for b in range(cfg.B):
        np.testing.assert_array_equal(np.sort(idx[b]), np.arange(cfg.vocab))
        ref = scipy.special.softmax(full[b])
        np.testing.assert_allclose(p[b], ref[idx[b]], rtol=1e-10, atol=1e-15)


def test_noiseless_full_head_reproduces_stage1():
    cfg = inputs.head_config("tiny", noise=0.0)
    x = inputs.make_head(cfg, seed=7)
    idx, s = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    z, _ = oracle.exact_rescore(x["h"], x["W"], idx)
    scale = np.abs(s).max()
    np.testing.assert_allclose(z, s, rtol=0, atol=1e-5 * scale)
    for b in range(cfg.B):
        gap = s[b, 0] - s[b, 1]
        if gap > 1e-4 * scale:
            assert int(np.argmax(z[b])) == 0


def test_softmax_invariants():
    cfg = inputs.HEAD_CONFIGS["tiny"]
    x = inputs.make_head(cfg, seed=11)
    idx, _ = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    z, p = oracle.exact_rescore(x["h"], x["W"], idx)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    for b in range(cfg.B):
        o = np.argsort(-z[b], kind="stable")
        assert np.all(np.diff(p[b][o]) <= 1e-15)
        assert np.all(p[b] > 0)


def test_rescore_flags_out_of_range_index():
    cfg = inputs.HEAD_CONFIGS["tiny"]
    x = inputs.make_head(cfg, seed=0)
    idx = np.zeros((cfg.B, cfg.K), dtype=np.int32)
    idx[1, 3] = cfg.vocab
    z, p = oracle.exact_rescore(x["h"], x["W"], idx)
    assert np.isnan(z[1, 3]) and not np.isnan(z[0]).any()


# ---------------------------------------------------------------- trees

def load_golden_trees():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "trees.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "ties": []}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key == "tie":
                cur["ties"].append(tuple(int(v) for v in vals))
            elif key == "vocab":
                cur["vocab"] = int(vals[0])
            else:
                cur[key] = [int(v) for v in vals]
    return cases


def golden_tree_arrays(case, dtype=np.float32):
    N, vocab = len(case["parent"]), case["vocab"]
    rng = np.random.default_rng(0)
    logits = rng.uniform(-1.0, 1.0, size=(1, N, vocab)).astype(dtype)
    for n, a in enumerate(case["argmax"]):
        logits[0, n, a] = 4.0
    for n, a, b in case["ties"]:
        logits[0, n, :] = np.minimum(logits[0, n, :], 1.0)
        logits[0, n, a] = logits[0, n, b] = 6.0
    parent = np.array([case["parent"]], dtype=np.int32)
    token = np.array([case["token"]], dtype=np.int32)
    return logits, parent, token


@pytest.mark.parametrize("case", load_golden_trees(), ids=lambda c: c["name"])
def test_golden_trees(case):
    logits, parent, token = golden_tree_arrays(case)
    out = oracle.tree_accept(logits, parent, token)
    N = parent.shape[1]
    assert out["len"][0] == case["expect_len"][0]
    assert out["bonus"][0] == case["expect_bonus"][0]
    want = case["expect_path"] + [-1] * (N - len(case["expect_path"]))
    assert out["path"][0].tolist() == want
    if case["expect_len"][0] >= 0:
        want_arg = list(case["argmax"])
        for n, a, _ in case["ties"]:
            want_arg[n] = a
        assert out["argmax"][0].tolist() == want_arg


def _brute_accept(a, parent, token):
    """Accept node n iff every edge on its root path drafts the target's argmax; return the
    accepted node of greatest depth (lowest index on ties) and its depth."""
    N = len(parent)
    best, best_depth = 0, 0
    for n in range(N):
        m, depth, ok = n, 0, True
        while m != 0:
            ok &= bool(token[m] == a[parent[m]])
            m, depth = parent[m], depth + 1
        if ok and depth > best_depth:
            best, best_depth = n, depth
    return best, best_depth


@pytest.mark.parametrize("tcfg", [inputs.TREE_CONFIGS["tiny_tree"],
                                  inputs.tree_config("tree", B=6, vocab=2048)],
                         ids=["tiny_tree", "deep_tree_small_vocab"])
def test_random_trees_against_brute_force(tcfg):
    t = inputs.make_tree(tcfg, seed=0)
    out = oracle.tree_accept(t["logits"], t["parent"], t["token"])
    L = t["logits"].float().numpy()
    par, tok = t["parent"].numpy(), t["token"].numpy()
    total_len = 0
    for b in range(tcfg.B):
        a = np.argmax(L[b], axis=-1)  # numpy returns the first maximum
        np.testing.assert_array_equal(out["argmax"][b], a)
        node, depth = _brute_accept(a, par[b], tok[b])
        assert out["len"][b] == depth
        path = out["path"][b]
        assert path[depth] == node and (depth + 1 == tcfg.N or path[depth + 1] == -1)
        for j in range(depth, 0, -1):
            assert par[b][path[j]] == path[j - 1]
        assert path[0] == 0
        assert out["bonus"][b] == a[node]
        total_len += depth
    assert total_len > 0  # the 0.7 boost makes acceptance non-trivial


def _brute_argmax_nan_last(row):
    """Lowest id holding the largest number of the row; NaN never wins; 0 if the row has no number."""
    best = None
    for v, x in enumerate(row.tolist()):
        if x != x:
            continue
        if best is None or x > row[best]:
            best = v
    return 0 if best is None else best


def test_tree_argmax_nan_ranks_below_numbers():
    nan, inf = np.nan, np.inf
    rows = np.array([[nan, 1.0, 3.0, 3.0, -2.0, nan, 0.5, 2.0],
                     [3.0, nan, 3.0, 1.0, nan, nan, 9.0, nan],
                     [nan] * 8,
                     [nan, -inf, -inf, nan, nan, nan, nan, nan],
                     [-inf, nan, 5.0, nan, 5.0, -1.0, nan, 4.0],
                     [nan, nan, nan, nan, nan, nan, nan, -7.0]], dtype=np.float32)
    N = rows.shape[0]
    logits = rows.reshape(1, N, 8)
    parent = np.array([[-1] + list(range(N - 1))], dtype=np.int32)
    want = [_brute_argmax_nan_last(r) for r in rows]
    assert want == [2, 6, 0, 1, 2, 7]
    token = np.array([[0] + want[:-1]], dtype=np.int32)  # every edge matches: a chain
    out = oracle.tree_accept(logits, parent, token)
    assert out["argmax"][0].tolist() == want
    assert out["len"][0] == N - 1 and out["bonus"][0] == want[-1]


def test_tree_generator_shape_limits():
    tcfg = inputs.tree_config("tree", B=8, vocab=1024)
    par = inputs.make_parents(tcfg.B, tcfg.N, 0, tcfg.max_depth, tcfg.max_children)
    for b in range(tcfg.B):
        depth = [0] * tcfg.N
        kids = [0] * tcfg.N
        for n in range(1, tcfg.N):
            assert 0 <= par[b, n] < n
            depth[n] = depth[par[b, n]] + 1
            kids[par[b, n]] += 1
        assert max(depth) <= 10 and max(kids) <= 4


# ---------------------------------------------------------------- step 7: expanding a frontier node

def load_golden_expansions():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "expand.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key in ("tokens", "expect_tokens"):
                cur[key] = [int(v) for v in vals]
            elif key in ("w", "expect_keep"):
                cur[key] = int(vals[0])
            elif key in ("parent", "min_benefit"):
                cur[key] = float(vals[0])
            else:
                cur[key] = [float(v) for v in vals]
    return cases


@pytest.mark.parametrize("case", load_golden_expansions(), ids=lambda c: c["name"])
def test_golden_expansions(case):
    tok, cp, keep = oracle.expand_children(np.array([case["probs"]], dtype=np.float32),
                                           np.array([case["tokens"]], dtype=np.int32), case["w"],
                                           parent_prob=np.array([case["parent"]], dtype=np.float32),
                                           min_benefit=case["min_benefit"])
    assert tok[0].tolist() == case["expect_tokens"]
    np.testing.assert_array_equal(cp[0], np.array(case["expect_probs"], dtype=np.float32))
    assert keep[0] == case["expect_keep"]


@pytest.mark.parametrize("w", [1, 4, 64])
def test_expansion_matches_lexsort(w):
    """Against numpy: lexsort by (probability desc, token asc), fp32 products, a prefix count."""
    rng = np.random.default_rng(40 + w)
    B, K = 6, 64
    p = rng.dirichlet(np.ones(K), size=B).astype(np.float32)
    p[:, 5] = p[:, 9]  # exact ties between candidates
    p[2, :8] = p[2, 8]
    tok = np.stack([rng.permutation(100000)[:K] for _ in range(B)]).astype(np.int32)
    par = rng.uniform(0.1, 1.0, size=B).astype(np.float32)
    thr = 0.01
    ct, cp, keep = oracle.expand_children(p, tok, w, parent_prob=par, min_benefit=thr)
    for b in range(B):
        order = np.lexsort((tok[b], -p[b].astype(np.float64)))[:w]
        assert ct[b].tolist() == tok[b][order].tolist()
        want = (np.float32(par[b]) * p[b][order]).astype(np.float32)
        np.testing.assert_array_equal(cp[b], want)
        assert keep[b] == int(np.sum(want > np.float32(thr)))
        assert np.all(np.diff(cp[b]) <= 0)
