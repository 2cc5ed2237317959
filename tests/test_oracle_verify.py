"""Pins of the oracle's chain verification at positive temperature (standard speculative sampling,
the rejection correction the EAGLE-4 summary page, section "Distribution preservation has
algorithmic and implementation conditions", requires; Leviathan, Kalman and Matias 2023; Chen et
al. 2023).

* Hand-worked cases (tests/golden/verify.txt): acceptance by the ratio, the residual max(0, p - q)
  after a rejection (skipping zero-weight tokens), the bonus token after L acceptances, a drafted
  token outside the candidate list, the temperature.
* Distribution preservation, the property the correction exists for: over many seeded uniforms the
  first emitted token follows the target's p_0, the second (given the first was accepted) follows
  p_1, and the bonus follows p_L.
* A numpy restatement on random small cases (softmax from scipy, inverse CDF by searchsorted).
"""
import os

import numpy as np
import pytest
import scipy.special

import oracle
from speculative_decoding_draft_dh_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden_verify():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "verify.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "prow": [], "pos": []}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key in ("vocab", "L"):
                cur[key] = int(vals[0])
            elif key in ("T", "us"):
                cur[key] = float(vals[0])
            elif key == "prow":
                cur["prow"].append([float(v) for v in vals])
            elif key == "cand":
                cur["pos"].append({"cand": [int(v) for v in vals]})
            elif key == "qprob":
                cur["pos"][-1]["q"] = [float(v) for v in vals]
            elif key == "draft":
                cur["pos"][-1]["x"] = int(vals[0])
            elif key == "u":
                cur["pos"][-1]["u"] = float(vals[0])
            elif key == "expect":
                cur["expect"] = (int(vals[0]), int(vals[1]))
    return cases


def golden_arrays(case):
    """One request: logits T ln(p) (fp32), the candidate lists padded to one K with probability 0."""
    L, V, T = case["L"], case["vocab"], case["T"]
    assert len(case["prow"]) == L + 1 and len(case["pos"]) == L
    logits = (T * np.log(np.array(case["prow"], dtype=np.float64))).astype(np.float32)[None]
    K = max([len(p["cand"]) for p in case["pos"]] + [1])
    ci = np.zeros((1, L, K), dtype=np.int32)
    cq = np.zeros((1, L, K), dtype=np.float32)
    for i, pos in enumerate(case["pos"]):
        n = len(pos["cand"])
        ci[0, i, :n] = pos["cand"]
        cq[0, i, :n] = pos["q"]
        ci[0, i, n:] = pos["cand"][0]  # padding: the first candidate again, with probability 0
    x = np.array([[p["x"] for p in case["pos"]]], dtype=np.int32)
    ua = np.array([[p["u"] for p in case["pos"]]], dtype=np.float32)
    us = np.array([case["us"]], dtype=np.float32)
    return logits, ci, cq, x, ua, us


@pytest.mark.parametrize("case", load_golden_verify(), ids=lambda c: c["name"])
def test_golden_verify(case):
    logits, ci, cq, x, ua, us = golden_arrays(case)
    out = oracle.verify_chain(logits, ci, cq, x, ua, us, temperature=case["T"])
    assert (int(out["n_accept"][0]), int(out["token"][0])) == case["expect"]
    assert out["first_close"][0] == case["L"] + 1  # every hand-worked decision is far from its threshold
    assert out["token_lo"][0] == out["token"][0] == out["token_hi"][0]


def _trials(n, seed, L=2, vocab=8, K=5):
    """n independent rounds with fixed target rows and draft distributions, fresh draws of the
    drafted tokens (from q) and of the uniforms."""
    rng = np.random.default_rng(seed)
    rows = rng.normal(0.0, 1.5, size=(L + 1, vocab)).astype(np.float32)
    cand = np.stack([rng.permutation(vocab)[:K] for _ in range(L)]).astype(np.int32)
    q = rng.dirichlet(np.full(K, 0.7), size=L).astype(np.float32)
    logits = np.broadcast_to(rows, (n, L + 1, vocab)).copy()
    ci = np.broadcast_to(cand, (n, L, K)).copy()
    cq = np.broadcast_to(q, (n, L, K)).copy()
    x = np.empty((n, L), dtype=np.int32)
    for i in range(L):
        w = q[i].astype(np.float64) / q[i].astype(np.float64).sum()
        x[:, i] = cand[i][rng.choice(K, size=n, p=w)]
    ua = rng.random((n, L), dtype=np.float32)
    us = rng.random(n, dtype=np.float32)
    p = scipy.special.softmax(rows.astype(np.float64), axis=-1)
    return logits, ci, cq, x, ua, us, p


def _assert_follows(tokens, p, what):
    n = len(tokens)
    f = np.bincount(tokens, minlength=len(p)) / n
    sigma = np.sqrt(p * (1 - p) / n)
    assert np.all(np.abs(f - p) <= 5 * sigma + 1e-12), f"{what}: {f} against {p}"


def test_emitted_tokens_follow_the_target_distribution():
    """Speculative sampling preserves the target distribution: whatever the draft proposes, the
    first emitted token of a round follows p_0, the next one (when the first was accepted) p_1 and
    the bonus after L acceptances p_L.  With 400000 rounds a count is off by more than 5 standard
    deviations with probability below 1e-5 per token."""
    n, L = 400000, 2
    logits, ci, cq, x, ua, us, p = _trials(n, seed=7, L=L)
    out = oracle.verify_chain(logits, ci, cq, x, ua, us)
    na, tok = out["n_accept"], out["token"]
    assert np.all((na >= 0) & (na <= L))
    first = np.where(na >= 1, x[:, 0], tok)
    _assert_follows(first, p[0], "first token")
    acc1 = na >= 1
    second = np.where(na[acc1] >= 2, x[acc1, 1], tok[acc1])
    _assert_follows(second, p[1], "second token")
    _assert_follows(tok[na == L], p[L], "bonus token")
    # the draft and the target differ, so both outcomes occur often
    assert 0.2 < acc1.mean() < 0.95


def test_temperature_scales_the_target():
    """At temperature T the target is softmax(logits / T): logits multiplied by T at temperature T
    give the T = 1 outcome on every round."""
    logits, ci, cq, x, ua, us, _ = _trials(2000, seed=3)
    a = oracle.verify_chain(logits, ci, cq, x, ua, us, temperature=1.0)
    b = oracle.verify_chain(logits * np.float32(4.0), ci, cq, x, ua, us, temperature=4.0)
    sure = (a["first_close"] > 2) & (a["token_lo"] == a["token_hi"])
    assert sure.mean() > 0.99
    np.testing.assert_array_equal(a["n_accept"][sure], b["n_accept"][sure])
    np.testing.assert_array_equal(a["token"][sure], b["token"][sure])


def _numpy_verify(logits, ci, cq, x, ua, us, T):
    """Independent restatement in numpy: probabilities from scipy's softmax, the residual by
    vectorised clipping, the inverse CDF by searchsorted on the cumulative sum."""
    B, L1, V = logits.shape
    L = L1 - 1
    na = np.zeros(B, dtype=np.int64)
    tok = np.zeros(B, dtype=np.int64)
    for b in range(B):
        p = scipy.special.softmax(logits[b].astype(np.float64) / T, axis=-1)
        q = np.zeros((L, V))
        for i in range(L):
            np.add.at(q[i], ci[b, i], cq[b, i].astype(np.float64))
        n = 0
        while n < L:
            qx = q[n, x[b, n]]
            if qx > 0 and not (ua[b, n] < p[n, x[b, n]] / qx):
                break
            n += 1
        w = np.clip(p[n] - q[n], 0, None) if n < L else p[L]
        if w.sum() <= 0:
            w = p[n]
        c = np.cumsum(w)
        tok[b] = min(int(np.searchsorted(c, us[b] * c[-1], side="right")), V - 1)
        na[b] = n
    return na, tok


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_matches_numpy_restatement(seed):
    cfg = inputs.verify_config("tiny_verify", vocab=512, K=12)
    v = inputs.make_verify(cfg, seed=seed)
    arr = {k: t.numpy() for k, t in v.items()}
    out = oracle.verify_chain(arr["logits"], arr["cand_idx"], arr["cand_prob"], arr["draft_token"],
                              arr["u_accept"], arr["u_sample"], temperature=1.3)
    na, tok = _numpy_verify(arr["logits"], arr["cand_idx"], arr["cand_prob"], arr["draft_token"],
                            arr["u_accept"], arr["u_sample"], 1.3)
    sure = out["first_close"] > cfg.L
    assert sure.mean() > 0.5
    np.testing.assert_array_equal(out["n_accept"][sure], na[sure])
    np.testing.assert_array_equal(out["token"][sure], tok[sure])
    assert np.all((out["token_lo"] <= out["token"]) & (out["token"] <= out["token_hi"]))


def test_generator_shapes_and_draws():
    cfg = inputs.verify_config("tiny_verify")
    v = inputs.make_verify(cfg, seed=0)
    B, L, K = cfg.B, cfg.L, cfg.K
    assert v["logits"].shape == (B, L + 1, cfg.vocab) and v["cand_idx"].shape == (B, L, K)
    ci = v["cand_idx"].numpy()
    for b in range(B):
        for i in range(L):
            assert len(set(ci[b, i].tolist())) == K
            assert v["draft_token"][b, i].item() in ci[b, i]
    np.testing.assert_allclose(v["cand_prob"].numpy().sum(-1), 1.0, atol=1e-5)
    assert (v["u_accept"] >= 0).all() and (v["u_accept"] < 1).all()
