"""Pins of the oracle's level sizing (step 9): the per-branch reading of the cost model of the
EAGLE-4 summary page, section "Why a draft tree needs a cost model".

* Hand-worked cases (tests/golden/sizing.txt): light and heavy load, bin lookup, ties to the lower
  parent, the strict threshold, the width limit.
* A brute force over random frontiers: every order of the children is tried against the rule
  "child j of the (A desc, parent, slot) order is kept while A_j > theta x (cost[j+1] - cost[j])",
  in numpy float32, and heavier loads never get a wider level from the synthetic table.
"""
import os

import numpy as np
import pytest

import oracle
from speculative_decoding_draft_dh_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden_sizing():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "sizing.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0], "cost": [], "nodes": [], "toks": [], "keep": []}
            elif key == "end":
                cases.append(cur)
                cur = None
            elif key == "bins":
                cur["bins"] = [int(v) for v in vals]
            elif key == "cost":
                cur["cost"].append([float(v) for v in vals])
            elif key in ("batch", "expect"):
                cur[key] = int(vals[0])
            elif key == "theta":
                cur["theta"] = float(vals[0])
            elif key == "node":
                cur["nodes"].append([float(v) for v in vals])
            elif key == "tok":
                cur["toks"].append([int(v) for v in vals])
            elif key == "keep":
                cur["keep"].append((int(vals[0]), int(vals[1])))
    return cases


def golden_arrays(case):
    F = len(case["nodes"])
    Wc = max(len(n) for n in case["nodes"])
    prob = np.zeros((1, F, Wc), dtype=np.float32)
    tok = np.full((1, F, Wc), -1, dtype=np.int32)
    nv = np.zeros((1, F), dtype=np.int32)
    for f, (ps, ts) in enumerate(zip(case["nodes"], case["toks"])):
        prob[0, f, :len(ps)] = ps
        tok[0, f, :len(ts)] = ts
        nv[0, f] = len(ps)
    return prob, tok, nv, np.array(case["cost"], dtype=np.float32), np.array(case["bins"], dtype=np.int32)


@pytest.mark.parametrize("case", load_golden_sizing(), ids=lambda c: c["name"])
def test_golden_sizing(case):
    prob, tok, nv, cost, bins = golden_arrays(case)
    out = oracle.size_level(prob, tok, cost, bins, case["batch"], case["theta"], n_valid=nv)
    w = case["expect"]
    assert out["width"][0] == w
    assert [(int(out["parent"][0, j]), int(np.where(tok[0, out["parent"][0, j]] == out["token"][0, j])[0][0]))
            for j in range(w)] == case["keep"]
    assert np.all(out["parent"][0, w:] == -1) and np.all(out["token"][0, w:] == -1)


def _brute(prob, tok, nv, cost, bins, batch, theta):
    """numpy float32 restatement: lexsort of (slot, parent, -A), then the first failing child."""
    R, F, Wc = prob.shape
    wmax = cost.shape[1] - 1
    b = next((i for i, x in enumerate(bins) if batch <= x), len(bins) - 1)
    thr = (np.float32(theta) * (cost[b, 1:] - cost[b, :-1]).astype(np.float32)).astype(np.float32)
    widths, kept = [], []
    for r in range(R):
        f_, k_ = np.nonzero(np.arange(Wc)[None, :] < nv[r][:, None])
        a = prob[r, f_, k_]
        order = np.lexsort((k_, f_, -a))
        w = 0
        while w < min(wmax, len(order)) and a[order[w]] > thr[w]:
            w += 1
        widths.append(w)
        kept.append([(int(f_[order[j]]), int(tok[r, f_[order[j]], k_[order[j]]])) for j in range(w)])
    return widths, kept


@pytest.mark.parametrize("batch", [1, 8, 30, 64, 512, 4096])
def test_random_frontiers_against_brute_force(batch):
    x = inputs.make_frontier_children(R=40, F=6, Wc=4, seed=batch)
    rng = np.random.default_rng(batch)
    x["n_valid"] = rng.integers(0, 5, size=(40, 6)).astype(np.int32)
    x["child_prob"][:, :, 1] = x["child_prob"][:, :, 0]  # equal probabilities within a node
    cost, bins = inputs.latency_table(wmax=12)
    theta = 0.004
    out = oracle.size_level(x["child_prob"], x["child_token"], cost, bins, batch, theta, n_valid=x["n_valid"])
    widths, kept = _brute(x["child_prob"], x["child_token"], x["n_valid"], cost, bins, batch, theta)
    assert out["width"].tolist() == widths
    for r in range(40):
        got = [(int(out["parent"][r, j]), int(out["token"][r, j])) for j in range(widths[r])]
        assert got == kept[r]
    if batch == 1:
        assert max(widths) > 1


def test_heavier_load_never_widens():
    x = inputs.make_frontier_children(R=64, F=8, Wc=4, seed=3)
    cost, bins = inputs.latency_table(wmax=16)
    prev = None
    for batch in (1, 8, 64, 512):
        w = oracle.size_level(x["child_prob"], x["child_token"], cost, bins, batch, 0.003)["width"]
        if prev is not None:
            assert np.all(w <= prev)
        prev = w
