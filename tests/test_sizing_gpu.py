"""GPU parity of sizing the next draft level (dh_size_level) against the oracle, bit for bit: the
decision is taken in fp32 on both sides with the same rounded operations."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_dh_gb300 import binding as dh
from speculative_decoding_draft_dh_gb300 import inputs
from tests.test_oracle_sizing import golden_arrays, load_golden_sizing

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def compare(prob, tok, nv, cost, bins, batch, theta):
    g = dh.size_level(to_dev(prob), to_dev(tok), to_dev(cost), to_dev(bins), batch, theta,
                      n_valid=None if nv is None else to_dev(nv))
    torch.cuda.synchronize()
    o = oracle.size_level(prob, tok, cost, bins, batch, theta, n_valid=nv)
    for k in ("width", "parent", "token", "prob"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), o[k], err_msg=k)
    return o


@pytest.mark.parametrize("case", load_golden_sizing(), ids=lambda c: c["name"])
def test_golden_sizing_on_gpu(case):
    prob, tok, nv, cost, bins = golden_arrays(case)
    o = compare(prob, tok, nv, cost, bins, case["batch"], case["theta"])
    assert o["width"][0] == case["expect"]


@pytest.mark.parametrize("batch", [1, 8, 40, 512])
@pytest.mark.parametrize("shape", [(40, 6, 4), (3, 64, 16), (7, 1, 1), (2, 512, 16)])
def test_random_frontiers(batch, shape):
    R, F, Wc = shape
    x = inputs.make_frontier_children(R, F, Wc, seed=F + batch)
    rng = np.random.default_rng(batch)
    nv = rng.integers(0, Wc + 1, size=(R, F)).astype(np.int32)
    x["child_prob"][:, ::3, 0] = x["child_prob"][:, ::3, -1]  # equal probabilities across nodes
    x["child_prob"][0, 0, 0] = np.nan                         # NaN ranks below every number
    x["child_prob"][-1, -1, -1] = -0.0
    cost, bins = inputs.latency_table(wmax=min(64, F * Wc))
    compare(x["child_prob"], x["child_token"], nv, cost, bins, batch, 0.004)
    compare(x["child_prob"], x["child_token"], None, cost, bins, batch, -1.0)  # every child passes


def test_draft_level_with_sizing_matches_oracle():
    """One draft level end to end on the GPU: the head for every frontier node of two requests, the
    children by exact probability, then the next level's width and children at the current load;
    each step checked against the oracle on the GPU's own inputs to it."""
    cfg = inputs.head_config("tiny", B=8, K=16)
    x = inputs.make_head(cfg, seed=34, device=DEV)
    idx, score, logits, probs = dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K)
    par = torch.linspace(1.0, 0.2, 8, dtype=torch.float32, device=DEV)
    tok, cp, keep = dh.expand_children(probs, idx, 4, parent_prob=par, min_benefit=0.001)
    cost, bins = inputs.latency_table(wmax=8)
    g = dh.size_level(cp.view(2, 4, 4), tok.view(2, 4, 4), to_dev(cost), to_dev(bins), 2, 0.002,
                      n_valid=keep.view(2, 4))
    torch.cuda.synchronize()
    o = oracle.size_level(cp.view(2, 4, 4).cpu().numpy(), tok.view(2, 4, 4).cpu().numpy(), cost, bins, 2, 0.002,
                          n_valid=keep.view(2, 4).cpu().numpy())
    for k in ("width", "parent", "token", "prob"):
        np.testing.assert_array_equal(g[k].cpu().numpy(), o[k], err_msg=k)
    assert o["width"].max() > 0
