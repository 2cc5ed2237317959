"""GPU parity of the vocabulary-sharded draft head: P shards run on one GPU one after another, then
the merge and the softmax combination, against the oracle (candidates with the tie band, logits and
probabilities within the usual tolerances) and the unsharded library call.

A candidate's low-rank score is the scores kernel's, or, when its group was re-scored exactly by the
selection (a group whose third score reaches the K-th), the refinement's, whose summation order
differs; which groups are refined depends on the shard.  So the merged scores equal the unsharded
ones to rounding, and the candidate lists agree except inside the tie band; where the ids agree the
logits are bit-identical (the same dot product)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_dh_gb300 import binding as dh
from speculative_decoding_draft_dh_gb300 import inputs, sharded
from tests.parity import check_candidates, check_logits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def sharded_vs_unsharded(cfg, P, seed, rows_for_oracle=None):
    x = inputs.make_head(cfg, seed=seed, device=DEV)
    h, U, V, W = x["h"], x["U"], x["V"], x["W"]
    shards = sharded.split_weights(V, W, P, align=8 if cfg.dtype == "bf16" else 4)
    idx, score, logits, probs = sharded.step_on_shards(h, U, shards, cfg.K)
    ui, us = dh.lowrank_topk(h, U, V, cfg.K)
    ul, up = dh.exact_rescore(h, W, ui)
    torch.cuda.synchronize()
    # stage 1 merged from the shards: the unsharded candidates (ties aside), scores to rounding
    same = idx == ui
    assert same.float().mean().item() > 0.98
    np.testing.assert_allclose(score.cpu().numpy(), us.cpu().numpy(), rtol=1e-5, atol=1e-5)
    # stage 2 from the owners: the unsharded logits bit for bit where the ids agree
    assert torch.equal(logits[same], ul[same])
    if bool(same.all()):
        np.testing.assert_allclose(probs.cpu().numpy(), up.cpu().numpy(), atol=1e-6, rtol=1e-5)
    # and against the oracle
    rows = list(range(cfg.B)) if rows_for_oracle is None else rows_for_oracle
    hc, Uc, Vc, Wc = h.cpu(), U.cpu(), V.cpu(), W.cpu()
    s_full = oracle.lowrank_scores(hc, Uc, Vc, rows=rows)
    oz, op = oracle.exact_rescore(hc, Wc, idx.cpu(), rows=rows)
    for n, b in enumerate(rows):
        check_candidates(idx[b].cpu().numpy(), score[b].cpu().numpy(), s_full[n], cfg.K, where=f"row {b}")
        check_logits(logits[b].cpu().numpy(), probs[b].cpu().numpy(), oz[n], op[n], where=f"row {b}")


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_tiny_shards(P):
    sharded_vs_unsharded(inputs.head_config("tiny", B=4, K=16), P, seed=40 + P)


@pytest.mark.parametrize("P", [2, 4, 8])
def test_batch1_shards(P):
    sharded_vs_unsharded(inputs.HEAD_CONFIGS["batch1"], P, seed=50 + P)


def test_moderate_shards():
    sharded_vs_unsharded(inputs.HEAD_CONFIGS["moderate"], 4, seed=60, rows_for_oracle=list(range(0, 64, 8)))


def test_merge_pads_and_skips_invalid_entries():
    """Fewer than K valid entries over the parts: the row is padded with (-1, -inf); ids < 0 and NaN
    scores never take a rank; equal scores go to the lower id across parts."""
    P, B, K = 3, 2, 4
    idx = torch.tensor([[[5, 9, -1, -1], [1, 2, 3, 4]], [[20, 21, -1, -1], [7, 8, 9, 10]],
                        [[30, -1, -1, -1], [11, 12, 13, 14]]], dtype=torch.int32, device=DEV)
    sc = torch.tensor([[[2.0, 1.0, 9.0, 9.0], [1.0, 1.0, 1.0, 1.0]], [[2.0, float("nan"), 9.0, 9.0], [5.0, 4.0, 3.0, 2.0]],
                       [[0.5, 9.0, 9.0, 9.0], [1.0, 0.5, 0.25, 0.1]]], dtype=torch.float32, device=DEV)
    sc[1, 0, 1] = float("nan")
    i, s = dh.merge_topk(idx, sc)
    torch.cuda.synchronize()
    assert i[0].tolist() == [5, 20, 9, 30]
    assert s[0].tolist() == [2.0, 2.0, 1.0, 0.5]
    assert i[1].tolist() == [7, 8, 9, 10]
    idx2 = idx.clone()
    idx2[:, 0, 1:] = -1
    i2, s2 = dh.merge_topk(idx2, sc)
    torch.cuda.synchronize()
    assert i2[0].tolist() == [5, 20, 30, -1] and s2[0, 3].item() == float("-inf")


def test_rescore_shard_owns_only_its_range():
    cfg = inputs.head_config("tiny", B=3, K=16)
    x = inputs.make_head(cfg, seed=70, device=DEV)
    idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    off, n = 1024, 2048
    z, st = dh.exact_rescore_shard(x["h"], x["W"][off:off + n], idx, off)
    ul, _ = dh.exact_rescore(x["h"], x["W"], idx)
    torch.cuda.synchronize()
    own = (idx >= off) & (idx < off + n)
    assert torch.equal(z[own], ul[own])
    assert torch.all(z[~own] == float("-inf"))
    zz = z.double().cpu().numpy()
    for b in range(cfg.B):
        o = own[b].cpu().numpy()
        if o.any():
            m = zz[b][o].max()
            assert st[b, 0].item() == pytest.approx(m)
            assert st[b, 1].item() == pytest.approx(np.exp(zz[b][o] - m).sum(), rel=1e-5)
        else:
            assert st[b, 0].item() == float("-inf") and st[b, 1].item() == 0.0
