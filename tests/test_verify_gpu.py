"""GPU parity of chain verification at positive temperature (dh_verify_chain) against the oracle.

The decisions are taken in fp32 on the GPU and in double in the oracle, so, as for the candidate tie
band of the head, a decision whose uniform lies within 1e-4 (relative) of its threshold may go
either way: the oracle reports the first such decision and the tokens whose cumulative interval
lies within 1e-4 of the total from the sampling point.  Everything else must match exactly: the
number of accepted tokens, and the emitted token within that window (in practice one token).
"""
import numpy as np
import pytest
import scipy.special
import torch

import oracle
from speculative_decoding_draft_dh_gb300 import binding as dh
from speculative_decoding_draft_dh_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
TOL = 1e-4


def run_verify(v, temperature=1.0):
    n, tok = dh.verify_chain(v["logits"], v["cand_idx"], v["cand_prob"], v["draft_token"], v["u_accept"],
                             v["u_sample"], temperature=temperature)
    torch.cuda.synchronize()
    return n.cpu().numpy(), tok.cpu().numpy()


def check_against_oracle(v, temperature=1.0):
    gn, gt = run_verify(v, temperature)
    cpu = {k: t.cpu() for k, t in v.items()}
    o = oracle.verify_chain(cpu["logits"], cpu["cand_idx"], cpu["cand_prob"], cpu["draft_token"], cpu["u_accept"],
                            cpu["u_sample"], temperature=temperature, tol=TOL)
    L = v["logits"].shape[1] - 1
    exact = 0
    for b in range(len(gn)):
        on, fc = int(o["n_accept"][b]), int(o["first_close"][b])
        assert 0 <= gn[b] <= L, f"request {b}: n_accept {gn[b]}"
        if fc > on:  # every decision the oracle took is clear of its threshold
            assert gn[b] == on, f"request {b}: accepted {gn[b]} against {on}"
            assert o["token_lo"][b] <= gt[b] <= o["token_hi"][b], \
                f"request {b}: token {gt[b]} outside [{o['token_lo'][b]}, {o['token_hi'][b]}] (oracle {o['token'][b]})"
            exact += int(gt[b] == o["token"][b])
        else:  # the decisions before the close one are clear
            assert gn[b] >= min(fc, on), f"request {b}: accepted {gn[b]}, clear decisions up to {fc}"
    return gn, gt, o, exact


@pytest.mark.parametrize("T", [1.0, 0.5, 2.0])
@pytest.mark.parametrize("seed", [0, 1])
def test_tiny_verify_matches_oracle(T, seed):
    cfg = inputs.VERIFY_CONFIGS["tiny_verify"]
    v = inputs.make_verify(cfg, seed=seed, device=DEV)
    gn, gt, o, exact = check_against_oracle(v, T)
    assert exact >= cfg.B - 1


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_ragged_segments_and_depths(dtype):
    """A vocabulary that ends inside a segment, depths 1 to 30, K from 1 to 200 (the staged walk up
    to 128 candidates and 2048 entries in all, the general one beyond)."""
    for L, K, vocab in ((1, 1, 1000), (3, 7, 2056), (9, 100, 5000), (5, 200, 4000), (30, 100, 3000)):
        cfg = inputs.verify_config("tiny_verify", B=16, L=L, K=K, vocab=vocab, dtype=dtype)
        v = inputs.make_verify(cfg, seed=L, device=DEV)
        check_against_oracle(v, 1.0)


def test_full_size_every_request():
    cfg = inputs.VERIFY_CONFIGS["verify"]
    v = inputs.make_verify(cfg, seed=0, device=DEV)
    gn, gt, o, exact = check_against_oracle(v)
    assert exact >= cfg.B - 2
    assert 0 < gn.mean() < cfg.L  # both outcomes occur


def test_bonus_only_and_outside_candidates():
    """L = 0 draws the bonus from p_0; a drafted token outside the candidate list is accepted."""
    cfg = inputs.verify_config("tiny_verify", L=0)
    v = inputs.make_verify(cfg, seed=4, device=DEV)
    gn, gt, o, _ = check_against_oracle(v)
    assert np.all(gn == 0)
    cfg = inputs.verify_config("tiny_verify", L=3)
    v = inputs.make_verify(cfg, seed=5, device=DEV)
    v["cand_idx"][:, 0, :] = (v["draft_token"][:, 0:1] + 1) % cfg.vocab  # x_0 never listed: q = 0
    gn, _, _, _ = check_against_oracle(v)
    assert np.all(gn >= 1)


@pytest.mark.parametrize("K", [8, 160])
def test_duplicate_candidates_and_extreme_uniforms(K):
    """Every id listed twice (q adds both), ids outside the vocabulary (no correction), uniforms at
    0 and just below 1; K = 8 takes the staged walk, K = 160 the general one."""
    cfg = inputs.verify_config("tiny_verify", B=16, L=2, K=K)
    v = inputs.make_verify(cfg, seed=6, device=DEV)
    h = K // 2
    v["cand_idx"][:, :, h:2 * h] = v["cand_idx"][:, :, :h]
    v["cand_idx"][:, 1, 0] = -1
    v["cand_idx"][:, 1, 1] = cfg.vocab + 5
    v["u_sample"][:8] = 0.0
    v["u_sample"][8:] = float(np.nextafter(np.float32(1.0), np.float32(0.0)))
    v["u_accept"][:4] = 0.0
    check_against_oracle(v)


def test_repeated_calls_are_identical():
    cfg = inputs.VERIFY_CONFIGS["tiny_verify"]
    v = inputs.make_verify(cfg, seed=9, device=DEV)
    a = run_verify(v)
    b = run_verify(v)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_gpu_preserves_the_target_distribution():
    """The property the correction exists for, on the GPU: over 200000 rounds with fixed target and
    draft distributions, the first emitted token follows p_0 and the bonus follows p_L."""
    n, L, vocab, K = 200000, 2, 64, 6
    rng = np.random.default_rng(11)
    rows = rng.normal(0.0, 1.5, size=(L + 1, vocab)).astype(np.float32)
    cand = np.stack([rng.permutation(vocab)[:K] for _ in range(L)]).astype(np.int32)
    q = rng.dirichlet(np.full(K, 0.7), size=L).astype(np.float32)
    x = np.empty((n, L), dtype=np.int32)
    for i in range(L):
        w = q[i].astype(np.float64) / q[i].astype(np.float64).sum()
        x[:, i] = cand[i][rng.choice(K, size=n, p=w)]
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)  # noqa: E731
    v = {"logits": to(np.broadcast_to(rows, (n, L + 1, vocab))), "cand_idx": to(np.broadcast_to(cand, (n, L, K))),
         "cand_prob": to(np.broadcast_to(q, (n, L, K))), "draft_token": to(x),
         "u_accept": to(rng.random((n, L), dtype=np.float32)), "u_sample": to(rng.random(n, dtype=np.float32))}
    gn, gt = run_verify(v)
    p = scipy.special.softmax(rows.astype(np.float64), axis=-1)
    first = np.where(gn >= 1, x[:, 0], gt)
    for tokens, pr in ((first, p[0]), (gt[gn == L], p[L])):
        f = np.bincount(tokens, minlength=vocab) / len(tokens)
        sigma = np.sqrt(pr * (1 - pr) / len(tokens))
        assert np.all(np.abs(f - pr) <= 5 * sigma + 1e-12)
