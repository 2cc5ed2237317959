"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle on the same seeded
inputs.  Small shapes are compared row by row in full; the full-size workloads are compared on
sampled rows that the oracle computes one by one, plus properties checked on every row."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_draft_dh_gb300 import binding as dh
from speculative_decoding_draft_dh_gb300 import inputs
from tests.parity import check_candidates, check_logits
from tests import test_oracle_pins as pins
from tests.test_oracle_pins import golden_tree_arrays, load_golden_trees

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_draft_dh_gb300 import build
    build.build()
    dh.load_library()
    yield
    torch.cuda.synchronize()


def run_head(x, K, rows=None, api="split"):
    """GPU stage 1 + stage 2 on device tensors (the two calls, or dh_draft_head with api="head");
    oracle on the listed rows.  Returns the GPU outputs."""
    h, U, V, W = x["h"], x["U"], x["V"], x["W"]
    if api == "head":
        idx, score, logits, probs = dh.draft_head(h, U, V, W, K)
    else:
        idx, score = dh.lowrank_topk(h, U, V, K)
        logits, probs = dh.exact_rescore(h, W, idx)
    torch.cuda.synchronize()
    B = h.shape[0]
    rows = list(range(B)) if rows is None else rows
    hc, Uc, Vc = h.cpu(), U.cpu(), V.cpu()
    s_full = oracle.lowrank_scores(hc, Uc, Vc, rows=rows)
    gi, gs = idx.cpu().numpy(), score.cpu().numpy()
    for n, b in enumerate(rows):
        check_candidates(gi[b], gs[b], s_full[n], K, where=f"row {b}")
    # stage 2 on the same ids: the oracle rescoring the GPU's own candidates
    Wc = W.cpu()
    oz, op = oracle.exact_rescore(hc, Wc, idx.cpu(), rows=rows)
    gl, gp = logits.cpu().numpy(), probs.cpu().numpy()
    for n, b in enumerate(rows):
        check_logits(gl[b], gp[b], oz[n], op[n], where=f"row {b}")
    # properties on every row
    assert np.all((gi >= 0) & (gi < V.shape[1]))
    assert np.all(np.diff(gs, axis=1) <= 0)
    np.testing.assert_allclose(gp.sum(axis=1), 1.0, atol=1e-4)
    return idx, score, logits, probs


# ---------------------------------------------------------------- small shapes, every row

@pytest.mark.parametrize("api", ["split", "head"])
@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_tiny_head(B, api):
    cfg = inputs.head_config("tiny", B=B)
    x = inputs.make_head(cfg, seed=0, device=DEV)
    run_head(x, cfg.K, api=api)


MID = inputs.HeadConfig("mid_bf16", 5, 512, 8200, 64, 32, "bf16", 0.1, True)  # ragged vocab tail


@pytest.mark.parametrize("api", ["split", "head"])
@pytest.mark.parametrize("seed", [0, 1])
def test_mid_bf16_ragged_vocab(seed, api):
    x = inputs.make_head(MID, seed=seed, device=DEV)
    run_head(x, MID.K, api=api)


@pytest.mark.parametrize("K", [1, 2, 3, 7, 16, 17, 33, 64, 65, 100, 128, 129, 1000, 1024])
@pytest.mark.parametrize("api", ["split", "head"])
def test_tiny_head_K_range(K, api):
    """K across the selection's sort regimes and every cluster shape of the small-batch rescore
    (1 to 8 CTAs of 2, 4, 8 or 16 warps), then the ticket kernel above K = 128; with api="head"
    the fused cluster kernel up to K = 256 and the two-call path above."""
    cfg = inputs.head_config("tiny", B=2, K=K)
    x = inputs.make_head(cfg, seed=3, device=DEV)
    run_head(x, K, api=api)


def test_K_equals_vocab_uses_exact_fallback():
    cfg = inputs.HeadConfig("k_eq_vocab", 2, 256, 1024, 32, 1024, "f32", 0.05, False)
    x = inputs.make_head(cfg, seed=4, device=DEV)
    idx, _, _, probs = run_head(x, cfg.K)
    assert sorted(idx[0].cpu().tolist()) == list(range(1024))


def _best_column(x):
    s = oracle.lowrank_scores(x["h"][:1].cpu(), x["U"].cpu(), x["V"].cpu())[0]
    return int(np.argmax(s))


@pytest.mark.parametrize("api", ["split", "head"])
def test_clustered_candidates_are_refined(api):
    """All top candidates inside one group of 64 ids: the group's third score reaches the
    candidate threshold and the group is re-scored exactly."""
    cfg = inputs.head_config("tiny", B=1, K=16)
    x = inputs.make_head(cfg, seed=5, device=DEV)
    v = _best_column(x)
    base = x["V"][:, v].clone()
    for j in range(64):
        x["V"][:, 128 + j] = base * (1.0 + 0.01 * j)
    run_head(x, cfg.K, api=api)


@pytest.mark.parametrize("select", ["auto", "radix"])
@pytest.mark.parametrize("B", [1, 8])
def test_tensor_core_path_fused_head_refines_clustered_rows(B, select, tune):
    """Tensor-core stage 1 (t in bf16, and the groups' best keys) followed by the fused cluster
    head, on rows whose top candidates crowd one group (refinement by the leader's block selection)
    and on plain rows: against the oracle, and bit for bit against the two calls; with the fast
    selection (auto) and the cooperative radix one."""
    tune("DH_FORCE_PATH", "mma")
    tune("DH_HEAD_SELECT", select)
    cfg = inputs.head_config("batch1", B=B, d=512, vocab=8192, r=64, K=32)
    x = inputs.make_head(cfg, seed=8, device=DEV)
    v = _best_column(x)
    base = x["V"][:, v].clone()
    for j in range(64):
        x["V"][:, 128 + j] = base * (1.0 + 0.01 * j)
    idx, score, logits, probs = run_head(x, cfg.K, api="head")
    i2, s2 = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    l2, p2 = dh.exact_rescore(x["h"], x["W"], i2)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2)
    assert torch.equal(logits, l2) and torch.equal(probs, p2)


@pytest.mark.parametrize("B,K,seed", [(3, 84, 1), (1, 256, 0), (2, 256, 1), (2, 192, 1), (8, 128, 2)])
def test_fused_head_refines_flagged_rows_in_place(B, K, seed, tune):
    """Rows whose certificate flags a group (a third score at or above tau; common from K = 128 on
    random rows) are refined inside the fused head, every CTA re-ranking the winners with the
    flagged groups scored exactly: bit for bit the two calls' outputs, and the oracle's top K."""
    tune("DH_FORCE_HEAD", "cluster")
    cfg = inputs.head_config("batch1", B=B, K=K)
    x = inputs.make_head(cfg, seed=seed, device=DEV)
    idx, score, logits, probs = run_head(x, K, api="head")
    i2, s2 = dh.lowrank_topk(x["h"], x["U"], x["V"], K)
    l2, p2 = dh.exact_rescore(x["h"], x["W"], i2)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2)
    assert torch.equal(logits, l2) and torch.equal(probs, p2)


@pytest.mark.parametrize("api", ["split", "head"])
def test_many_clustered_groups_use_full_rescan(api):
    cfg = inputs.head_config("tiny", B=1, K=128)
    x = inputs.make_head(cfg, seed=6, device=DEV)
    v = _best_column(x)
    base = x["V"][:, v].clone()
    for g in range(40):
        for q in range(3):
            x["V"][:, 64 * g + q] = base * (2.0 + 0.001 * (3 * g + q))
    run_head(x, cfg.K, api=api)


@pytest.mark.parametrize("path", ["auto", "mma"])
def test_fast_selection_overflow_takes_the_exact_path(path, tune):
    """Every group's two best scores tie with the K-th group best (identical V columns), so far more
    than the candidate list's capacity reach the threshold: the fused head falls back to the
    leader's exact selection, and still equals the two calls and the oracle (ties to the lowest id).
    After the small-batch scores kernel (auto) and after the tensor-core one."""
    if path != "auto":
        tune("DH_FORCE_PATH", path)
    cfg = inputs.head_config("batch1", B=1, d=512, vocab=65536, r=128, K=64)
    x = inputs.make_head(cfg, seed=9, device=DEV)
    x["V"][:, 1:] = x["V"][:, :1]
    idx, score, logits, probs = run_head(x, cfg.K, api="head")
    i2, s2 = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    l2, p2 = dh.exact_rescore(x["h"], x["W"], i2)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2)
    assert torch.equal(logits, l2) and torch.equal(probs, p2)
    assert idx[0].tolist() == list(range(cfg.K))


@pytest.mark.parametrize("api", ["split", "head"])
def test_equal_scores_resolve_to_lowest_id(api):
    cfg = inputs.head_config("tiny", B=1, K=16)
    x = inputs.make_head(cfg, seed=7, device=DEV)
    v = _best_column(x)
    col = x["V"][:, v].clone() * 3.0
    for c in (4000, 17, 2222, 640):
        x["V"][:, c] = col
    idx, score, _, _ = run_head(x, cfg.K, api=api)
    assert idx[0, :4].cpu().tolist() == [17, 640, 2222, 4000]
    assert len(set(score[0, :4].cpu().tolist())) == 1


def test_empty_batch_is_a_noop():
    cfg = inputs.head_config("tiny", B=1)
    x = inputs.make_head(cfg, seed=0, device=DEV)
    h0 = x["h"][:0]
    idx, score = dh.lowrank_topk(h0, x["U"], x["V"], cfg.K)
    assert idx.shape == (0, cfg.K)
    logits, probs = dh.exact_rescore(h0, x["W"], idx)
    assert logits.shape == (0, cfg.K)


def test_rescore_bad_index_gives_nan_row():
    cfg = inputs.head_config("tiny", B=3)
    x = inputs.make_head(cfg, seed=0, device=DEV)
    idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    idx[1, 5] = cfg.vocab + 10
    idx[2, 0] = -1
    logits, probs = dh.exact_rescore(x["h"], x["W"], idx)
    lg, pr = logits.cpu().numpy(), probs.cpu().numpy()
    assert np.isnan(lg[1, 5]) and np.isnan(lg[2, 0])
    assert np.isnan(pr[1]).all() and np.isnan(pr[2]).all()
    assert np.isfinite(lg[0]).all() and np.isfinite(pr[0]).all()


@pytest.mark.parametrize("path", ["direct", "ring", "ticket", "sweep", "bucket"])
def test_rescore_paths_small_shapes(path, tune):
    """Each stage-2 kernel (direct = the cluster kernel for K <= 128) on fp32 and bf16 rows, K not a
    multiple of the ring's chunk nor of the cluster's warps."""
    tune("DH_FORCE_RESCORE", path)
    for cfg in (inputs.head_config("tiny", B=3, K=45), inputs.HeadConfig("r", 5, 768, 4096, 64, 70, "bf16", 0.1, True)):
        x = inputs.make_head(cfg, seed=17, device=DEV)
        idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
        logits, probs = dh.exact_rescore(x["h"], x["W"], idx)
        torch.cuda.synchronize()
        oz, op = oracle.exact_rescore(x["h"].cpu(), x["W"].cpu(), idx.cpu())
        for b in range(cfg.B):
            check_logits(logits[b].cpu().numpy(), probs[b].cpu().numpy(), oz[b], op[b], where=f"{cfg.name} row {b}")
    assert dh.workspace_status() == 0


def test_rescore_paths_agree_bit_for_bit(tune):
    """Every stage-2 kernel gives the same logits and probabilities bit for bit: one dot-product
    order and one softmax order, whatever the kernel (cluster, ticket, bucketed ring, sweep); on
    rows whose candidates spread over the vocabulary and on rows that all fall in one bucket."""
    cfgs = (inputs.head_config("tiny", B=3, K=45), inputs.HeadConfig("r", 5, 768, 4096, 64, 70, "bf16", 0.1, True),
            inputs.HeadConfig("rr", 40, 512, 4096, 64, 256, "bf16", 0.1, True))
    for cfg in cfgs:
        x = inputs.make_head(cfg, seed=23, device=DEV)
        idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
        idx_lo = torch.sort(idx % 700, dim=1).values.contiguous()  # every row's ids in the lowest bucket
        for ids in (idx, idx_lo):
            outs = {}
            for path in ("direct", "ring", "ticket", "sweep", "bucket"):
                tune("DH_FORCE_RESCORE", path)
                outs[path] = dh.exact_rescore(x["h"], x["W"], ids)
            torch.cuda.synchronize()
            lg0, pr0 = outs["direct"]
            for path, (lg, pr) in outs.items():
                assert torch.equal(lg, lg0), (cfg.name, path)
                assert torch.equal(pr, pr0), (cfg.name, path)
    assert dh.workspace_status() == 0


def test_rescore_without_probs():
    cfg = inputs.head_config("tiny", B=2)
    x = inputs.make_head(cfg, seed=0, device=DEV)
    idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    logits, probs = dh.exact_rescore(x["h"], x["W"], idx, with_probs=False)
    assert probs is None
    oz, _ = oracle.exact_rescore(x["h"].cpu(), x["W"].cpu(), idx.cpu())
    check_logits(logits.cpu().numpy(), None, oz, None)


# ---------------------------------------------------------------- full-size workloads

@pytest.mark.parametrize("api", ["split", "head"])
def test_batch1_full_size(api):
    cfg = inputs.HEAD_CONFIGS["batch1"]
    x = inputs.make_head(cfg, seed=0, device=DEV)
    run_head(x, cfg.K, api=api)


@pytest.mark.parametrize("mode", ["auto", "cluster8", "split", "radix"])
@pytest.mark.parametrize("name,B", [("batch1", 1), ("batch1", 3), ("batch1", 8), ("tiny", 4), ("moderate", 64),
                                    ("high", 512)])
def test_draft_head_matches_the_two_calls(name, B, mode, tune):
    """dh_draft_head gives bit-identical outputs to dh_lowrank_topk + dh_exact_rescore: the same
    selection rule on the same records and the same per-candidate dot product order; twice in a
    row with one workspace (its state resets itself).  "auto" takes the fused cluster kernel
    (selection and rescoring in one launch) where the batch is small enough, "cluster8" the same
    with 8-CTA clusters, "split" the two kernels, "radix" the cooperative radix selection in the
    cluster kernel."""
    if mode == "cluster8":
        tune("DH_HEAD_CTAS", "8")
    elif mode == "radix":
        tune("DH_HEAD_SELECT", "radix")
    elif mode != "auto":
        tune("DH_FORCE_HEAD", mode)
    cfg = inputs.head_config(name, B=B)
    x = inputs.make_head(cfg, seed=11, device=DEV)
    h, U, V, W = x["h"], x["U"], x["V"], x["W"]
    idx, score = dh.lowrank_topk(h, U, V, cfg.K)
    logits, probs = dh.exact_rescore(h, W, idx)
    ws = dh.Workspace()
    for _ in range(2):
        i2, s2, l2, p2 = dh.draft_head(h, U, V, W, cfg.K, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(i2, idx)
        assert torch.equal(s2, score)
        assert torch.equal(l2, logits)
        assert torch.equal(p2, probs)
    assert dh.workspace_status(ws) == 0


@pytest.mark.parametrize("select", ["auto", "radix"])
@pytest.mark.parametrize("ctas", ["auto", "8", "4", "2"])
@pytest.mark.parametrize("K", [1, 7, 64, 100, 128, 256])
def test_fused_head_matches_the_two_calls_over_K(K, ctas, select, tune):
    """The fused small-batch head against the two calls, bit for bit, over K (up to a full warp
    of candidates per CTA, and beyond one candidate per warp), with 16-CTA clusters where they fit
    and with 8, 4 and 2; with the group-best threshold selection (auto) and the cooperative radix one."""
    tune("DH_FORCE_HEAD", "cluster")
    tune("DH_HEAD_SELECT", select)
    if ctas != "auto":
        tune("DH_HEAD_CTAS", ctas)
    cfg = inputs.head_config("tiny", B=3, K=K)
    x = inputs.make_head(cfg, seed=21, device=DEV)
    h, U, V, W = x["h"], x["U"], x["V"], x["W"]
    idx, score = dh.lowrank_topk(h, U, V, K)
    logits, probs = dh.exact_rescore(h, W, idx)
    i2, s2, l2, p2 = dh.draft_head(h, U, V, W, K)
    torch.cuda.synchronize()
    assert torch.equal(i2, idx) and torch.equal(s2, score)
    assert torch.equal(l2, logits) and torch.equal(p2, probs)


@pytest.mark.parametrize("B", [1, 2, 3])
def test_fused_head_back_to_back_calls(B):
    """Calls queued back to back on one stream with one workspace and no host synchronisation in
    between (each call's kernels start, by programmatic dependent launch, while the previous ones
    finish, and the workspace state resets itself): every call equals the two calls on its own
    inputs, bit for bit."""
    cfg = inputs.head_config("batch1", B=B)
    base = inputs.make_head(cfg, seed=31, device=DEV)
    U, V, W = base["U"], base["V"], base["W"]
    g = torch.Generator(device="cpu").manual_seed(32)
    hs = [(torch.randn(B, cfg.d, generator=g) * base["h"].float().std().item()).to(base["h"].dtype).to(DEV)
          for _ in range(12)]
    ws = dh.Workspace()
    outs = [dh.draft_head(h, U, V, W, cfg.K, workspace=ws) for h in hs]
    torch.cuda.synchronize()
    for h, (i2, s2, l2, p2) in zip(hs, outs):
        idx, score = dh.lowrank_topk(h, U, V, cfg.K)
        logits, probs = dh.exact_rescore(h, W, idx)
        torch.cuda.synchronize()
        assert torch.equal(i2, idx) and torch.equal(s2, score)
        assert torch.equal(l2, logits) and torch.equal(p2, probs)
    assert dh.workspace_status(ws) == 0


@pytest.mark.parametrize("B,K,full", [(16, 64, False), (32, 64, False), (33, 128, True), (64, 64, True)])
def test_fused_head_small_clusters(B, K, full):
    """Batches of 16 and 32 rows of 64 candidates, and 33 rows of 128 at the full shape (the
    four-CTA clusters where eight- and sixteen-CTA ones do not fit one wave; 4224 pairs), and 64
    rows of 64 at the full shape (two-CTA clusters): against
    the oracle on every row (on five rows at the full shape), logits bit for bit against the two
    calls (same per-candidate dot product order); probabilities to rounding."""
    cfg = (inputs.head_config("batch1", B=B, K=K) if full
           else inputs.head_config("batch1", B=B, d=512, vocab=8192, r=64, K=K))
    x = inputs.make_head(cfg, seed=9, device=DEV)
    idx, score, logits, probs = run_head(x, cfg.K, api="head", rows=[0, 1, B // 2, B - 2, B - 1] if full else None)
    i2, s2 = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    l2, p2 = dh.exact_rescore(x["h"], x["W"], i2)
    torch.cuda.synchronize()
    assert torch.equal(idx, i2) and torch.equal(score, s2) and torch.equal(logits, l2)
    torch.testing.assert_close(probs, p2, rtol=0, atol=1e-6)


def test_draft_head_without_probs_and_bad_rows():
    cfg = inputs.head_config("tiny", B=3)
    x = inputs.make_head(cfg, seed=12, device=DEV)
    i2, s2, l2, p2 = dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K, with_probs=False)
    torch.cuda.synchronize()
    assert p2 is None
    oz, _ = oracle.exact_rescore(x["h"].cpu(), x["W"].cpu(), i2.cpu())
    for b in range(cfg.B):
        check_logits(l2[b].cpu().numpy(), None, oz[b], None, where=f"row {b}")


@pytest.mark.parametrize("api", ["split", "head"])
def test_moderate_load_every_row(api):
    cfg = inputs.HEAD_CONFIGS["moderate"]
    x = inputs.make_head(cfg, seed=0, device=DEV)
    run_head(x, cfg.K, api=api)


# 64 rows of the 512: in each of the four 128-row tiles of the tensor-core stage 1, in each of
# the four 32-row lane quarters of its accumulator, the first and last row of each half
HIGH_ROWS = [t * 128 + q * 32 + o for t in range(4) for q in range(4) for o in (0, 15, 16, 31)]


@pytest.mark.parametrize("api", ["split", "head"])
def test_high_load_stratified_rows(api):
    cfg = inputs.HEAD_CONFIGS["high"]
    x = inputs.make_head(cfg, seed=0, device=DEV)
    run_head(x, cfg.K, rows=HIGH_ROWS, api=api)


# ---------------------------------------------------------------- trees

def run_tree(t, reqs=None):
    out = dh.tree_accept(t["logits"], t["parent"], t["token"])
    torch.cuda.synchronize()
    B = t["parent"].shape[0]
    reqs = list(range(B)) if reqs is None else reqs
    sel = torch.tensor(reqs)
    o = oracle.tree_accept(t["logits"][sel.to(t["logits"].device)].cpu(), t["parent"][sel.to(DEV)].cpu(),
                           t["token"][sel.to(DEV)].cpu())
    g = {k: v.cpu().numpy() for k, v in out.items()}
    np.testing.assert_array_equal(g["argmax"][reqs], o["argmax"])
    np.testing.assert_array_equal(g["path"][reqs], o["path"])
    np.testing.assert_array_equal(g["len"][reqs], o["len"])
    np.testing.assert_array_equal(g["bonus"][reqs], o["bonus"])
    # properties on every request
    par = t["parent"].cpu().numpy()
    for b in range(B):
        L = g["len"][b]
        assert g["err"][b] == 0 and L >= 0
        p = g["path"][b]
        assert p[0] == 0 and np.all(p[L + 1:] == -1)
        for j in range(1, L + 1):
            assert par[b, p[j]] == p[j - 1]
        assert g["bonus"][b] == g["argmax"][b, p[L]]
    return g


def test_tiny_trees():
    t = inputs.make_tree(inputs.TREE_CONFIGS["tiny_tree"], seed=0, device=DEV)
    run_tree(t)


@pytest.mark.parametrize("case", load_golden_trees(), ids=lambda c: c["name"])
def test_golden_trees_on_gpu(case):
    logits, parent, token = golden_tree_arrays(case)
    # pad the vocabulary to a multiple of 4 fp32 values (16 bytes); padding never wins the argmax
    out = dh.tree_accept(torch.from_numpy(logits).to(DEV), torch.from_numpy(parent).to(DEV),
                         torch.from_numpy(token).to(DEV))
    torch.cuda.synchronize()
    N = parent.shape[1]
    assert out["len"][0].item() == case["expect_len"][0]
    assert out["bonus"][0].item() == case["expect_bonus"][0]
    want = case["expect_path"] + [-1] * (N - len(case["expect_path"]))
    assert out["path"][0].cpu().tolist() == want
    assert out["err"][0].item() == (6 if case["expect_len"][0] < 0 else 0)


def test_tree_bf16_ties_and_single_node():
    tcfg = inputs.tree_config("tree", B=3, N=1, vocab=4096)
    t = inputs.make_tree(tcfg, seed=2, device=DEV)
    t["logits"][1, 0, :] = 0.5  # all equal: argmax is id 0
    g = run_tree(t)
    assert g["argmax"][1, 0] == 0 and g["len"].tolist() == [0, 0, 0]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tree_argmax_nan_rows(dtype):
    """NaN ranks below every number (a row of NaN only gives id 0), as in the oracle."""
    tcfg = inputs.tree_config("tree", B=2, N=8, vocab=4104, dtype=dtype)
    t = inputs.make_tree(tcfg, seed=5, device=DEV)
    L = t["logits"]
    nan = float("nan")
    L[0, 0, :64] = nan                # NaN vectors first in every thread's scan
    L[0, 1, :] = nan                  # NaN only
    L[0, 2, 1::2] = nan               # NaN in every vector
    L[0, 3, :] = float("-inf")
    L[0, 3, 7::11] = nan              # -inf numbers beat NaN
    L[1, 4, 4096:] = nan              # NaN in the ragged tail
    L[1, 5, :] = nan                  # one number left, in the tail
    L[1, 5, 4101] = -3.0
    g = run_tree(t)
    assert g["argmax"][0, 1] == 0 and g["argmax"][0, 3] == 0 and g["argmax"][1, 5] == 4101


def test_tree_full_size_every_request():
    t = inputs.make_tree(inputs.TREE_CONFIGS["tree"], seed=0, device=DEV)
    g = run_tree(t)
    assert g["len"].mean() > 0.5


# ---------------------------------------------------------------- both stage-1 paths on each shape

MMA_SHAPES = [
    inputs.HeadConfig("mma_r64", 5, 512, 8200, 64, 32, "bf16", 0.1, True),      # ragged vocab tail
    inputs.HeadConfig("mma_r128_b1", 1, 1024, 16384, 128, 64, "bf16", 0.1, True),
    inputs.HeadConfig("mma_two_mtiles", 130, 512, 4096, 128, 16, "bf16", 0.1, True),  # 2 row tiles
    inputs.HeadConfig("mma_r512", 40, 512, 6144, 512, 256, "bf16", 0.1, True),   # deepest K loop
    inputs.HeadConfig("mma_r192", 20, 768, 4096, 192, 32, "bf16", 0.1, True),    # 192-wide projection tile
]


@pytest.mark.parametrize("cfg", MMA_SHAPES, ids=lambda c: c.name)
@pytest.mark.parametrize("path", ["mma", "gemv", "fused"])
def test_forced_stage1_path(cfg, path, tune):
    tune("DH_FORCE_PATH", path)
    x = inputs.make_head(cfg, seed=11, device=DEV)
    rows = list(range(cfg.B)) if cfg.B <= 8 else [0, 1, cfg.B // 2, cfg.B - 1]
    run_head(x, cfg.K, rows=rows)
    assert dh.workspace_status() == 0


@pytest.mark.parametrize("B", [1, 4, 8])
@pytest.mark.parametrize("path", ["gemv", "fused"])
def test_small_batch_paths_fp32(B, path, tune):
    tune("DH_FORCE_PATH", path)
    cfg = inputs.head_config("tiny", B=B, K=32)
    x = inputs.make_head(cfg, seed=20 + B, device=DEV)
    run_head(x, cfg.K)
    assert dh.workspace_status() == 0


@pytest.mark.parametrize("scale", [1e-4, 1e4])
@pytest.mark.parametrize("B", [1, 3])
def test_small_batch_projection_scaled_h(scale, B, tune):
    """The small-batch projection's fixed-point sum (32 fraction bits) against the oracle with h far
    from its usual scale: small values keep their relative precision, large ones stay in range."""
    tune("DH_FORCE_PATH", "fused")
    cfg = inputs.head_config("batch1", B=B, vocab=16384)
    x = inputs.make_head(cfg, seed=3, device=DEV)
    x["h"] = (x["h"].float() * scale).to(torch.bfloat16)
    ws = dh.Workspace()
    idx, score = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, workspace=ws)
    torch.cuda.synchronize()
    assert dh.workspace_status(ws) == 0
    s_full = oracle.lowrank_scores(x["h"].cpu(), x["U"].cpu(), x["V"].cpu())
    for b in range(B):
        check_candidates(idx[b].cpu().numpy(), score[b].cpu().numpy(), s_full[b], cfg.K, where=f"scale {scale} row {b}")


def test_small_batch_projection_overflow_is_reported(tune):
    """A projection beyond the fixed-point range (|t| >= 2^31) raises DH_ERR_UNSUPPORTED in the
    workspace status word instead of passing silently."""
    tune("DH_FORCE_PATH", "fused")
    cfg = inputs.head_config("batch1", vocab=16384)
    x = inputs.make_head(cfg, seed=3, device=DEV)
    x["h"] = (x["h"].float() * 1e12).to(torch.bfloat16)
    ws = dh.Workspace()
    dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, workspace=ws)
    torch.cuda.synchronize()
    assert dh.workspace_status(ws) & (1 << 2)
    # the workspace stays usable: a call at the usual scale is exact again
    x2 = inputs.make_head(cfg, seed=4, device=DEV)
    idx, score = dh.lowrank_topk(x2["h"], x2["U"], x2["V"], cfg.K, workspace=ws)
    torch.cuda.synchronize()
    assert dh.workspace_status(ws) == 0
    s_full = oracle.lowrank_scores(x2["h"].cpu(), x2["U"].cpu(), x2["V"].cpu())
    check_candidates(idx[0].cpu().numpy(), score[0].cpu().numpy(), s_full[0], cfg.K, where="after overflow")


def test_batch1_forced_gemv(tune):
    tune("DH_FORCE_PATH", "gemv")
    cfg = inputs.HEAD_CONFIGS["batch1"]
    x = inputs.make_head(cfg, seed=2, device=DEV)
    run_head(x, cfg.K)


@pytest.mark.parametrize("path", ["fused", "auto"])
def test_fused_path_batch8_bf16_full_vocab(path, tune):
    """Eight rows at full size: the small-batch pipeline (forced) and the automatic choice (the
    tensor-core path from five rows on)."""
    if path == "fused":
        tune("DH_FORCE_PATH", "fused")
    cfg = inputs.HeadConfig("b8", 8, 5120, 151936, 256, 64, "bf16", 0.1, True)
    x = inputs.make_head(cfg, seed=3, device=DEV)
    run_head(x, cfg.K, rows=[0, 7])
    assert dh.workspace_status() == 0


def test_moderate_load_forced_gemv(tune):
    tune("DH_FORCE_PATH", "gemv")
    cfg = inputs.HEAD_CONFIGS["moderate"]
    x = inputs.make_head(cfg, seed=1, device=DEV)
    run_head(x, cfg.K, rows=[3, 60])


def test_mma_and_gemv_paths_agree_on_candidates(tune):
    cfg = inputs.HeadConfig("agree", 24, 512, 16384, 128, 64, "bf16", 0.1, True)
    x = inputs.make_head(cfg, seed=12, device=DEV)
    tune("DH_FORCE_PATH", "mma")
    i1, s1 = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    tune("DH_FORCE_PATH", "gemv")
    i2, s2 = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    torch.cuda.synchronize()
    # the paths round t from different fp32 summation orders, so near-equal scores may swap places;
    # positionwise scores still agree within the documented score tolerance
    same = (i1 == i2).float().mean().item()
    assert same > 0.95
    np.testing.assert_allclose(s1.cpu().numpy(), s2.cpu().numpy(), rtol=1e-2, atol=2e-3)


def test_one_workspace_across_shapes():
    """Calls of different shapes and paths sharing one workspace object: state that must be zero
    between calls may not be left where another shape keeps its data."""
    ws = dh.Workspace()
    shapes = [inputs.head_config("tiny", B=4, K=16), inputs.head_config("tiny", B=1, K=1),
              inputs.head_config("tiny", B=3, K=64), MID, inputs.head_config("tiny", B=2, K=7),
              inputs.HeadConfig("wide", 20, 512, 4096, 128, 32, "bf16", 0.1, True), inputs.head_config("tiny", B=1, K=5)]
    for n, cfg in enumerate(shapes):
        x = inputs.make_head(cfg, seed=40 + n, device=DEV)
        idx, score = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K, workspace=ws)
        logits, probs = dh.exact_rescore(x["h"], x["W"], idx, workspace=ws)
        torch.cuda.synchronize()
        s_full = oracle.lowrank_scores(x["h"].cpu(), x["U"].cpu(), x["V"].cpu())
        oz, op = oracle.exact_rescore(x["h"].cpu(), x["W"].cpu(), idx.cpu())
        for b in range(cfg.B):
            check_candidates(idx[b].cpu().numpy(), score[b].cpu().numpy(), s_full[b], cfg.K, where=f"{cfg.name} row {b}")
            check_logits(logits[b].cpu().numpy(), probs[b].cpu().numpy(), oz[b], op[b], where=f"{cfg.name} row {b}")
    assert dh.workspace_status(ws) == 0


def test_draft_head_one_workspace_across_shapes():
    """dh_draft_head calls of different shapes sharing one workspace: the rescoring's per-row tickets
    sit after stage 1's layout, which depends on the shape, so a larger call leaves its records where
    a smaller call keeps its tickets; the smaller call must still give the two calls' outputs."""
    ws = dh.Workspace()
    big = inputs.head_config("moderate", B=64, K=128)
    x = inputs.make_head(big, seed=3, device=DEV)
    dh.draft_head(x["h"], x["U"], x["V"], x["W"], big.K, workspace=ws)
    del x
    for cfg in (inputs.HeadConfig("ring_small", 40, 512, 4096, 64, 64, "bf16", 0.1, True),
                inputs.HeadConfig("ticket_small", 24, 512, 4096, 64, 160, "bf16", 0.1, True)):
        y = inputs.make_head(cfg, seed=4, device=DEV)
        i2, s2, l2, p2 = dh.draft_head(y["h"], y["U"], y["V"], y["W"], cfg.K, workspace=ws)
        idx, score = dh.lowrank_topk(y["h"], y["U"], y["V"], cfg.K)
        logits, probs = dh.exact_rescore(y["h"], y["W"], idx)
        torch.cuda.synchronize()
        assert torch.equal(i2, idx) and torch.equal(s2, score), cfg.name
        assert torch.equal(l2, logits) and torch.equal(p2, probs), cfg.name
    assert dh.workspace_status(ws) == 0


def test_fresh_workspace_on_a_side_stream():
    """A call on a stream other than the current one, with a fresh workspace (zeroed on the call's
    stream) while the current stream is still busy: it equals the same call on the current stream
    and leaves no status bit."""
    cfg = inputs.head_config("batch1", B=2)
    x = inputs.make_head(cfg, seed=5, device=DEV)
    ref = dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K, workspace=dh.Workspace())
    torch.cuda.synchronize()
    nbytes = dh.load_library().dh_draft_head_workspace(cfg.B, cfg.d, cfg.r, cfg.vocab, cfg.K, dh._dtype_code(x["h"]))
    junk = torch.full((nbytes + 4096,), 255, dtype=torch.uint8, device=DEV)
    del junk  # its block is free again, with ones in it
    a = torch.randn(2048, 2048, device=DEV)
    for _ in range(20):  # keeps the current stream busy
        a = torch.tanh(a @ a)
    side = torch.cuda.Stream()
    ws = dh.Workspace()
    out = dh.draft_head(x["h"], x["U"], x["V"], x["W"], cfg.K, workspace=ws, stream=side)
    torch.cuda.synchronize()
    for o, r_ in zip(out, ref):
        assert torch.equal(o, r_)
    assert dh.workspace_status(ws) == 0


def test_repeated_calls_are_identical():
    cfg = inputs.head_config("tiny", B=4)
    x = inputs.make_head(cfg, seed=13, device=DEV)
    outs = []
    for _ in range(3):
        idx, score = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
        logits, probs = dh.exact_rescore(x["h"], x["W"], idx)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (idx, score, logits, probs)])
    for o in outs[1:]:
        for a, b in zip(outs[0], o):
            assert torch.equal(a, b)
    assert dh.workspace_status() == 0


# ---------------------------------------------------------------- bounded waits

def test_bounded_waits_time_out_and_leave_the_context_usable():
    status = dh.selftest_wait_timeout(limit_us=20000)
    assert status == (1 << 5)
    cfg = inputs.head_config("tiny", B=2)
    x = inputs.make_head(cfg, seed=0, device=DEV)
    run_head(x, cfg.K)


@pytest.mark.parametrize("path", ["direct", "ring", "ticket", "sweep", "bucket"])
def test_rescore_large_batch_with_repeats(path, tune):
    """Stage 2 on a large batch whose rows draw from a small candidate pool (many repeated W rows),
    with two out-of-range ids; a second call reuses the workspace tickets."""
    tune("DH_FORCE_RESCORE", path)
    cfg = inputs.HeadConfig("rescore_big", 256, 512, 4096, 64, 128, "bf16", 0.1, True)
    x = inputs.make_head(cfg, seed=31, device=DEV)
    g = torch.Generator(device="cpu").manual_seed(5)
    idx = torch.randint(0, 600, (cfg.B, cfg.K), generator=g, dtype=torch.int32)
    idx[3, 7] = cfg.vocab + 1
    idx[200, 0] = -5
    idx = idx.to(DEV)
    logits, probs = dh.exact_rescore(x["h"], x["W"], idx)
    torch.cuda.synchronize()
    rows = [0, 3, 100, 200, 255]
    oz, op = oracle.exact_rescore(x["h"].cpu(), x["W"].cpu(), idx.cpu(), rows=rows)
    gl, gp = logits.cpu().numpy(), probs.cpu().numpy()
    for n, b in enumerate(rows):
        if b in (3, 200):
            ib = idx[b].cpu().numpy()
            ok = (ib >= 0) & (ib < cfg.vocab)
            assert np.isnan(gl[b][~ok]).all() and np.isnan(gp[b]).all()
            check_logits(gl[b][ok], None, oz[n][ok], None, where=f"row {b}")
        else:
            check_logits(gl[b], gp[b], oz[n], op[n], where=f"row {b}")
    logits2, probs2 = dh.exact_rescore(x["h"], x["W"], idx)
    torch.cuda.synchronize()
    assert torch.equal(torch.nan_to_num(logits2), torch.nan_to_num(logits))
    assert torch.equal(torch.nan_to_num(probs2), torch.nan_to_num(probs))


def test_sweep_matches_ring_at_high_load(tune):
    """The vocabulary-sweep rescoring (the default from two rows per SM) against the bulk-copy ring on
    the high-load candidates: the same dot products, so bit-identical logits; the softmax sums in
    another order, so probabilities agree to rounding."""
    cfg = inputs.HEAD_CONFIGS["high"]
    x = inputs.make_head(cfg, seed=2, device=DEV)
    idx, _ = dh.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    tune("DH_FORCE_RESCORE", "sweep")
    l1, p1 = dh.exact_rescore(x["h"], x["W"], idx)
    tune("DH_FORCE_RESCORE", "ring")
    l2, p2 = dh.exact_rescore(x["h"], x["W"], idx)
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)
    np.testing.assert_allclose(p1.cpu().numpy(), p2.cpu().numpy(), atol=1e-7, rtol=1e-5)
    assert dh.workspace_status() == 0


# ---------------------------------------------------------------- expanding frontier nodes

@pytest.mark.parametrize("case", pins.load_golden_expansions(), ids=lambda c: c["name"])
def test_expand_golden_on_gpu(case):
    tok, cp, keep = dh.expand_children(torch.tensor([case["probs"]], dtype=torch.float32, device=DEV),
                                       torch.tensor([case["tokens"]], dtype=torch.int32, device=DEV), case["w"],
                                       parent_prob=torch.tensor([case["parent"]], dtype=torch.float32, device=DEV),
                                       min_benefit=case["min_benefit"])
    torch.cuda.synchronize()
    assert tok[0].cpu().tolist() == case["expect_tokens"]
    np.testing.assert_array_equal(cp[0].cpu().numpy(), np.array(case["expect_probs"], dtype=np.float32))
    assert int(keep[0]) == case["expect_keep"]


@pytest.mark.parametrize("K,w", [(1, 1), (17, 4), (64, 1), (64, 4), (64, 64), (256, 8), (1024, 32)])
def test_expand_matches_oracle(K, w):
    """Random probabilities with exact ties, a NaN row and repeated tokens: bit-exact against the
    oracle (tokens, fp32 path probabilities, kept counts)."""
    rng = np.random.default_rng(K * 7 + w)
    B = 9
    p = rng.dirichlet(np.ones(K), size=B).astype(np.float32)
    if K > 3:
        p[:, 1] = p[:, 3]
        p[4, : K // 2] = p[4, 0]
    p[6, K // 2] = np.nan
    tok = rng.integers(0, 151936, size=(B, K)).astype(np.int32)
    tok[5, :] = 42  # one token repeated: positions decide
    par = rng.uniform(0.05, 1.0, size=B).astype(np.float32)
    thr = float(np.float32(0.3 / K))
    et, ep, ek = oracle.expand_children(p, tok, w, parent_prob=par, min_benefit=thr)
    gt, gp, gk = dh.expand_children(torch.from_numpy(p).to(DEV), torch.from_numpy(tok).to(DEV), w,
                                    parent_prob=torch.from_numpy(par).to(DEV), min_benefit=thr)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(gt.cpu().numpy(), et)
    np.testing.assert_array_equal(gp.cpu().numpy(), ep)
    np.testing.assert_array_equal(gk.cpu().numpy(), ek)


def test_draft_level_step_matches_oracle():
    """One draft level: the head's candidates and probabilities for every frontier node, then their
    children; the expansion checked against the oracle on the GPU's own probabilities, the head as
    in the other parity tests."""
    cfg = inputs.head_config("tiny", B=4, K=16)
    x = inputs.make_head(cfg, seed=33, device=DEV)
    idx, score, logits, probs = run_head(x, cfg.K, api="head")
    par = torch.tensor([1.0, 0.5, 0.25, 0.125], dtype=torch.float32, device=DEV)
    tok, cp, keep = dh.expand_children(probs, idx, 4, parent_prob=par, min_benefit=0.01)
    torch.cuda.synchronize()
    et, ep, ek = oracle.expand_children(probs.cpu().numpy(), idx.cpu().numpy(), 4,
                                        parent_prob=par.cpu().numpy(), min_benefit=0.01)
    np.testing.assert_array_equal(tok.cpu().numpy(), et)
    np.testing.assert_array_equal(cp.cpu().numpy(), ep)
    np.testing.assert_array_equal(keep.cpu().numpy(), ek)
