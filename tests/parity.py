"""Comparison rules between the CUDA path and the CPU oracle.

Candidate sets (EAGLE-4 summary page, section "Reading correctness marks alongside speed": a
near-tie explanation needs an explicit tolerance): let s_K be the oracle's K-th best low-rank score
of a row; an id is ambiguous when |s_v - s_K| <= 1e-3 |s_K| + 1e-6.  The GPU list must hold every
oracle candidate above that band, nothing below it, and draw the rest from the band.  Its order
must follow its own scores (equal scores -> lower id first) and may only disagree with the
oracle's order between ids whose oracle scores are within the band of each other.

Scores and logits: |g - o| <= 2e-3 + 1e-2 |o| (bf16 inputs, fp32 accumulation).  Probabilities:
|g - o| <= 1e-4.  Tree results: bit-exact.
"""
import numpy as np

BAND_REL, BAND_ABS = 1e-3, 1e-6
LOGIT_ATOL, LOGIT_RTOL = 2e-3, 1e-2
PROB_ATOL = 1e-4


def check_candidates(gidx, gscore, s_row, K, where=""):
    """gidx, gscore: the GPU's K ids and scores for one row; s_row: oracle scores of every id."""
    gidx = np.asarray(gidx, dtype=np.int64)
    gscore = np.asarray(gscore, dtype=np.float64)
    vocab = len(s_row)
    assert gidx.shape == (K,), where
    assert np.all((gidx >= 0) & (gidx < vocab)), f"{where}: id out of range"
    assert len(set(gidx.tolist())) == K, f"{where}: duplicate ids"
    order = np.lexsort((np.arange(vocab), -s_row))
    sK = s_row[order[K - 1]]
    band = BAND_REL * abs(sK) + BAND_ABS
    gs = s_row[gidx]
    assert np.all(gs >= sK - band), f"{where}: id below the tie band: {gidx[gs < sK - band]}"
    must = order[:K][s_row[order[:K]] > sK + band]
    missing = set(must.tolist()) - set(gidx.tolist())
    assert not missing, f"{where}: missing candidates {sorted(missing)[:8]}"
    err = np.abs(gscore - gs)
    assert np.all(err <= LOGIT_ATOL + LOGIT_RTOL * np.abs(gs)), f"{where}: score error {err.max()}"
    # own order: non-increasing scores, equal scores by ascending id
    assert np.all(np.diff(gscore) <= 0), f"{where}: scores not sorted"
    eq = np.diff(gscore) == 0
    assert np.all(np.diff(gidx)[eq] > 0), f"{where}: equal scores not in id order"
    # agreement with the oracle's order outside the band
    for i in range(K - 1):
        later = gs[i + 1:]
        assert np.all(later <= gs[i] + band), f"{where}: order disagrees with the oracle at {i}"
    return int(len(must))


def check_logits(glog, gprob, olog, oprob, where=""):
    glog = np.asarray(glog, dtype=np.float64)
    err = np.abs(glog - olog)
    assert np.all(err <= LOGIT_ATOL + LOGIT_RTOL * np.abs(olog)), f"{where}: logit error {err.max()}"
    if gprob is not None:
        perr = np.abs(np.asarray(gprob, dtype=np.float64) - oprob)
        assert np.all(perr <= PROB_ATOL), f"{where}: probability error {perr.max()}"
