"""Seeded synthetic inputs for the two-stage draft LM head and greedy tree acceptance.

This module only draws random tensors with the shapes and distributions of the workloads; it holds
none of the method's arithmetic (no projection, scoring, selection, softmax or tree logic), so both
the CUDA path and the CPU oracle can consume what it produces.

Workloads (sizes are the benchmark's, since the EAGLE-4 pages give no drafter dimensions):

* ``tiny``      B<=4, d=256, vocab=4096, r=32, K=16, fp32, noise 0.05, h ~ N(0,1)
* ``batch1``    B=1,   d=5120, vocab=151936, r=128, K=64,  bf16, noise 0.1
* ``moderate``  B=64,  d=5120, vocab=151936, r=256, K=128, bf16, noise 0.1
* ``high``      B=512, d=5120, vocab=151936, r=512, K=256, bf16, noise 0.1

U ~ N(0, std 1/sqrt(d)) [d x r], V ~ N(0, std 1/sqrt(r)) [r x vocab], the full-rank head
W = (U V)^T + noise * N(0, std 1/sqrt(d)) [vocab x d], all built in fp32 and then cast to the
workload dtype independently.  For the bf16 workloads h is scaled by 3/sqrt(1+noise^2) so that the
exact logits have standard deviation about 3.

Trees: node 0 is the root; node n picks its parent uniformly among earlier nodes that are below the
depth limit and have fewer children than the branching limit (no limits: uniform over [0, n)).
Draft tokens are uniform over the vocabulary.  Target logits are N(0, std^2); each non-root node is
"marked" with probability ``match``, and for every parent the lowest-index marked child gets its
token's logit set to rowmax + 2, a strict row maximum (after rounding to the dtype), so the target
agrees with that draft edge.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np
import torch


@dataclass(frozen=True)
class HeadConfig:
    name: str
    B: int
    d: int
    vocab: int
    r: int
    K: int
    dtype: str  # "f32" or "bf16"
    noise: float
    scale_h: bool

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


@dataclass(frozen=True)
class TreeConfig:
    name: str
    B: int
    N: int
    vocab: int
    dtype: str
    logit_std: float
    max_depth: int | None
    max_children: int | None
    match: float = 0.7
    boost: float = 2.0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


HEAD_CONFIGS = {
    "tiny": HeadConfig("tiny", 4, 256, 4096, 32, 16, "f32", 0.05, False),
    "batch1": HeadConfig("batch1", 1, 5120, 151936, 128, 64, "bf16", 0.1, True),
    "moderate": HeadConfig("moderate", 64, 5120, 151936, 256, 128, "bf16", 0.1, True),
    "high": HeadConfig("high", 512, 5120, 151936, 512, 256, "bf16", 0.1, True),
    # one draft level: eight frontier nodes through the head, then four children each
    "level": HeadConfig("level", 8, 5120, 151936, 128, 64, "bf16", 0.1, True),
}

TREE_CONFIGS = {
    "tiny_tree": TreeConfig("tiny_tree", 4, 8, 4096, "f32", 1.0, None, None),
    "tree": TreeConfig("tree", 256, 64, 151936, "bf16", 3.0, 10, 4),
}


@dataclass(frozen=True)
class VerifyConfig:
    """Chain verification at positive temperature: B requests, each with L drafted tokens (the
    round's depth, fixed before the round), target logits for the L+1 positions, and the draft's
    distribution at each drafted position given as K candidate ids with their probabilities."""
    name: str
    B: int
    L: int
    vocab: int
    K: int
    dtype: str
    logit_std: float = 3.0
    match: float = 0.7
    boost: float = 2.0
    temperature: float = 1.0

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16


VERIFY_CONFIGS = {
    "tiny_verify": VerifyConfig("tiny_verify", 8, 4, 4096, 16, "f32", 1.0),
    "verify": VerifyConfig("verify", 64, 7, 151936, 64, "bf16"),
}


def head_config(name: str, **overrides) -> HeadConfig:
    return replace(HEAD_CONFIGS[name], **overrides)


def tree_config(name: str, **overrides) -> TreeConfig:
    return replace(TREE_CONFIGS[name], **overrides)


def verify_config(name: str, **overrides) -> VerifyConfig:
    return replace(VERIFY_CONFIGS[name], **overrides)


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_head(cfg: HeadConfig, seed: int = 0, device="cpu", chunk_rows: int = 8192,
              with_W: bool = True) -> dict:
    """Draw h [B x d], U [d x r], V [r x vocab] and W [vocab x d] in the workload dtype.

    Everything is drawn from one generator in a fixed order (U, V, h, then the noise of W in row
    chunks), so a seed fixes the tensors on a given device.
    """
    dev = torch.device(device)
    g = _gen(dev, seed)
    f32 = torch.float32
    U = torch.randn(cfg.d, cfg.r, generator=g, device=dev, dtype=f32) / math.sqrt(cfg.d)
    V = torch.randn(cfg.r, cfg.vocab, generator=g, device=dev, dtype=f32) / math.sqrt(cfg.r)
    h = torch.randn(cfg.B, cfg.d, generator=g, device=dev, dtype=f32)
    if cfg.scale_h:
        h = h * (3.0 / math.sqrt(1.0 + cfg.noise * cfg.noise))
    out = {"h": h.to(cfg.torch_dtype).contiguous(), "U": U.to(cfg.torch_dtype).contiguous(),
           "V": V.to(cfg.torch_dtype).contiguous()}
    if with_W:
        W = torch.empty(cfg.vocab, cfg.d, device=dev, dtype=cfg.torch_dtype)
        Ut = U.t().contiguous()
        prev = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = False
        try:
            for v0 in range(0, cfg.vocab, chunk_rows):
                v1 = min(cfg.vocab, v0 + chunk_rows)
                blk = V[:, v0:v1].t() @ Ut
                if cfg.noise:
                    noise = torch.randn(v1 - v0, cfg.d, generator=g, device=dev, dtype=f32)
                    blk = blk + noise * (cfg.noise / math.sqrt(cfg.d))
                W[v0:v1] = blk.to(cfg.torch_dtype)
        finally:
            torch.backends.cuda.matmul.allow_tf32 = prev
        out["W"] = W
    return out


def make_h(cfg: HeadConfig, seed: int, device="cpu") -> torch.Tensor:
    """A fresh hidden-state batch drawn like ``make_head``'s h (used for per-step inputs)."""
    dev = torch.device(device)
    g = _gen(dev, seed)
    h = torch.randn(cfg.B, cfg.d, generator=g, device=dev, dtype=torch.float32)
    if cfg.scale_h:
        h = h * (3.0 / math.sqrt(1.0 + cfg.noise * cfg.noise))
    return h.to(cfg.torch_dtype).contiguous()


def make_parents(B: int, N: int, seed: int, max_depth=None, max_children=None) -> np.ndarray:
    """Random parent arrays [B x N] (int32, parent[:,0] = -1, 0 <= parent[n] < n)."""
    rng = np.random.default_rng(seed)
    parent = np.full((B, N), -1, dtype=np.int32)
    for b in range(B):
        depth = [0]
        nchild = [0]
        for n in range(1, N):
            elig = [p for p in range(n)
                    if (max_depth is None or depth[p] < max_depth)
                    and (max_children is None or nchild[p] < max_children)]
            p = elig[int(rng.integers(len(elig)))]
            parent[b, n] = p
            depth.append(depth[p] + 1)
            nchild.append(0)
            nchild[p] += 1
    return parent


def make_tree(cfg: TreeConfig, seed: int = 0, device="cpu") -> dict:
    """Draw parent [B x N] int32, token [B x N] int32 and target logits [B x N x vocab]."""
    dev = torch.device(device)
    parent = make_parents(cfg.B, cfg.N, seed, cfg.max_depth, cfg.max_children)
    rng = np.random.default_rng(seed + 1)
    token = rng.integers(0, cfg.vocab, size=(cfg.B, cfg.N), dtype=np.int64).astype(np.int32)
    marked = rng.random((cfg.B, cfg.N)) < cfg.match
    marked[:, 0] = False
    g = _gen(dev, seed)
    logits = torch.empty(cfg.B, cfg.N, cfg.vocab, device=dev, dtype=cfg.torch_dtype)
    for b in range(cfg.B):
        blk = torch.randn(cfg.N, cfg.vocab, generator=g, device=dev, dtype=torch.float32)
        logits[b] = (blk * cfg.logit_std).to(cfg.torch_dtype)
    # boost: per parent, the lowest-index marked child
    bs, ps, ts = [], [], []
    for b in range(cfg.B):
        seen = set()
        for c in range(1, cfg.N):
            p = int(parent[b, c])
            if marked[b, c] and p not in seen:
                seen.add(p)
                bs.append(b); ps.append(p); ts.append(int(token[b, c]))
    for s in range(0, len(bs), 1024):
        bi = torch.tensor(bs[s:s + 1024], device=dev)
        pi = torch.tensor(ps[s:s + 1024], device=dev)
        ti = torch.tensor(ts[s:s + 1024], device=dev)
        rowmax = logits[bi, pi].float().amax(dim=-1)
        logits[bi, pi, ti] = (rowmax + cfg.boost).to(cfg.torch_dtype)
    return {"logits": logits, "parent": torch.from_numpy(parent).to(dev),
            "token": torch.from_numpy(token).to(dev)}


def _distinct_ids(rng, vocab: int, k: int) -> np.ndarray:
    """k distinct ids, uniform over [0, vocab), in the order first drawn."""
    out, seen = [], set()
    while len(out) < k:
        for v in rng.integers(0, vocab, size=2 * k).tolist():
            if v not in seen:
                seen.add(v)
                out.append(v)
                if len(out) == k:
                    break
    return np.asarray(out, dtype=np.int32)


def make_verify(cfg: VerifyConfig, seed: int = 0, device="cpu") -> dict:
    """Draw the inputs of chain verification.

    cand_idx int32 [B, L, K] (distinct ids per position), cand_prob fp32 [B, L, K] (a Dirichlet(0.5)
    draw per position), draft_token int32 [B, L] (drawn from that distribution), the uniforms
    u_accept fp32 [B, L] and u_sample fp32 [B] in [0, 1), and target logits [B, L+1, vocab] ~
    N(0, logit_std^2) in the workload dtype; at a fraction ``match`` of the drafted positions the
    drafted token's target logit is set to rowmax + boost, so that the target often agrees.
    """
    dev = torch.device(device)
    rng = np.random.default_rng(seed)
    B, L, K = cfg.B, cfg.L, cfg.K
    cand = np.stack([_distinct_ids(rng, cfg.vocab, K) for _ in range(B * L)]).reshape(B, L, K) if L else \
        np.zeros((B, 0, K), dtype=np.int32)
    q64 = rng.dirichlet(np.full(K, 0.5), size=(B, L)) if L else np.zeros((B, 0, K))
    q = q64.astype(np.float32)
    draft = np.zeros((B, L), dtype=np.int32)
    for b in range(B):
        for i in range(L):
            w = q64[b, i] / q64[b, i].sum()
            draft[b, i] = cand[b, i, int(rng.choice(K, p=w))]
    u_accept = rng.random((B, L), dtype=np.float32)
    u_sample = rng.random(B, dtype=np.float32)
    marked = rng.random((B, L)) < cfg.match
    g = _gen(dev, seed)
    logits = torch.empty(B, L + 1, cfg.vocab, device=dev, dtype=cfg.torch_dtype)
    for b in range(B):
        blk = torch.randn(L + 1, cfg.vocab, generator=g, device=dev, dtype=torch.float32)
        logits[b] = (blk * cfg.logit_std).to(cfg.torch_dtype)
    bs, is_, ts = [], [], []
    for b in range(B):
        for i in range(L):
            if marked[b, i]:
                bs.append(b); is_.append(i); ts.append(int(draft[b, i]))
    if bs:
        bi = torch.tensor(bs, device=dev)
        ii = torch.tensor(is_, device=dev)
        ti = torch.tensor(ts, device=dev)
        rowmax = logits[bi, ii].float().amax(dim=-1)
        logits[bi, ii, ti] = (rowmax + cfg.boost).to(cfg.torch_dtype)
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    return {"logits": logits, "cand_idx": to(cand), "cand_prob": to(q), "draft_token": to(draft),
            "u_accept": to(u_accept), "u_sample": to(u_sample)}


# Synthetic latency table for sizing a draft level (the pages' tables come from engine profiling,
# which is out of scope): bins of batch size and, per bin, the latency in microseconds of a draft
# level of w nodes and its verification, base + slope x w for w >= 1 and 0 for w = 0.  Heavier
# loads cost more per node, so they favour narrower, shallower trees.
SIZING_BINS = (1, 8, 64, 512)
SIZING_BASE_US = (30.0, 35.0, 50.0, 120.0)
SIZING_SLOPE_US = (1.0, 2.5, 12.0, 80.0)


def latency_table(wmax: int) -> tuple:
    """(cost fp32 [len(SIZING_BINS), wmax + 1], bin_batch int32 [len(SIZING_BINS)])."""
    cost = np.zeros((len(SIZING_BINS), wmax + 1), dtype=np.float32)
    for i, (b0, s0) in enumerate(zip(SIZING_BASE_US, SIZING_SLOPE_US)):
        cost[i, 1:] = [b0 + s0 * w for w in range(1, wmax + 1)]
    return cost, np.asarray(SIZING_BINS, dtype=np.int32)


def make_frontier_children(R: int, F: int, Wc: int, seed: int = 0, vocab: int = 151936) -> dict:
    """Candidate children of R requests' frontiers of F nodes, Wc children each, as an expansion
    would leave them: per node a path probability (uniform in [0.05, 1)) times Dirichlet(0.3)
    child probabilities in descending order; tokens uniform; n_valid = Wc."""
    rng = np.random.default_rng(seed)
    par = rng.uniform(0.05, 1.0, size=(R, F, 1))
    kid = -np.sort(-rng.dirichlet(np.full(max(Wc, 2), 0.3), size=(R, F))[..., :Wc], axis=-1)
    prob = (par * kid).astype(np.float32)
    token = rng.integers(0, vocab, size=(R, F, Wc)).astype(np.int32)
    return {"child_prob": prob, "child_token": token, "n_valid": np.full((R, F), Wc, dtype=np.int32)}
