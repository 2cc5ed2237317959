"""The draft head with its vocabulary split over P shards (tensor-parallel serving).

EAGLE-4 summary page, section "Adaptation has not eliminated high-load regressions": the release
serves the target with tensor parallelism over four GPUs; a vocabulary-parallel head keeps each
GPU's share of V and W.  One step (the library does every computation; this module only moves
tensors between shards):

1. each shard: its K best (global id, score) per row (``lowrank_topk_shard``);
2. all-gather of the P lists (8 B K bytes per shard), then ``merge_topk``: the K best of the union,
   bit-identical to the unsharded stage 1;
3. each shard: the logits of the merged candidates it owns and its (max, sum of exp) per row
   (``exact_rescore_shard``);
4. all-gather of those (4 B K + 8 B bytes per shard), then ``combine_softmax``.

``step_on_shards`` runs the P shards one after another on one device (what a single GPU can check);
``step_distributed`` runs this rank's shard and exchanges with ``torch.distributed`` (NCCL between
GPUs, gloo on CPU for the exchange alone).
"""
from __future__ import annotations

import torch

from . import binding as dh


def shard_bounds(vocab: int, P: int, align: int = 8) -> list[tuple[int, int]]:
    """P contiguous (offset, size) ranges covering [0, vocab); sizes are multiples of `align` ids
    (16-byte rows for bf16 when align = 8) except possibly the last."""
    base = (vocab // P) // align * align
    out, off = [], 0
    for p in range(P):
        n = base if p < P - 1 else vocab - off
        out.append((off, n))
        off += n
    return out


def split_weights(V: torch.Tensor, W: torch.Tensor, P: int, align: int = 8):
    """[(offset, V_p contiguous [r, n_p], W_p [n_p, d])] for P shards of the vocabulary."""
    vocab = V.shape[1]
    return [(o, V[:, o:o + n].contiguous(), W[o:o + n]) for o, n in shard_bounds(vocab, P, align)]


def step_on_shards(h, U, shards, K, workspaces=None, stream=None):
    """One head step over P shards on one device.  Returns (idx, score, logits, probs) as
    dh_draft_head does for the whole vocabulary."""
    P = len(shards)
    B = h.shape[0]
    dev = h.device
    ws = workspaces or [dh.Workspace() for _ in range(P)]
    idx_parts = torch.empty(P, B, K, dtype=torch.int32, device=dev)
    score_parts = torch.empty(P, B, K, dtype=torch.float32, device=dev)
    for p, (off, Vp, _) in enumerate(shards):
        dh.lowrank_topk_shard(h, U, Vp, K, off, idx_out=idx_parts[p], score_out=score_parts[p], workspace=ws[p],
                              stream=stream)
    idx, score = dh.merge_topk(idx_parts, score_parts, stream=stream)
    logit_parts = torch.empty(P, B, K, dtype=torch.float32, device=dev)
    stat_parts = torch.empty(P, B, 2, dtype=torch.float32, device=dev)
    for p, (off, _, Wp) in enumerate(shards):
        dh.exact_rescore_shard(h, Wp, idx, off, logits_out=logit_parts[p], stats_out=stat_parts[p], workspace=ws[p],
                               stream=stream)
    logits, probs = dh.combine_softmax(logit_parts, stat_parts, stream=stream)
    return idx, score, logits, probs


def all_gather_parts(x: torch.Tensor, group=None) -> torch.Tensor:
    """[P, *x.shape]: every rank's x, in rank order (the exchange of steps 2 and 4)."""
    import torch.distributed as dist
    P = dist.get_world_size(group)
    out = torch.empty((P,) + tuple(x.shape), dtype=x.dtype, device=x.device)
    if dist.get_backend(group) == "nccl":
        dist.all_gather_into_tensor(out, x.contiguous(), group=group)
    else:
        dist.all_gather(list(out.unbind(0)), x.contiguous(), group=group)
    return out


def step_distributed(h, U, V_shard, W_shard, offset, K, group=None, workspace=None, stream=None):
    """This rank's shard of one head step, exchanging candidates and logits with the other ranks."""
    idx_p, score_p = dh.lowrank_topk_shard(h, U, V_shard, K, offset, workspace=workspace, stream=stream)
    idx, score = dh.merge_topk(all_gather_parts(idx_p, group), all_gather_parts(score_p, group), stream=stream)
    logit_p, stat_p = dh.exact_rescore_shard(h, W_shard, idx, offset, workspace=workspace, stream=stream)
    logits, probs = dh.combine_softmax(all_gather_parts(logit_p, group), all_gather_parts(stat_p, group),
                                       stream=stream)
    return idx, score, logits, probs


def exchanged_bytes_per_step(B: int, K: int, P: int) -> dict:
    """Bytes each rank receives per step: the candidate lists and the logits with their pairs."""
    return {"candidates": 8 * B * K * P, "logits_and_pairs": (4 * B * K + 8 * B) * P}
