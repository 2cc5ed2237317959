"""Multi-rank host logic on CPU with gloo (world size 2).

* bench.py's replica mode: barrier, max-over-ranks timing and the weak-scaling aggregate.
* The vocabulary-parallel merge rule of the sharded head design: each rank takes a contiguous
  vocabulary shard, finds its shard's top-K (here with the CPU oracle, ids offset to global ids),
  the ranks all-gather their K (score, id) pairs, and the K best of the union in (score desc, id asc)
  order equal the unsharded top-K.  Any global top-K member is in its own shard's top-K, so the
  union always contains the answer.
* Tree acceptance with vocabulary-sharded target logits: each rank packs its shard's per-node
  maximum as (order-preserving value key << 32 | ~global id) into a 64-bit integer, one all-reduce
  MAX gives the global argmax with ties to the lowest id, and the walk on the merged argmax equals
  the unsharded acceptance.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    _init(rank, world, port)
    try:
        bench.barrier(world)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slowest
        slowest = bench.max_over_ranks(ms, world)
        value = bench.weak_scaling_value(64, 100, world, slowest)
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def _shard_worker(rank, world, port, q):
    """One rank of the vocabulary-sharded head on the CPU: its shard's candidates and owned logits
    from the oracle, exchanged with the package's own all-gather (sharded.all_gather_parts, gloo),
    merged and combined here as the library's merge and softmax kernels do."""
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from speculative_decoding_draft_dh_gb300 import inputs, sharded
    _init(rank, world, port)
    try:
        cfg = inputs.head_config("tiny", B=3, K=16)
        x = inputs.make_head(cfg, seed=21)
        lo, n = sharded.shard_bounds(cfg.vocab, world, align=4)[rank]
        idx, sc = oracle.lowrank_topk(x["h"], x["U"], x["V"][:, lo:lo + n].contiguous(), cfg.K)
        ids = torch.from_numpy((idx + lo).astype(np.int32))
        scores = torch.from_numpy(sc.astype(np.float32))
        all_ids = sharded.all_gather_parts(ids).numpy()        # [P, B, K]
        all_sc = sharded.all_gather_parts(scores).numpy()
        merged = []
        for b in range(cfg.B):
            s_, i_ = all_sc[:, b].ravel(), all_ids[:, b].ravel().astype(np.int64)
            merged.append(i_[np.lexsort((i_, -s_))[: cfg.K]])
        merged = np.stack(merged).astype(np.int32)
        # owner-only logits, the shard's (max, sum of exp), exchanged and combined
        z, _ = oracle.exact_rescore(x["h"], x["W"], merged)
        own = (merged >= lo) & (merged < lo + n)
        zl = np.where(own, z, -np.inf)
        m = zl.max(axis=1)
        ssum = np.where(np.isfinite(m), np.exp(zl - np.where(np.isfinite(m), m, 0)[:, None]).sum(axis=1), 0.0)
        parts_z = sharded.all_gather_parts(torch.from_numpy(zl)).numpy()
        parts_st = sharded.all_gather_parts(torch.from_numpy(np.stack([m, ssum], axis=1))).numpy()
        logits = parts_z.max(axis=0)
        M = parts_st[:, :, 0].max(axis=0)
        S = sum(np.where(np.isfinite(parts_st[p, :, 0]), parts_st[p, :, 1] * np.exp(parts_st[p, :, 0] - M), 0.0)
                for p in range(world))
        probs = np.exp(logits - M[:, None]) / S[:, None]
        q.put((rank, merged, logits, probs))
    finally:
        dist.destroy_process_group()


def _packed_max(vals, lo):
    """(value key << 32 | ~global id) per row of vals [rows, n] (fp32); the row maximum."""
    bits = vals.astype(np.float32).view(np.uint32).astype(np.uint64)
    neg = (bits >> np.uint64(31)) == 1
    key = np.where(neg, (~bits) & np.uint64(0xFFFFFFFF), bits | np.uint64(0x80000000))
    ids = np.arange(vals.shape[1], dtype=np.uint64) + np.uint64(lo)
    packed = (key << np.uint64(32)) | ((~ids) & np.uint64(0xFFFFFFFF))
    return packed.max(axis=1)


def _tree_shard_worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    from speculative_decoding_draft_dh_gb300 import inputs
    _init(rank, world, port)
    try:
        tcfg = inputs.tree_config("tiny_tree")
        t = inputs.make_tree(tcfg, seed=5)
        L = t["logits"].float().numpy()
        B, N, vocab = L.shape
        lo, hi = vocab * rank // world, vocab * (rank + 1) // world
        local = _packed_max(L[:, :, lo:hi].reshape(B * N, hi - lo), lo)
        # the packed keys fit a signed int64 only after flipping the top bit (order preserving)
        ten = torch.from_numpy((local ^ np.uint64(1 << 63)).view(np.int64).copy())
        dist.all_reduce(ten, op=dist.ReduceOp.MAX)
        merged = ten.numpy().view(np.uint64) ^ np.uint64(1 << 63)
        argmax = (~(merged & np.uint64(0xFFFFFFFF)) & np.uint64(0xFFFFFFFF)).astype(np.int64).reshape(B, N)
        q.put((rank, argmax))
    finally:
        dist.destroy_process_group()


def _run(worker, world=2):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return sorted(out, key=lambda t: t[0])


def test_bench_spawns_one_rank_per_requested_gpu():
    """bench.py --gpus 2 without a launcher starts two ranks itself; with --dry-run they meet over
    gloo on the CPU, and rank 0 reports both ranks and the world size."""
    import json
    import subprocess
    import sys
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_PORT")}
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--dry-run"],
                         capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = lines[0]
    assert line["n_gpus"] == 2 and line["gpus_requested"] == 2
    assert sorted(r["rank"] for r in line["ranks"]) == [0, 1]
    assert line["ms_slowest"] == pytest.approx(max(r["ms"] for r in line["ranks"]))


def test_replicas_take_the_slowest_rank_and_scale_weakly():
    out = _run(_bench_worker)
    for rank, slowest, value in out:
        assert slowest == 15.0
        assert value == pytest.approx(64 * 100 * 2 / 0.015)


@pytest.mark.parametrize("world", [2, 3])
def test_vocab_sharded_step_equals_unsharded(world):
    """The sharded head's exchange path (all-gather of the candidate lists, merge; all-gather of
    owned logits and (max, sum) pairs, combination) gives the unsharded oracle's candidates,
    logits and probabilities on every rank."""
    import oracle
    from speculative_decoding_draft_dh_gb300 import inputs
    out = _run(_shard_worker, world=world)
    cfg = inputs.head_config("tiny", B=3, K=16)
    x = inputs.make_head(cfg, seed=21)
    idx, _ = oracle.lowrank_topk(x["h"], x["U"], x["V"], cfg.K)
    z, p = oracle.exact_rescore(x["h"], x["W"], idx)
    for _, merged, logits, probs in out:
        np.testing.assert_array_equal(merged, idx)
        np.testing.assert_array_equal(logits, z)
        np.testing.assert_allclose(probs, p, rtol=1e-12, atol=1e-15)


def test_vocab_sharded_tree_argmax_equals_unsharded():
    import oracle
    from speculative_decoding_draft_dh_gb300 import inputs
    out = _run(_tree_shard_worker)
    tcfg = inputs.tree_config("tiny_tree")
    t = inputs.make_tree(tcfg, seed=5)
    ref = oracle.tree_accept(t["logits"], t["parent"], t["token"])
    for _, argmax in out:
        np.testing.assert_array_equal(argmax, ref["argmax"])
