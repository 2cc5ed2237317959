"""ctypes binding of libdh (include/dh.h).  Argument marshalling only: every step of the path runs
in the CUDA library.  torch supplies device memory and the current stream.

The library is loaded on first use from this package directory; if it is missing or cannot be
loaded the call raises (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdh.so")

DH_OK = 0
STATUS = {0: "DH_OK", 1: "DH_ERR_INVALID_ARG", 2: "DH_ERR_UNSUPPORTED", 3: "DH_ERR_WORKSPACE",
          4: "DH_ERR_CUDA", 5: "DH_ERR_TIMEOUT", 6: "DH_ERR_BAD_INPUT"}
F32, BF16 = 0, 1

EXPORTS = ["dh_status_string", "dh_version", "dh_last_error", "dh_lowrank_topk_workspace", "dh_lowrank_topk",
           "dh_exact_rescore_workspace", "dh_exact_rescore", "dh_draft_head_workspace", "dh_draft_head",
           "dh_expand_children",
           "dh_tree_accept_workspace",
           "dh_tree_accept", "dh_tree_accept_noalloc", "dh_workspace_status", "dh_selftest_wait_timeout", "dh_prof_enable", "dh_prof_read",
           "dh_set_tuning", "dh_verify_chain_workspace", "dh_verify_chain", "dh_size_level",
           "dh_lowrank_topk_shard", "dh_merge_topk", "dh_exact_rescore_shard_workspace", "dh_exact_rescore_shard",
           "dh_combine_softmax"]

_lib = None
_lock = threading.Lock()


class DhError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        msg = f"{what} failed: {STATUS.get(status, status)}"
        super().__init__(msg + (f" ({detail})" if detail else ""))
        self.status = status


def load_library(path: str | None = None):
    """Load libdh.so and declare the C signatures (raises if the library is missing)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libdh.so not found at {p}: build it with "
                               "`python -m speculative_decoding_draft_dh_gb300.build`")
        lib = ctypes.CDLL(p)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        lib.dh_status_string.argtypes = [I]
        lib.dh_status_string.restype = ctypes.c_char_p
        lib.dh_version.restype = I
        lib.dh_last_error.restype = ctypes.c_char_p
        lib.dh_lowrank_topk_workspace.argtypes = [I, I, I, I, I, I]
        lib.dh_lowrank_topk_workspace.restype = Z
        lib.dh_lowrank_topk.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, Z, P]
        lib.dh_lowrank_topk.restype = I
        lib.dh_exact_rescore_workspace.argtypes = [I, I, I, I, I]
        lib.dh_exact_rescore_workspace.restype = Z
        lib.dh_exact_rescore.argtypes = [P, P, P, I, I, I, I, I, P, P, P, Z, P]
        lib.dh_exact_rescore.restype = I
        lib.dh_draft_head_workspace.argtypes = [I, I, I, I, I, I]
        lib.dh_draft_head_workspace.restype = Z
        lib.dh_draft_head.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P, P, P, P, Z, P]
        lib.dh_draft_head.restype = I
        lib.dh_expand_children.argtypes = [P, P, P, I, I, I, ctypes.c_float, P, P, P, P]
        lib.dh_expand_children.restype = I
        lib.dh_tree_accept_workspace.argtypes = [I, I, I]
        lib.dh_tree_accept_workspace.restype = Z
        lib.dh_tree_accept.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P, Z, P]
        lib.dh_tree_accept.restype = I
        lib.dh_tree_accept_noalloc.argtypes = [P, P, P, I, I, I, I, P, P, P, P, P, P]
        lib.dh_tree_accept_noalloc.restype = I
        lib.dh_workspace_status.argtypes = [P, P, P]
        lib.dh_workspace_status.restype = I
        lib.dh_selftest_wait_timeout.argtypes = [I, I, P, Z, P]
        lib.dh_selftest_wait_timeout.restype = I
        lib.dh_prof_enable.argtypes = [I]
        lib.dh_prof_enable.restype = I
        lib.dh_prof_read.argtypes = [P, I, P, P, I]
        lib.dh_prof_read.restype = I
        lib.dh_verify_chain_workspace.argtypes = [I, I, I, I]
        lib.dh_verify_chain_workspace.restype = Z
        lib.dh_verify_chain.argtypes = [P, P, P, P, P, P, I, I, I, I, I, ctypes.c_float, P, P, P, Z, P]
        lib.dh_verify_chain.restype = I
        lib.dh_size_level.argtypes = [P, P, P, I, I, I, P, P, I, I, I, ctypes.c_float, P, P, P, P, P]
        lib.dh_size_level.restype = I
        lib.dh_lowrank_topk_shard.argtypes = [P, P, P, I, I, I, I, I, I, I, P, P, P, Z, P]
        lib.dh_lowrank_topk_shard.restype = I
        lib.dh_merge_topk.argtypes = [P, P, I, I, I, P, P, P]
        lib.dh_merge_topk.restype = I
        lib.dh_exact_rescore_shard_workspace.argtypes = [I, I, I, I, I]
        lib.dh_exact_rescore_shard_workspace.restype = Z
        lib.dh_exact_rescore_shard.argtypes = [P, P, P, I, I, I, I, I, I, P, P, P, Z, P]
        lib.dh_exact_rescore_shard.restype = I
        lib.dh_combine_softmax.argtypes = [P, P, I, I, I, P, P, P]
        lib.dh_combine_softmax.restype = I
        lib.dh_set_tuning.argtypes = [ctypes.c_char_p, ctypes.c_char_p]
        lib.dh_set_tuning.restype = I
        if path is None:
            _lib = lib
        return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _dev(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Workspace:
    """Zero-initialised device workspaces, grown on demand: one buffer per (device, call kind), so
    one object can serve all three calls.  Calls using the same object must not overlap in time."""

    def __init__(self):
        self.buf = {}

    def get(self, nbytes: int, device, kind: str, stream=None) -> torch.Tensor | None:
        """The buffer for one call kind, at least nbytes long; a new one is zeroed on `stream` (the
        call's stream, else the current one), so that the call that follows finds it zeroed."""
        if nbytes == 0:
            return None
        key = (torch.device(device), kind)
        cur = self.buf.get(key)
        if cur is None or cur.numel() < nbytes:
            with torch.cuda.stream(torch.cuda.current_stream(key[0]) if stream is None else stream):
                cur = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=key[0])
            self.buf[key] = cur
        return cur


_default_ws = Workspace()


def _check(status, what):
    if status != DH_OK:
        detail = ""
        if status == 4 and _lib is not None:
            detail = (_lib.dh_last_error() or b"").decode(errors="replace")
        raise DhError(status, what, detail)


def lowrank_topk(h, U, V, K, *, idx_out=None, score_out=None, workspace=None, stream=None):
    """Stage 1: the K best low-rank scores per row.  Returns (idx int32 [B,K], score fp32 [B,K])."""
    lib = load_library()
    _dev(h, "h"), _dev(U, "U"), _dev(V, "V")
    B, d = h.shape
    r, vocab = V.shape
    dt = _dtype_code(h)
    if U.dtype != h.dtype or V.dtype != h.dtype or U.shape != (d, r):
        raise ValueError("h, U, V must share a dtype and have shapes [B,d], [d,r], [r,vocab]")
    if idx_out is None:
        idx_out = torch.empty(B, K, dtype=torch.int32, device=h.device)
    if score_out is None:
        score_out = torch.empty(B, K, dtype=torch.float32, device=h.device)
    nbytes = lib.dh_lowrank_topk_workspace(B, d, r, vocab, K, dt)
    ws = (workspace or _default_ws).get(nbytes, h.device, "topk", stream)
    _check(lib.dh_lowrank_topk(_ptr(h), _ptr(U), _ptr(V), B, d, r, vocab, K, dt, _ptr(idx_out),
                               _ptr(score_out), _ptr(ws), nbytes, _stream(stream)), "dh_lowrank_topk")
    return idx_out, score_out


def exact_rescore(h, W, idx, *, with_probs=True, logits_out=None, probs_out=None, workspace=None,
                  stream=None):
    """Stage 2: exact logits of the candidates and (optionally) their softmax."""
    lib = load_library()
    _dev(h, "h"), _dev(W, "W"), _dev(idx, "idx")
    B, d = h.shape
    vocab = W.shape[0]
    K = idx.shape[1]
    dt = _dtype_code(h)
    if W.dtype != h.dtype or W.shape[1] != d or idx.dtype != torch.int32 or idx.shape[0] != B:
        raise ValueError("h [B,d], W [vocab,d] share a dtype; idx is int32 [B,K]")
    if logits_out is None:
        logits_out = torch.empty(B, K, dtype=torch.float32, device=h.device)
    if with_probs and probs_out is None:
        probs_out = torch.empty(B, K, dtype=torch.float32, device=h.device)
    nbytes = lib.dh_exact_rescore_workspace(B, d, vocab, K, dt)
    ws = (workspace or _default_ws).get(nbytes, h.device, "rescore", stream)
    _check(lib.dh_exact_rescore(_ptr(h), _ptr(W), _ptr(idx), B, d, vocab, K, dt, _ptr(logits_out),
                                _ptr(probs_out if with_probs else None), _ptr(ws), nbytes,
                                _stream(stream)), "dh_exact_rescore")
    return logits_out, (probs_out if with_probs else None)


def draft_head(h, U, V, W, K, *, with_probs=True, idx_out=None, score_out=None, logits_out=None,
               probs_out=None, workspace=None, stream=None):
    """Both stages in one call (dh_draft_head: the outputs of lowrank_topk followed by
    exact_rescore, with selection and rescoring fused into one cluster kernel for small batches:
    up to 32 rows of 64 candidates on a GB300).  Returns (idx int32 [B,K], score fp32 [B,K],
    logits fp32 [B,K], probs fp32 [B,K] or None)."""
    lib = load_library()
    _dev(h, "h"), _dev(U, "U"), _dev(V, "V"), _dev(W, "W")
    B, d = h.shape
    r, vocab = V.shape
    dt = _dtype_code(h)
    if U.dtype != h.dtype or V.dtype != h.dtype or W.dtype != h.dtype or U.shape != (d, r) \
            or W.shape != (vocab, d):
        raise ValueError("h, U, V, W must share a dtype and have shapes [B,d], [d,r], [r,vocab], [vocab,d]")
    dev = h.device
    if idx_out is None:
        idx_out = torch.empty(B, K, dtype=torch.int32, device=dev)
    if score_out is None:
        score_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    if logits_out is None:
        logits_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    if with_probs and probs_out is None:
        probs_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    nbytes = lib.dh_draft_head_workspace(B, d, r, vocab, K, dt)
    ws = (workspace or _default_ws).get(nbytes, dev, "head", stream)
    _check(lib.dh_draft_head(_ptr(h), _ptr(U), _ptr(V), _ptr(W), B, d, r, vocab, K, dt, _ptr(idx_out),
                             _ptr(score_out), _ptr(logits_out), _ptr(probs_out if with_probs else None),
                             _ptr(ws), nbytes, _stream(stream)), "dh_draft_head")
    return idx_out, score_out, logits_out, (probs_out if with_probs else None)


def expand_children(probs, idx, w, *, parent_prob=None, min_benefit=0.0, child_token=None, child_prob=None,
                    n_keep=None, stream=None):
    """The w children of each frontier node by exact probability.  Returns (child_token int32
    [B,w], child_prob fp32 [B,w], n_keep int32 [B])."""
    lib = load_library()
    _dev(probs, "probs"), _dev(idx, "idx")
    if probs.dtype != torch.float32 or idx.dtype != torch.int32 or probs.shape != idx.shape:
        raise ValueError("probs fp32 [B,K] and idx int32 [B,K]")
    B, K = probs.shape
    dev = probs.device
    if parent_prob is not None:
        _dev(parent_prob, "parent_prob")
        if parent_prob.dtype != torch.float32 or parent_prob.shape != (B,):
            raise ValueError("parent_prob must be fp32 [B]")
    if child_token is None:
        child_token = torch.empty(B, w, dtype=torch.int32, device=dev)
    if child_prob is None:
        child_prob = torch.empty(B, w, dtype=torch.float32, device=dev)
    if n_keep is None:
        n_keep = torch.empty(B, dtype=torch.int32, device=dev)
    _check(lib.dh_expand_children(_ptr(probs), _ptr(idx), _ptr(parent_prob), B, K, w, float(min_benefit),
                                  _ptr(child_token), _ptr(child_prob), _ptr(n_keep), _stream(stream)),
           "dh_expand_children")
    return child_token, child_prob, n_keep


def tree_accept(logits, parent, token, *, with_argmax=True, workspace=None, stream=None):
    """Greedy acceptance over draft trees.  Returns dict(argmax, path, len, bonus, err)."""
    lib = load_library()
    _dev(logits, "logits"), _dev(parent, "parent"), _dev(token, "token")
    B, N, vocab = logits.shape
    dt = _dtype_code(logits)
    if parent.dtype != torch.int32 or token.dtype != torch.int32 or parent.shape != (B, N) \
            or token.shape != (B, N):
        raise ValueError("parent and token must be int32 [B,N]")
    dev = logits.device
    out = {"argmax": torch.empty(B, N, dtype=torch.int32, device=dev) if with_argmax else None,
           "path": torch.empty(B, N, dtype=torch.int32, device=dev),
           "len": torch.empty(B, dtype=torch.int32, device=dev),
           "bonus": torch.empty(B, dtype=torch.int32, device=dev),
           "err": torch.empty(B, dtype=torch.int32, device=dev)}
    nbytes = lib.dh_tree_accept_workspace(B, N, vocab)
    ws = (workspace or _default_ws).get(nbytes, dev, "tree", stream)
    _check(lib.dh_tree_accept(_ptr(logits), _ptr(parent), _ptr(token), B, N, vocab, dt,
                              _ptr(out["argmax"]), _ptr(out["path"]), _ptr(out["len"]),
                              _ptr(out["bonus"]), _ptr(out["err"]), _ptr(ws), nbytes,
                              _stream(stream)), "dh_tree_accept")
    return out


def lowrank_topk_shard(h, U, V_shard, K, vocab_offset, *, idx_out=None, score_out=None, workspace=None,
                       stream=None):
    """Stage 1 on one vocabulary shard (V_shard [r, n] holds the columns vocab_offset .. + n):
    the shard's K best (global id, score) per row."""
    lib = load_library()
    _dev(h, "h"), _dev(U, "U"), _dev(V_shard, "V_shard")
    B, d = h.shape
    r, n = V_shard.shape
    dt = _dtype_code(h)
    if U.dtype != h.dtype or V_shard.dtype != h.dtype or U.shape != (d, r):
        raise ValueError("h, U, V_shard must share a dtype and have shapes [B,d], [d,r], [r,n]")
    if idx_out is None:
        idx_out = torch.empty(B, K, dtype=torch.int32, device=h.device)
    if score_out is None:
        score_out = torch.empty(B, K, dtype=torch.float32, device=h.device)
    nbytes = lib.dh_lowrank_topk_workspace(B, d, r, n, K, dt)
    ws = (workspace or _default_ws).get(nbytes, h.device, "topk", stream)
    _check(lib.dh_lowrank_topk_shard(_ptr(h), _ptr(U), _ptr(V_shard), B, d, r, n, int(vocab_offset), K, dt,
                                     _ptr(idx_out), _ptr(score_out), _ptr(ws), nbytes, _stream(stream)),
           "dh_lowrank_topk_shard")
    return idx_out, score_out


def merge_topk(idx_parts, score_parts, *, idx_out=None, score_out=None, stream=None):
    """The K best of P shard lists per row (dh_merge_topk).  idx_parts int32 / score_parts fp32
    [P, B, K]."""
    lib = load_library()
    _dev(idx_parts, "idx_parts"), _dev(score_parts, "score_parts")
    P, B, K = idx_parts.shape
    if idx_parts.dtype != torch.int32 or score_parts.dtype != torch.float32 or score_parts.shape != (P, B, K):
        raise ValueError("idx_parts int32 and score_parts fp32 [P, B, K]")
    dev = idx_parts.device
    if idx_out is None:
        idx_out = torch.empty(B, K, dtype=torch.int32, device=dev)
    if score_out is None:
        score_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    _check(lib.dh_merge_topk(_ptr(idx_parts), _ptr(score_parts), P, B, K, _ptr(idx_out), _ptr(score_out),
                             _stream(stream)), "dh_merge_topk")
    return idx_out, score_out


def exact_rescore_shard(h, W_shard, idx, vocab_offset, *, logits_out=None, stats_out=None, workspace=None,
                        stream=None):
    """Stage 2 on one shard: logits of the candidates this shard owns (-inf elsewhere) and the row's
    (max, sum of exp) pair [B, 2]."""
    lib = load_library()
    _dev(h, "h"), _dev(W_shard, "W_shard"), _dev(idx, "idx")
    B, d = h.shape
    n = W_shard.shape[0]
    K = idx.shape[1]
    dt = _dtype_code(h)
    if W_shard.dtype != h.dtype or W_shard.shape[1] != d or idx.dtype != torch.int32 or idx.shape[0] != B:
        raise ValueError("h [B,d], W_shard [n,d] share a dtype; idx is int32 [B,K]")
    if logits_out is None:
        logits_out = torch.empty(B, K, dtype=torch.float32, device=h.device)
    if stats_out is None:
        stats_out = torch.empty(B, 2, dtype=torch.float32, device=h.device)
    nbytes = lib.dh_exact_rescore_shard_workspace(B, d, n, K, dt)
    ws = (workspace or _default_ws).get(nbytes, h.device, "rescore_shard", stream)
    _check(lib.dh_exact_rescore_shard(_ptr(h), _ptr(W_shard), _ptr(idx), B, d, n, int(vocab_offset), K, dt,
                                      _ptr(logits_out), _ptr(stats_out), _ptr(ws), nbytes, _stream(stream)),
           "dh_exact_rescore_shard")
    return logits_out, stats_out


def combine_softmax(logits_parts, stats_parts, *, with_probs=True, logits_out=None, probs_out=None, stream=None):
    """Each candidate's logit from its owner shard and the softmax over the K candidates
    (dh_combine_softmax).  logits_parts [P, B, K], stats_parts [P, B, 2] fp32."""
    lib = load_library()
    _dev(logits_parts, "logits_parts"), _dev(stats_parts, "stats_parts")
    P, B, K = logits_parts.shape
    if logits_parts.dtype != torch.float32 or stats_parts.dtype != torch.float32 or stats_parts.shape != (P, B, 2):
        raise ValueError("logits_parts [P, B, K] and stats_parts [P, B, 2], fp32")
    dev = logits_parts.device
    if logits_out is None:
        logits_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    if with_probs and probs_out is None:
        probs_out = torch.empty(B, K, dtype=torch.float32, device=dev)
    _check(lib.dh_combine_softmax(_ptr(logits_parts), _ptr(stats_parts), P, B, K, _ptr(logits_out),
                                  _ptr(probs_out if with_probs else None), _stream(stream)), "dh_combine_softmax")
    return logits_out, (probs_out if with_probs else None)


def size_level(child_prob, child_token, cost, bin_batch, batch, theta, *, n_valid=None, out=None, stream=None):
    """Width and children of the next draft level per request (dh_size_level).  child_prob fp32 /
    child_token int32 [R, F, Wc]; cost fp32 [n_bins, wmax+1] and bin_batch int32 [n_bins] on the
    device.  Returns dict(width int32 [R], parent, token int32 [R, wmax], prob fp32 [R, wmax])."""
    lib = load_library()
    _dev(child_prob, "child_prob"), _dev(child_token, "child_token"), _dev(cost, "cost"), _dev(bin_batch, "bin_batch")
    R, F, Wc = child_prob.shape
    n_bins, w1 = cost.shape
    wmax = w1 - 1
    if child_prob.dtype != torch.float32 or child_token.dtype != torch.int32 or child_token.shape != (R, F, Wc) \
            or cost.dtype != torch.float32 or bin_batch.dtype != torch.int32 or bin_batch.shape != (n_bins,):
        raise ValueError("child_prob fp32 / child_token int32 [R,F,Wc], cost fp32 [n_bins,wmax+1], "
                         "bin_batch int32 [n_bins]")
    if n_valid is not None:
        _dev(n_valid, "n_valid")
    dev = child_prob.device
    if out is None:
        out = {"width": torch.empty(R, dtype=torch.int32, device=dev),
               "parent": torch.empty(R, wmax, dtype=torch.int32, device=dev),
               "token": torch.empty(R, wmax, dtype=torch.int32, device=dev),
               "prob": torch.empty(R, wmax, dtype=torch.float32, device=dev)}
    _check(lib.dh_size_level(_ptr(child_prob), _ptr(child_token), _ptr(n_valid), R, F, Wc, _ptr(cost), _ptr(bin_batch),
                             n_bins, wmax, int(batch), float(theta), _ptr(out["width"]), _ptr(out["parent"]),
                             _ptr(out["token"]), _ptr(out["prob"]), _stream(stream)), "dh_size_level")
    return out


def verify_chain(logits, cand_idx, cand_prob, draft_token, u_accept, u_sample, *, temperature=1.0,
                 n_accept_out=None, token_out=None, workspace=None, stream=None):
    """Speculative sampling over a chain of L drafted tokens per request (dh_verify_chain).
    logits [B, L+1, vocab] (bf16 or fp32); cand_idx int32 / cand_prob fp32 [B, L, K]; draft_token
    int32 / u_accept fp32 [B, L]; u_sample fp32 [B].  Returns (n_accept int32 [B], token int32 [B])."""
    lib = load_library()
    _dev(logits, "logits"), _dev(u_sample, "u_sample")
    B, L1, vocab = logits.shape
    L = L1 - 1
    K = cand_idx.shape[2] if L > 0 else 0
    for t, name, dt in ((cand_idx, "cand_idx", torch.int32), (cand_prob, "cand_prob", torch.float32),
                        (draft_token, "draft_token", torch.int32), (u_accept, "u_accept", torch.float32)):
        if L > 0:
            _dev(t, name)
            if t.dtype != dt:
                raise ValueError(f"{name} must be {dt}")
    if u_sample.dtype != torch.float32 or u_sample.shape != (B,):
        raise ValueError("u_sample must be fp32 [B]")
    dev = logits.device
    if n_accept_out is None:
        n_accept_out = torch.empty(B, dtype=torch.int32, device=dev)
    if token_out is None:
        token_out = torch.empty(B, dtype=torch.int32, device=dev)
    dt = _dtype_code(logits)
    nbytes = lib.dh_verify_chain_workspace(B, L, vocab, dt)
    ws = (workspace or _default_ws).get(nbytes, dev, "verify", stream)
    _check(lib.dh_verify_chain(_ptr(logits), _ptr(cand_idx if L > 0 else None), _ptr(cand_prob if L > 0 else None),
                               _ptr(draft_token if L > 0 else None), _ptr(u_accept if L > 0 else None),
                               _ptr(u_sample), B, L, vocab, K, dt, float(temperature), _ptr(n_accept_out),
                               _ptr(token_out), _ptr(ws), nbytes, _stream(stream)), "dh_verify_chain")
    return n_accept_out, token_out


def workspace_status(workspace: "Workspace | None" = None, device=None, stream=None) -> int:
    """Read and clear the device status words of a workspace object (OR over its buffers)."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    status = 0
    for (d, _kind), ws in (workspace or _default_ws).buf.items():
        if d != dev:
            continue
        out = ctypes.c_int(0)
        _check(lib.dh_workspace_status(_ptr(ws), _stream(stream), ctypes.byref(out)), "dh_workspace_status")
        status |= out.value
    return status


def selftest_wait_timeout(limit_us: int = 50000, stream=None) -> int:
    """Run the bounded-wait self-test (an mbarrier wait that nothing completes) on a fresh workspace
    and return the status word it left (expected: 1 << DH_ERR_TIMEOUT)."""
    lib = load_library()
    with torch.cuda.stream(torch.cuda.current_stream() if stream is None else stream):
        ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _check(lib.dh_selftest_wait_timeout(0, limit_us, _ptr(ws), 256, _stream(stream)),
           "dh_selftest_wait_timeout")
    out = ctypes.c_int(0)
    _check(lib.dh_workspace_status(_ptr(ws), _stream(stream), ctypes.byref(out)), "dh_workspace_status")
    return out.value


def set_tuning(name: str, value: str | None):
    """Set one test or tuning switch (kernel choice only; None restores the default)."""
    lib = load_library()
    _check(lib.dh_set_tuning(name.encode(), None if value is None else str(value).encode()), "dh_set_tuning")


def prof_enable(on: bool):
    load_library().dh_prof_enable(1 if on else 0)


def prof_read(max_kernels: int = 64) -> dict:
    """{kernel name: (total ms, launches)} recorded since the last read (waits for the events)."""
    lib = load_library()
    L = 64
    names = ctypes.create_string_buffer(L * max_kernels)
    tot = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int * max_kernels)()
    n = lib.dh_prof_read(names, L, tot, cnt, max_kernels)
    if n < 0:
        raise DhError(4, "dh_prof_read")
    out = {}
    for k in range(min(n, max_kernels)):
        nm = names.raw[k * L:(k + 1) * L].split(b"\0", 1)[0].decode()
        out[nm] = (tot[k], cnt[k])
    return out
