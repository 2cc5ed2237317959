"""CPU oracle for the draft-head path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import this package.  The product library never loads it, and it shares no code with the CUDA
path.  ``build()`` compiles ``dh_oracle.cpp`` with g++ (OpenMP, no fp contraction) into
``liboracle.so`` next to it; the wrappers below take numpy arrays / CPU torch tensors.

Parity unpinned: the bf16 stage-1 scores of the full-size workloads are checked only through this
oracle's own pins on smaller shapes (brute force, closed forms, hand-built trees).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dh_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile the oracle shared library (idempotent)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
               _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def bind(path: str):
    """Load an oracle shared library from ``path`` and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_round_bf16.argtypes = [P, I, P]
    lib.oracle_lowrank_project.argtypes = [P, P, I, I, I, I, P, I, P]
    lib.oracle_lowrank_scores.argtypes = [P, P, P, I, I, I, I, I, P, I, P]
    lib.oracle_lowrank_topk.argtypes = [P, P, P, I, I, I, I, I, I, P, I, P, P]
    lib.oracle_exact_rescore.argtypes = [P, P, P, I, I, I, I, I, P, I, P, P]
    lib.oracle_tree_accept.argtypes = [P, P, P, I, I, I, I, P, I, P, P, P, P]
    lib.oracle_expand_children.argtypes = [P, P, P, I, I, I, ctypes.c_float, P, P, P]
    D = ctypes.c_double
    lib.oracle_verify_chain.argtypes = [P, I, I, I, I, I, P, P, P, P, P, D, D, P, P, P, P, P]
    lib.oracle_verify_chain.restype = I
    lib.oracle_size_level.argtypes = [P, P, P, I, I, I, P, P, I, I, I, ctypes.c_float, P, P, P, P]
    lib.oracle_size_level.restype = I
    for f in ("oracle_round_bf16", "oracle_lowrank_project", "oracle_lowrank_scores",
              "oracle_lowrank_topk", "oracle_exact_rescore", "oracle_tree_accept"):
        getattr(lib, f).restype = I
    return lib


def load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def _raw(x):
    """(contiguous numpy array holding the stored bits, dtype code) for a tensor or array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return np.ascontiguousarray(x.view(torch.int16).numpy().view(np.uint16)), BF16
            if x.dtype == torch.float32:
                return np.ascontiguousarray(x.numpy()), F32
            if x.dtype == torch.int32:
                return np.ascontiguousarray(x.numpy()), None
            raise TypeError(f"unsupported tensor dtype {x.dtype}")
    except ImportError:
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.uint16:
        return x, BF16
    if x.dtype == np.int32:
        return x, None
    raise TypeError(f"unsupported array dtype {x.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _rows(rows, n_all):
    if rows is None:
        return None, n_all
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    return r, len(r)


def _check(rc, what):
    if rc not in (0, -2):
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")
    return rc


def round_bf16(x) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty_like(x)
    _check(load().oracle_round_bf16(_ptr(x), x.size, _ptr(out)), "round_bf16")
    return out


def lowrank_project(h, U, rows=None) -> np.ndarray:
    hh, dt = _raw(h)
    uu, _ = _raw(U)
    B, d = hh.shape
    r = uu.shape[1]
    rr, n = _rows(rows, B)
    out = np.empty((n, r), dtype=np.float64)
    _check(load().oracle_lowrank_project(_ptr(hh), _ptr(uu), B, d, r, dt,
                                         None if rr is None else _ptr(rr), n, _ptr(out)), "project")
    return out


def lowrank_scores(h, U, V, rows=None) -> np.ndarray:
    hh, dt = _raw(h)
    uu, _ = _raw(U)
    vv, _ = _raw(V)
    B, d = hh.shape
    r, vocab = vv.shape
    rr, n = _rows(rows, B)
    out = np.empty((n, vocab), dtype=np.float64)
    _check(load().oracle_lowrank_scores(_ptr(hh), _ptr(uu), _ptr(vv), B, d, r, vocab, dt,
                                        None if rr is None else _ptr(rr), n, _ptr(out)), "scores")
    return out


def lowrank_topk(h, U, V, K, rows=None):
    hh, dt = _raw(h)
    uu, _ = _raw(U)
    vv, _ = _raw(V)
    B, d = hh.shape
    r, vocab = vv.shape
    rr, n = _rows(rows, B)
    idx = np.empty((n, K), dtype=np.int32)
    sc = np.empty((n, K), dtype=np.float64)
    _check(load().oracle_lowrank_topk(_ptr(hh), _ptr(uu), _ptr(vv), B, d, r, vocab, K, dt,
                                      None if rr is None else _ptr(rr), n, _ptr(idx), _ptr(sc)),
           "topk")
    return idx, sc


def exact_rescore(h, W, idx, rows=None):
    hh, dt = _raw(h)
    ww, _ = _raw(W)
    ii, _ = _raw(idx)
    B, d = hh.shape
    vocab = ww.shape[0]
    K = ii.shape[1]
    rr, n = _rows(rows, B)
    z = np.empty((n, K), dtype=np.float64)
    p = np.empty((n, K), dtype=np.float64)
    _check(load().oracle_exact_rescore(_ptr(hh), _ptr(ww), _ptr(ii), B, d, vocab, K, dt,
                                       None if rr is None else _ptr(rr), n, _ptr(z), _ptr(p)),
           "rescore")
    return z, p


def tree_accept(logits, parent, token, reqs=None):
    ll, dt = _raw(logits)
    pp, _ = _raw(parent)
    tt, _ = _raw(token)
    B, N, vocab = ll.shape
    rr, n = _rows(reqs, B)
    am = np.empty((n, N), dtype=np.int32)
    path = np.empty((n, N), dtype=np.int32)
    ln = np.empty((n,), dtype=np.int32)
    bonus = np.empty((n,), dtype=np.int32)
    _check(load().oracle_tree_accept(_ptr(ll), _ptr(pp), _ptr(tt), B, N, vocab, dt,
                                     None if rr is None else _ptr(rr), n, _ptr(am), _ptr(path),
                                     _ptr(ln), _ptr(bonus)), "tree_accept")
    return {"argmax": am, "path": path, "len": ln, "bonus": bonus}


def expand_children(probs, idx, w, parent_prob=None, min_benefit=0.0):
    """Step 7: the w children of each frontier node by exact probability.  probs fp32 [B, K],
    idx int32 [B, K], parent_prob fp32 [B] or None (1).  Returns (child_token int32 [B, w],
    child_prob fp32 [B, w], n_keep int32 [B])."""
    pp = np.ascontiguousarray(np.asarray(probs, dtype=np.float32))
    ii = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    B, K = pp.shape
    par = None if parent_prob is None else np.ascontiguousarray(np.asarray(parent_prob, dtype=np.float32))
    tok = np.empty((B, w), dtype=np.int32)
    cp = np.empty((B, w), dtype=np.float32)
    keep = np.empty((B,), dtype=np.int32)
    _check(load().oracle_expand_children(_ptr(pp), _ptr(ii), None if par is None else _ptr(par), B, K, w,
                                         float(min_benefit), _ptr(tok), _ptr(cp), _ptr(keep)), "expand_children")
    return tok, cp, keep


def verify_chain(logits, cand_idx, cand_prob, draft_token, u_accept, u_sample, temperature=1.0, tol=1e-4):
    """Step 8: speculative sampling over a chain of L drafted tokens per request.

    logits [B, L+1, vocab] (fp32 or bf16), cand_idx int32 [B, L, K], cand_prob fp32 [B, L, K],
    draft_token int32 [B, L], u_accept fp32 [B, L], u_sample fp32 [B].  Returns a dict with
    n_accept, token (the emitted correction or bonus token), and for comparisons in other
    precisions first_close (first decision within tol of its threshold, L+1 if none) and
    token_lo / token_hi (the tokens within tol x total of the sampling point)."""
    ll, dt = _raw(logits)
    B, L1, vocab = ll.shape
    L = L1 - 1
    ci = np.ascontiguousarray(np.asarray(cand_idx, dtype=np.int32))
    K = ci.shape[2] if ci.ndim == 3 else 0
    ci = ci.reshape(B, L, K)
    cp = np.ascontiguousarray(np.asarray(cand_prob, dtype=np.float32)).reshape(B, L, K)
    xt = np.ascontiguousarray(np.asarray(draft_token, dtype=np.int32)).reshape(B, L)
    ua = np.ascontiguousarray(np.asarray(u_accept, dtype=np.float32)).reshape(B, L)
    us = np.ascontiguousarray(np.asarray(u_sample, dtype=np.float32)).reshape(B)
    out = {k: np.empty((B,), dtype=np.int32) for k in ("n_accept", "token", "first_close", "token_lo", "token_hi")}
    _check(load().oracle_verify_chain(_ptr(ll), dt, B, L, vocab, K, _ptr(ci), _ptr(cp), _ptr(xt), _ptr(ua),
                                      _ptr(us), float(temperature), float(tol), _ptr(out["n_accept"]),
                                      _ptr(out["token"]), _ptr(out["first_close"]), _ptr(out["token_lo"]),
                                      _ptr(out["token_hi"])), "verify_chain")
    return out


def size_level(child_prob, child_token, cost, bin_batch, batch, theta, n_valid=None):
    """Step 9: the next level's width and children for each request.

    child_prob fp32 / child_token int32 [R, F, Wc]; n_valid int32 [R, F] or None; cost fp32
    [n_bins, wmax + 1]; bin_batch int32 [n_bins].  Returns dict(width [R], parent, token, prob
    [R, wmax])."""
    cp = np.ascontiguousarray(np.asarray(child_prob, dtype=np.float32))
    R, F, Wc = cp.shape
    ct = np.ascontiguousarray(np.asarray(child_token, dtype=np.int32)).reshape(R, F, Wc)
    nv = None if n_valid is None else np.ascontiguousarray(np.asarray(n_valid, dtype=np.int32)).reshape(R, F)
    c = np.ascontiguousarray(np.asarray(cost, dtype=np.float32))
    n_bins, w1 = c.shape
    wmax = w1 - 1
    bb = np.ascontiguousarray(np.asarray(bin_batch, dtype=np.int32)).reshape(n_bins)
    out = {"width": np.empty(R, dtype=np.int32), "parent": np.empty((R, wmax), dtype=np.int32),
           "token": np.empty((R, wmax), dtype=np.int32), "prob": np.empty((R, wmax), dtype=np.float32)}
    _check(load().oracle_size_level(_ptr(cp), _ptr(ct), None if nv is None else _ptr(nv), R, F, Wc, _ptr(c), _ptr(bb),
                                    n_bins, wmax, int(batch), float(theta), _ptr(out["width"]), _ptr(out["parent"]),
                                    _ptr(out["token"]), _ptr(out["prob"])), "size_level")
    return out
