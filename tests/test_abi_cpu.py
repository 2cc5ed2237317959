"""CPU-side checks of the C ABI: the library loads, exports every function that include/dh.h
declares, sizes workspaces, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

from speculative_decoding_draft_dh_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dh.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(dh_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_three_calls():
    fns = declared_functions()
    for name in ("dh_lowrank_topk", "dh_exact_rescore", "dh_tree_accept"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    missing = [f for f in declared_functions() if not hasattr(lib, f)]
    assert not missing, missing
    assert sorted(binding.EXPORTS) == sorted(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        assert lib.dh_status_string(code)
    assert lib.dh_status_string(99) == b"unknown status"
    assert lib.dh_version() >= 100


def test_workspace_sizes(lib):
    # batch-1 draft head: t, projection partials and one 16-byte record per group of 64 ids
    ws = lib.dh_lowrank_topk_workspace(1, 5120, 128, 151936, 64, binding.BF16)
    assert ws >= 151936 // 64 * 16
    assert ws % 256 == 0
    big = lib.dh_lowrank_topk_workspace(512, 5120, 512, 151936, 256, binding.BF16)
    assert big >= 512 * (151936 // 64) * 16
    assert lib.dh_lowrank_topk_workspace(0, 5120, 128, 151936, 64, binding.BF16) == 0
    assert lib.dh_tree_accept_workspace(256, 64, 151936) >= 256 * 64 * 4


FAKE = 0x10000  # 16-byte aligned host-side stand-in; never dereferenced by rejected calls


def _topk(lib, B=1, d=256, r=32, vocab=4096, K=16, dt=binding.F32, h=FAKE, U=FAKE, V=FAKE,
          idx=FAKE, sc=FAKE, ws=FAKE * 16, nbytes=1 << 30):
    P = ctypes.c_void_p
    return lib.dh_lowrank_topk(P(h), P(U), P(V), B, d, r, vocab, K, dt, P(idx), P(sc), P(ws), nbytes,
                               None)


def test_topk_rejects_bad_arguments_on_host(lib):
    assert _topk(lib, K=0) == 1
    assert _topk(lib, K=4097) == 1                      # K > vocab
    assert _topk(lib, vocab=8192, K=1025) == 1          # K > 1024
    assert _topk(lib, d=0) == 1
    assert _topk(lib, h=0) == 1                         # null pointer
    assert _topk(lib, dt=7) == 2                        # unknown dtype
    assert _topk(lib, h=FAKE + 4) == 2                  # misaligned base pointer
    assert _topk(lib, dt=binding.BF16, r=36) == 2       # bf16 row of 72 bytes
    assert _topk(lib, r=2048) == 2                      # above the rank limit
    assert _topk(lib, ws=0) == 3
    assert _topk(lib, ws=FAKE * 16 + 16) == 3           # workspace not 256-byte aligned
    assert _topk(lib, nbytes=64) == 3                   # workspace too small
    assert _topk(lib, B=0) == 0                         # empty batch: nothing to do


def test_rescore_and_tree_reject_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    assert lib.dh_exact_rescore(P(FAKE), P(FAKE), P(FAKE), 1, 256, 4096, 0, 0, P(FAKE), None, None, 0,
                                None) == 1
    assert lib.dh_exact_rescore(P(FAKE), P(FAKE), P(FAKE), 1, 250, 4096, 4, 0, P(FAKE), None, None, 0,
                                None) == 2
    assert lib.dh_exact_rescore(P(FAKE), P(FAKE), P(FAKE), 0, 256, 4096, 4, 0, P(FAKE), None, None, 0,
                                None) == 0
    assert lib.dh_tree_accept(P(FAKE), P(FAKE), P(FAKE), 1, 2048, 4096, 0, None, P(FAKE), P(FAKE),
                              P(FAKE), None, P(FAKE * 16), 1 << 20, None) == 2  # N above limit
    assert lib.dh_tree_accept(P(FAKE), P(FAKE), P(FAKE), 1, 8, 4096, 0, None, None, P(FAKE),
                              P(FAKE), None, P(FAKE * 16), 1 << 20, None) == 1  # path_out missing
    assert lib.dh_tree_accept(P(FAKE), P(FAKE), P(FAKE), 4, 8, 4096, 0, None, P(FAKE), P(FAKE),
                              P(FAKE), None, P(FAKE * 16), 8, None) == 3        # workspace too small


def test_draft_head_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p

    def call(B=1, d=256, r=32, vocab=4096, K=16, dt=binding.F32, W=FAKE, ws=FAKE * 16, nbytes=1 << 30):
        return lib.dh_draft_head(P(FAKE), P(FAKE), P(FAKE), P(W), B, d, r, vocab, K, dt, P(FAKE), P(FAKE),
                                 P(FAKE), None, P(ws) if ws else None, nbytes, None)
    assert call(K=0) == 1
    assert call(W=0) == 1                    # W missing
    assert call(dt=7) == 2
    assert call(d=250) == 2                  # fp32 row of 1000 bytes
    assert call(d=16384) == 2                # above the rescoring limit
    assert call(nbytes=64) == 3
    assert call(B=0) == 0
    need = lib.dh_draft_head_workspace(1, 5120, 128, 151936, 64, binding.BF16)
    assert need >= lib.dh_lowrank_topk_workspace(1, 5120, 128, 151936, 64, binding.BF16)
    assert need % 256 == 0


def test_expand_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float

    def call(B=2, K=16, w=4, probs=FAKE, out=FAKE):
        return lib.dh_expand_children(P(probs) if probs else None, P(FAKE), None, B, K, w, f(0.0),
                                      P(out) if out else None, P(FAKE), None, None)
    assert call(w=0) == 1
    assert call(w=17) == 1        # more children than candidates
    assert call(K=2048, w=4) == 1  # above DH_MAX_K
    assert call(probs=0) == 1
    assert call(out=0) == 1
    assert call(B=0) == 0


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="libdh.so not found"):
        binding.load_library(str(tmp_path / "libdh.so"))


def test_verify_chain_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float

    def call(B=4, L=3, vocab=4096, K=16, dt=binding.F32, T=1.0, logits=FAKE, cand=FAKE, ws=FAKE * 16,
             nbytes=1 << 30):
        return lib.dh_verify_chain(P(logits), P(cand) if cand else None, P(FAKE), P(FAKE), P(FAKE), P(FAKE), B, L,
                                   vocab, K, dt, f(T), P(FAKE), P(FAKE), P(ws) if ws else None, nbytes, None)
    assert call(T=0.0) == 1
    assert call(T=float("inf")) == 1
    assert call(T=float("nan")) == 1
    assert call(K=0) == 1                    # candidates needed when L > 0
    assert call(K=2048) == 1
    assert call(cand=0) == 1
    assert call(dt=5) == 2
    assert call(L=65) == 2                   # deeper than a round may be
    assert call(vocab=4095) == 2             # fp32 row not a multiple of 16 bytes
    assert call(logits=FAKE + 4) == 2        # misaligned
    assert call(nbytes=64) == 3
    assert call(B=0) == 0
    need = lib.dh_verify_chain_workspace(64, 7, 151936, binding.BF16)
    assert need >= 64 * 8 * (151936 // 1024) * 8 and need % 256 == 0  # one (max, sum) pair per 1024 ids
    assert lib.dh_verify_chain_workspace(4, 65, 4096, binding.F32) == 0


def test_size_level_rejects_bad_arguments_on_host(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float

    def call(R=2, F=4, Wc=4, n_bins=2, wmax=8, batch=1, theta=0.01, prob=FAKE, out=FAKE):
        return lib.dh_size_level(P(prob) if prob else None, P(FAKE), None, R, F, Wc, P(FAKE), P(FAKE), n_bins, wmax,
                                 batch, f(theta), P(out) if out else None, P(FAKE), P(FAKE), P(FAKE), None)
    assert call(F=0) == 1
    assert call(n_bins=0) == 1
    assert call(wmax=0) == 1
    assert call(batch=-1) == 1
    assert call(theta=float("nan")) == 1
    assert call(prob=0) == 1
    assert call(out=0) == 1
    assert call(F=4096, Wc=4) == 2           # more children than one block ranks
    assert call(wmax=2048) == 2
    assert call(R=0) == 0
