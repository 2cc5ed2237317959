"""The workspace-free tree acceptance entry point, called through the C ABI.

dh_tree_accept_noalloc serves callers that cannot allocate device memory (allocation is not
allowed where they run, or they own no device allocator): it keeps its scratch in a fixed array
inside the library.  Its results must equal dh_tree_accept's on the same inputs, call after call
(the shared array keeps the previous call's contents).  This file is collected last so that a run
stopping at the first failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_draft_dh_gb300 import binding as dh
from speculative_decoding_draft_dh_gb300 import inputs

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, t):
    logits, parent, token = t["logits"], t["parent"], t["token"]
    B, N, vocab = logits.shape
    dev = logits.device
    out = {k: torch.full((B, N) if k in ("argmax", "path") else (B,), -7, dtype=torch.int32, device=dev)
           for k in ("argmax", "path", "len", "bonus", "err")}
    dt = dh.BF16 if logits.dtype == torch.bfloat16 else dh.F32
    rc = lib.dh_tree_accept_noalloc(_p(logits), _p(parent), _p(token), B, N, vocab, dt, _p(out["argmax"]),
                                    _p(out["path"]), _p(out["len"]), _p(out["bonus"]), _p(out["err"]),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.dh_last_error()
    return out


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_draft_dh_gb300 import build
    build.build()
    return dh.load_library()


@pytest.mark.parametrize("tcfg", [inputs.TREE_CONFIGS["tiny_tree"], inputs.tree_config("tree", B=48, vocab=20000)],
                         ids=["tiny_f32", "bf16_48x64"])
def test_noalloc_matches_workspace_entry_point(lib, tcfg):
    t = inputs.make_tree(tcfg, seed=3, device="cuda")
    ref = dh.tree_accept(t["logits"], t["parent"], t["token"])
    torch.cuda.synchronize()
    for call in range(2):  # two calls in a row share the scratch array
        got = _noalloc(lib, t)
        torch.cuda.synchronize()
        for k in ("argmax", "path", "len", "bonus", "err"):
            np.testing.assert_array_equal(got[k].cpu().numpy(), ref[k].cpu().numpy(), err_msg=f"{k}, call {call}")


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    B, N, vocab = 513, 1024, 16  # B * N above DH_TREE_NOALLOC_MAX_NODES (262144)
    P = ctypes.c_void_p
    fake = 0x10000
    rc = lib.dh_tree_accept_noalloc(P(fake), P(fake), P(fake), B, N, vocab, dh.F32, None, P(fake), P(fake),
                                    P(fake), None, None)
    assert rc == 2
    assert b"DH_TREE_NOALLOC_MAX_NODES" in lib.dh_last_error()
