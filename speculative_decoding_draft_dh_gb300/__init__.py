"""GB300-native two-stage draft LM head (low-rank top-K retrieval + exact rescoring) and greedy
draft-tree acceptance.  The compute runs in the CUDA library ``libdh.so`` behind a C ABI
(``include/dh.h``); this package only marshals arguments to it (``binding``), draws seeded
synthetic inputs (``inputs``) and builds the library (``build``)."""

__version__ = "1.0.0"


def __getattr__(name):
    if name in ("lowrank_topk", "exact_rescore", "tree_accept", "prof_enable", "prof_read",
                "load_library", "DhError", "Workspace"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
