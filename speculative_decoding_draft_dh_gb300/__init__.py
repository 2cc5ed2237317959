"""GB300-native two-stage draft LM head (low-rank top-K retrieval + exact rescoring) and greedy
draft-tree acceptance.  The compute runs in the CUDA library ``libdh.so`` behind a C ABI
(``include/dh.h``); this package only marshals arguments to it."""
