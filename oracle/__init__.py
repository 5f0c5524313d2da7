"""CPU oracle of the DFlash 2 draft-verify hot path (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never does.
"""
from . import philox
from .dflash_oracle import (C, commit, conv2tap, draft_verify_cycle, gate,
                            lmhead_topk, pair_score, path_total,
                            path_viterbi, path_walk, round_bf16, to_storage,
                            top16_recall, verify)

__all__ = ["philox", "C", "commit", "conv2tap", "draft_verify_cycle", "gate",
           "lmhead_topk", "pair_score", "path_total", "path_viterbi",
           "path_walk", "round_bf16", "to_storage", "top16_recall", "verify"]
