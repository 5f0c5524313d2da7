"""CPU oracle of the DFlash 2 draft-verify hot path (test infrastructure).

Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never does.
"""
from . import philox
from .dflash_oracle import (C, E4M3_MAX, commit, conv2tap,
                            dequantize_e4m3_rows, dequantize_nvfp4_rows,
                            draft_verify_cycle, e2m1_decode, e2m1_encode,
                            e4m3_decode, e4m3_encode, gate, lmhead_topk,
                            lmhead_topk_e4m3, lmhead_topk_nvfp4, pair_score,
                            path_total,
                            path_viterbi, path_walk, quantize_e4m3_rows,
                            quantize_nvfp4_rows,
                            round_bf16, to_storage,
                            top16_recall, verify)

__all__ = ["philox", "C", "E4M3_MAX", "commit", "conv2tap",
           "dequantize_e4m3_rows", "dequantize_nvfp4_rows",
           "draft_verify_cycle", "e2m1_decode", "e2m1_encode", "e4m3_decode",
           "e4m3_encode", "gate", "lmhead_topk", "lmhead_topk_e4m3",
           "lmhead_topk_nvfp4",
           "quantize_e4m3_rows", "quantize_nvfp4_rows", "pair_score", "path_total", "path_viterbi",
           "path_walk", "round_bf16", "to_storage", "top16_recall", "verify"]
