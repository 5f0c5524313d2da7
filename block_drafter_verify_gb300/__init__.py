"""DFlash 2 draft-verify hot path on GB300 (sm_103a).

The work happens in ``_build/libdflash.so`` (CUDA kernels behind the C ABI
of include/dflash.h); this package is its ctypes binding.
"""
from .binding import (BF16, C, COMMIT_STATS, FP32, STAGES, DFlashError,
                      DraftVerify, EXPORTS, dflash_check, dflash_commit,
                      dflash_cycle, dflash_draft, dflash_draft_e4m3, dflash_lmhead_topk,
                      dflash_path_viterbi, dflash_quantize_e4m3_rows,
                      dflash_top16_recall, dflash_set_wait_limit_ns,
                      dflash_pair_score, dflash_path_walk, dflash_philox4x32,
                      dflash_profile_stage, dflash_verify,
                      dflash_verify_noalloc, dflash_workspace_bytes,
                      dflash_lmhead_topk_shard, dflash_topk_merge_shards,
                      dflash_verify_shard_stats, dflash_verify_shard_decide,
                      dflash_verify_shard_draw, SHARD_STATS, SHARD_PLAN,
                      library_path, load)

__all__ = ["BF16", "C", "COMMIT_STATS", "FP32", "STAGES", "DFlashError",
           "DraftVerify", "EXPORTS", "dflash_check", "dflash_commit",
           "dflash_cycle", "dflash_draft", "dflash_draft_e4m3", "dflash_lmhead_topk",
           "dflash_path_viterbi", "dflash_quantize_e4m3_rows",
           "dflash_top16_recall", "dflash_set_wait_limit_ns",
           "dflash_pair_score", "dflash_path_walk", "dflash_philox4x32",
           "dflash_profile_stage", "dflash_verify", "dflash_verify_noalloc",
           "dflash_workspace_bytes", "dflash_lmhead_topk_shard",
           "dflash_topk_merge_shards", "dflash_verify_shard_stats",
           "dflash_verify_shard_decide", "dflash_verify_shard_draw",
           "SHARD_STATS", "SHARD_PLAN", "library_path", "load"]
