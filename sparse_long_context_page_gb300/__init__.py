"""GB300-native (sm_103a) hot path of MOIRA-style sparse decoding.

MOIRA ("Mass-Oriented Indexing with Ragged Attention for Long-Context
Decoding", arXiv 2610.04313): at each decode step, per request, layer and KV
head, the fewest KV-cache pages whose estimated share of the attention adds
up to gamma are picked, and an attention kernel that plans its own work from
the list lengths reads only those pages.  The compute lives in ``libmoira.so`` (hand-written CUDA, C ABI in
``include/moira.h``); this package only marshals torch tensors into it.
The library is loaded on first use; there is no CPU fallback.
"""
from ._binding import (DEV_BADLEN, DEV_BADPAGE, DEV_TIMEOUT, EXPORTS, GROUP, HEAD_DIM,
                       MAX_PAGES_PER_SEQ, MAX_UNITS, PAGE_SIZE, RULE_COVERAGE, RULE_TOPDELTA,
                       RULE_TOPK, SUMM_BF16, SUMM_Q2, SUMM_Q8, MoiraError, Shape, append_kv, attend,
                       attend_grid_blocks, decode_step, decode_step_ex, decode_step_host,
                       library_path, load_library, make_summaries, make_workspace,
                       read_device_status, select, select_attend, select_attend_is_fused, select_cluster_size,
                       select_clustered, select_ex, select_rule, shape_of, summary_page_bytes, update_summaries, workspace_bytes, workspace_init)

__all__ = ["DEV_BADLEN", "DEV_BADPAGE", "DEV_TIMEOUT", "EXPORTS", "GROUP", "HEAD_DIM",
           "MAX_PAGES_PER_SEQ", "MAX_UNITS", "PAGE_SIZE", "RULE_COVERAGE", "RULE_TOPDELTA",
           "RULE_TOPK", "SUMM_BF16", "SUMM_Q2", "SUMM_Q8", "MoiraError", "Shape", "append_kv",
           "attend", "attend_grid_blocks", "decode_step", "decode_step_ex", "decode_step_host",
           "library_path", "load_library", "make_summaries", "make_workspace",
           "read_device_status", "select", "select_attend", "select_attend_is_fused", "select_cluster_size",
           "select_clustered", "select_ex", "select_rule", "shape_of",
           "summary_page_bytes", "update_summaries", "workspace_bytes", "workspace_init"]
