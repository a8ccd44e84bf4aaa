"""DFlash2 draft + select + verify step on GB300 (sm_103a): a C-ABI CUDA library
(include/dflash2.h, sources in csrc/) and its thin Python binding."""
from .binding import (  # noqa: F401
    Drafter, Dflash2Error, dflash2_create, dflash2_destroy, dflash2_draft_block, dflash2_select, dflash2_verify,
    dflash2_advance, dflash2_block_width, dflash2_set_select_mode, dflash2_head_topk, dflash2_tree_build,
    dflash2_tree_verify, dflash2_step, dflash2_step_graphs_clear,
    dflash2_head_topk_noalloc, dflash2_debug_set_pipeline_error, dflash2_debug_noalloc_inject_error,
    dflash2_launch_count, dflash2_set_lmhead_events, dflash2_lmhead_bytes, dflash2_set_projection_events,
    dflash2_projection_launches, dflash2_projection_bytes, lib, make_config, upload_weights,
)
from .builder import build, LIB  # noqa: F401
