"""GB300-native DFlash 2 draft cycle: a C-ABI CUDA library (sm_103a) and its binding.

    inject_context  target hidden states -> per-layer paged draft KV
    draft_block     one non-causal drafter pass over a block, per-position top-k
    draft_block_inject  inject_context + draft_block in one pass (K/V weights read once)
    select_path     low-rank bilinear Viterbi over the candidate lattice
    accept_greedy   longest prefix matching the target's argmax + bonus token
    sample_path     temperature-1 sampling walk over the same pair scores
    select_greedy   the pages' context-gated pair scores, greedy best-successor walk
    accept_sample   lossless speculative rejection sampling against the target
"""

from . import _lib  # noqa: F401
from ._lib import (  # noqa: F401
    DEV_PAGE_RANGE,
    DEV_POS_RANGE,
    DEV_REQ_RANGE,
    DEV_TIMEOUT,
    DEV_TOKEN_RANGE,
    DFlashError,
    lib,
)
from .api import (  # noqa: F401
    DeviceWeights,
    DraftCycle,
    PagedKV,
    Workspace,
    accept_greedy,
    accept_greedy_noalloc,
    accept_sample,
    clear_device_status,
    draft_block,
    draft_block_inject,
    draft_hidden,
    inject_context,
    launch_count,
    linear,
    linear_q4,
    linear_splits,
    make_config,
    pack_q4,
    prepare_selector,
    read_device_status,
    sample_path,
    select_greedy,
    select_path,
    workspace_bytes,
)
