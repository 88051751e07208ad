"""CPU oracle of the DFlash 2 draft cycle.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check in
__graft_entry__ and the CPU-baseline leg of bench.py may import or run this
package.  The product path (the C-ABI library and its Python binding) never
calls it and shares no code with it.

Plain, slow and step-by-step: NumPy in float64, loops over requests, layers
and positions, np.matmul for dense products.  Each function names the passage
of the DFlash pages it follows.  Pins that hold it to something other than
itself live in tests/test_oracle_*.py.  The end-to-end composition (a whole
draft pass on random weights) has no printed value to compare with: parity
unpinned for the composition; each step is pinned separately.
"""

from .dflash import (  # noqa: F401
    round_bf16,
    storage_round,
    dequantize_affine,
    quantized_weights,
    rmsnorm,
    rope,
    conv_two_tap,
    block_attention,
    inject_context,
    draft_block,
    draft_block_request,
    topk_logp,
    select_path,
    select_path_request,
    accept_greedy,
    accept_greedy_request,
    draw_index,
    sample_path,
    sample_path_request,
    accept_sample,
    accept_sample_request,
    context_gate,
    select_greedy,
    select_greedy_request,
)
