"""Seeded synthetic inputs for the DFlash 2 draft cycle.

This module is shared by the CPU oracle's tests and by the CUDA path's tests and
benchmark. It draws random numbers and lays them out; it performs none of the
drafter's arithmetic (no norms, projections, attention, selection or acceptance).

Every tensor has its own random stream: the seed of a tensor is derived from
(base seed, tensor name, chunk index) through numpy's SeedSequence, and values
are drawn with PCG64. Large tensors are drawn in fixed 4 Mi-element chunks so
the result does not depend on how many threads draw them.

Distributions follow the workload descriptions of the DFlash 2 pages and of the
configurations built here (weights N(0, 0.02), target hidden states N(0, 1),
target logits N(0, 3), uniform token ids); the two readings added here are
norm gains 1 + 0.02 N(0, 1) (so a gain multiply is exercised) and conv base
kernels N(0, 1) (so the sigmoid gates take a spread of values).
"""

from .configs import PRESETS, preset, validate_dims  # noqa: F401
from .gen import (  # noqa: F401
    bf16_bits_to_f32,
    f32_to_bf16_bits,
    make_weights,
    make_q4_weights,
    q4_names,
    make_hiddens,
    make_anchors,
    make_target_logits,
    make_paged_layout,
    make_ctx_lens,
    weight_names,
    stream,
)
