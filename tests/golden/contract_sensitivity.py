"""Measures how far the oracle's own logits move when every value is perturbed
by 1e-6 (relative) just before each bf16 storage rounding - the size of the
difference between float32 and float64 arithmetic.  Writes
contract_sensitivity.json beside this file.  Calls only oracle/ and synth/.

The full drafter (width 4096, 5 layers, vocab 151936) on one B=1, K=8 request
with 1024 context keys: the bf16 storage contract turns sub-ulp differences
into rounding flips that cascade through the GEMMs, so the logit shift is of
the order of the bf16 rounding noise itself.  The full-size parity tests
compare decisions against the oracle only where the oracle's margin exceeds
twice this shift.

    python tests/golden/contract_sensitivity.py
"""

import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import synth  # noqa: E402
from oracle import dflash as od  # noqa: E402


def main():
    cfg = synth.preset("full")
    W = synth.make_weights(cfg, seed=0, sel_scale=0.3)
    ctx, n = 2048, cfg["window"]
    g = synth.stream(7, "sensitivity_ctx")
    shape = (ctx, cfg["n_kv_heads"], cfg["head_dim"])
    ck, cv = [], []
    for _ in range(cfg["n_layers"]):
        a = np.zeros(shape)
        a[ctx - n:] = od.round_bf16(g.standard_normal((n,) + shape[1:]))
        ck.append(a)
        a = np.zeros(shape)
        a[ctx - n:] = od.round_bf16(g.standard_normal((n,) + shape[1:]))
        cv.append(a)
    anchor = int(synth.make_anchors(cfg, 1, seed=7)[0])
    base = od.draft_block_request(cfg, W, ck, cv, anchor, ctx, 8, "bf16")["logits"]
    exact = od.draft_block_request(cfg, W, ck, cv, anchor, ctx, 8, "none")["logits"]
    orig = od.storage_round
    shifts = []
    for seed in (1, 2):
        rng = np.random.default_rng(seed)

        def noisy(x, contract, rng=rng):
            x = np.asarray(x, dtype=np.float64)
            if contract == "bf16":
                x = x * (1.0 + 1e-6 * rng.standard_normal(x.shape))
            return orig(x, contract)

        od.storage_round = noisy
        try:
            pert = od.draft_block_request(cfg, W, ck, cv, anchor, ctx, 8, "bf16")["logits"]
        finally:
            od.storage_round = orig
        shifts.append(float(np.abs(pert - base).max()))
    out = {
        "what": "max |logit change| of the full-size oracle (bf16 contract) when each value is "
                "perturbed by 1e-6 relative before every bf16 rounding; two perturbation seeds",
        "config": "full drafter, B=1, K=8, ctx 2048, window 1024, synth seed 0 (sel_scale 0.3)",
        "shift_per_seed": shifts,
        "shift": max(shifts),
        "bf16_vs_float64_gap": float(np.abs(base - exact).max()),
        "max_abs_logit": float(np.abs(base).max()),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "contract_sensitivity.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
