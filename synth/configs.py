"""Dimension presets of the drafter workloads.

`full` is the full-size drafter of a 27B-class target (DFlash 2 Architecture
page, Component Breakdown table: 5 layers, 1024-token sliding window; the
remaining widths are the ones the workloads fix: target hidden 5120 from 5
tapped layers, draft width 4096, 32 q / 8 kv heads of 128, SwiGLU 14336, vocab
151936, top-16, selector rank 256).  `tiny` is the small drafter used for fast
exact checks.  `small` and `small_gqa` are extra shapes that span several GEMM
tiles with ragged tails (vocab and gate widths not multiples of 128).
"""

BASE = dict(
    page_size=64,
    conv_group=16,
    rms_eps=1e-6,
    rope_theta=1.0e6,
)

PRESETS = {
    "tiny": dict(
        d_model=256, d_target=256, n_taps=3, n_layers=2, n_q_heads=4, n_kv_heads=2,
        head_dim=64, d_ff=512, vocab=4096, window=64, top_k=4, sel_rank=16,
        dtype="f32", **BASE),
    "tiny_bf16": dict(
        d_model=256, d_target=256, n_taps=3, n_layers=2, n_q_heads=4, n_kv_heads=2,
        head_dim=64, d_ff=512, vocab=4096, window=64, top_k=4, sel_rank=16,
        dtype="bf16", **BASE),
    "small": dict(
        d_model=512, d_target=384, n_taps=2, n_layers=2, n_q_heads=8, n_kv_heads=2,
        head_dim=64, d_ff=1344, vocab=5000, window=96, top_k=16, sel_rank=32,
        dtype="bf16", **BASE),
    "small_gqa": dict(
        d_model=1024, d_target=512, n_taps=3, n_layers=1, n_q_heads=8, n_kv_heads=2,
        head_dim=128, d_ff=2048, vocab=9000, window=128, top_k=8, sel_rank=64,
        dtype="bf16", **BASE),
    "full": dict(
        d_model=4096, d_target=5120, n_taps=5, n_layers=5, n_q_heads=32, n_kv_heads=8,
        head_dim=128, d_ff=14336, vocab=151936, window=1024, top_k=16, sel_rank=256,
        dtype="bf16", **BASE),
}


def preset(name, **overrides):
    cfg = dict(PRESETS[name])
    cfg.update(overrides)
    cfg.setdefault("mask_token_id", cfg["vocab"] - 1)
    validate_dims(cfg)
    return cfg


def validate_dims(cfg):
    """Shape rules the drafter dimensions must satisfy (raises ValueError)."""
    d = cfg
    need = [
        (d["d_model"] % 64 == 0, "d_model must be a multiple of 64"),
        (d["d_ff"] % 64 == 0, "d_ff must be a multiple of 64"),
        ((d["n_taps"] * d["d_target"]) % 64 == 0, "n_taps*d_target must be a multiple of 64"),
        (d["head_dim"] in (64, 128), "head_dim must be 64 or 128"),
        (d["n_q_heads"] % d["n_kv_heads"] == 0, "n_q_heads must be a multiple of n_kv_heads"),
        ((d["n_q_heads"] * d["head_dim"]) % 64 == 0, "q width must be a multiple of 64"),
        (d["d_model"] % d["conv_group"] == 0, "d_model must be a multiple of conv_group"),
        (1 <= d["top_k"] <= 32, "top_k must be in 1..32"),
        (d["sel_rank"] % 16 == 0 and d["sel_rank"] <= 1024, "sel_rank must be a multiple of 16, <= 1024"),
        (d["window"] >= 1, "window must be >= 1"),
        (d["page_size"] >= 1, "page_size must be >= 1"),
        (0 <= d.get("mask_token_id", d["vocab"] - 1) < d["vocab"], "mask_token_id out of range"),
        (d["dtype"] in ("f32", "bf16"), "dtype must be f32 or bf16"),
    ]
    for ok, msg in need:
        if not ok:
            raise ValueError(msg)
    return True
