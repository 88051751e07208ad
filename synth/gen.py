"""Seeded generators: weights, target hidden states, anchors, target logits,
context lengths and paged-cache layouts.  Pure data preparation."""

import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 22  # elements drawn per independent stream chunk


def _seq(base_seed, name, chunk=0):
    return np.random.SeedSequence([int(base_seed) & 0xFFFFFFFF, zlib.crc32(name.encode()), int(chunk)])


def stream(base_seed, name, chunk=0):
    """A PCG64 generator for tensor `name` (and chunk) under `base_seed`."""
    return np.random.Generator(np.random.PCG64(_seq(base_seed, name, chunk)))


def f32_to_bf16_bits(x):
    """Round float32 values to the nearest bfloat16 (ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    r = (b >> 16) & 1                       # finite values cannot overflow 32 bits here
    r += 0x7FFF
    r += b
    r >>= 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits):
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _to_storage(x, dtype):
    if dtype == "bf16":
        return bf16_bits_to_f32(f32_to_bf16_bits(x))
    return x.astype(np.float32, copy=False)


def _normal(base_seed, name, shape, mean, std, dtype, threads=None):
    """N(mean, std) draws in fixed chunks, rounded to the storage dtype."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        g = stream(base_seed, name, c)
        v = g.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        if mean != 0.0:
            v += np.float32(mean)
        out[lo:hi] = _to_storage(v, dtype)

    if nchunks == 1:
        fill(0)
    else:
        workers = threads or min(16, os.cpu_count() or 1)
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def weight_names(cfg):
    """(name, shape, kind) of every drafter weight; kind picks the distribution."""
    D, F, V = cfg["d_model"], cfg["d_ff"], cfg["vocab"]
    Hq, Hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    Tin = cfg["n_taps"] * cfg["d_target"]
    G = 2 * D // cfg["conv_group"]
    r = cfg["sel_rank"]
    out = [
        ("fc_norm", (Tin,), "gain"),
        ("fc", (D, Tin), "w"),
        ("embed", (V, D), "w"),
        ("lm_head", (V, D), "w"),
        ("final_norm", (D,), "gain"),
        ("sel_pu", (r, D), "sel"),
        ("sel_pv", (r, D), "sel"),
        ("sel_gate", (r, D), "sel"),
    ]
    for l in range(cfg["n_layers"]):
        p = f"layers.{l}."
        out += [
            (p + "attn_norm", (D,), "gain"),
            (p + "mlp_norm", (D,), "gain"),
            (p + "wqkv", ((Hq + 2 * Hkv) * dh, D), "w"),
            (p + "wo", (D, Hq * dh), "w"),
            (p + "q_norm", (dh,), "gain"),
            (p + "k_norm", (dh,), "gain"),
            (p + "w_gate_up", (2 * F, D), "w"),
            (p + "w_down", (D, F), "w"),
        ]
        for i in range(4):
            out += [(p + f"conv_w.{i}", (G, D), "w"), (p + f"conv_base.{i}", (2 * D,), "base")]
    return out


def make_weights(cfg, seed=0, sel_scale=0.02, base_scale=1.0, w_scale=0.02, names=None):
    """All drafter weights as float32 arrays holding storage-dtype values.

    sel_scale sets the std of the selector projections P_u, P_v (0.02 by
    default, like every other matrix; tests raise it so the pair term competes
    with the per-position log-probabilities)."""
    dtype = cfg["dtype"]
    W = {}
    for name, shape, kind in weight_names(cfg):
        if names is not None and name not in names:
            continue
        if kind == "w":
            W[name] = _normal(seed, name, shape, 0.0, w_scale, dtype)
        elif kind == "sel":
            W[name] = _normal(seed, name, shape, 0.0, sel_scale, dtype)
        elif kind == "gain":
            W[name] = _normal(seed, name, shape, 1.0, 0.02, dtype)
        elif kind == "base":
            W[name] = _normal(seed, name, shape, 0.0, base_scale, dtype)
    return W


def q4_names(cfg):
    """The matrices a 4-bit drafter keeps in 4 bits: the injection fc, every layer's
    QKV, O, gate/up and down projections, and the lm_head."""
    out = ["fc", "lm_head"]
    for l in range(cfg["n_layers"]):
        out += [f"layers.{l}.{n}" for n in ("wqkv", "wo", "w_gate_up", "w_down")]
    return out


def _uniform_u4(base_seed, name, shape, threads=None):
    """Integers uniform on 0..15 (uint8), drawn in fixed chunks."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8)
    nchunks = (n + CHUNK - 1) // CHUNK

    def fill(c):
        lo, hi = c * CHUNK, min(n, (c + 1) * CHUNK)
        out[lo:hi] = stream(base_seed, name, c).integers(0, 16, hi - lo, dtype=np.uint8)

    if nchunks == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(threads or min(16, os.cpu_count() or 1)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out.reshape(shape)


def make_q4_weights(cfg, seed=0, group=64, names=None):
    """4-bit weights of the matrices in q4_names: name -> (q, scale, bias) with q
    [N, K] uint8 uniform on 0..15 and, per group of `group` input features of a
    row, scale uniform on [0.002, 0.006] and bias -7.5*scale + N(0, 0.002), both
    bf16 values (float32 arrays), so the weights s*q + b spread over about
    +-0.03 around zero (std ~0.018, like the N(0, 0.02) bf16 weights)."""
    shapes = {n: sh for n, sh, _ in weight_names(cfg)}
    Q = {}
    for name in q4_names(cfg):
        if names is not None and name not in names:
            continue
        N, K = shapes[name]
        q = _uniform_u4(seed, name + ".q", (N, K))
        g = stream(seed, name + ".scale")
        sc = _to_storage(g.uniform(0.002, 0.006, (N, K // group)).astype(np.float32), "bf16")
        nb = stream(seed, name + ".bias").standard_normal((N, K // group), dtype=np.float32)
        bias = _to_storage(np.float32(-7.5) * sc + np.float32(0.002) * nb, "bf16")
        Q[name] = (q, sc, bias)
    return Q


def make_hiddens(cfg, N, seed=0, name="hiddens"):
    """Concatenated target hidden states of the tapped layers, [N, n_taps*d_target], N(0,1)."""
    return _normal(seed, name, (N, cfg["n_taps"] * cfg["d_target"]), 0.0, 1.0, cfg["dtype"])


def make_anchors(cfg, B, seed=0, name="anchors"):
    """Anchor (last verified) token ids, uniform on [0, vocab-2] so the mask id never appears."""
    g = stream(seed, name)
    return g.integers(0, cfg["vocab"] - 1, size=B, dtype=np.int64).astype(np.int32)


def make_target_logits(cfg, B, K, seed=0, name="target_logits", std=3.0):
    """Synthetic target-verification logits [B, K, vocab], N(0, std), float32."""
    return _normal(seed, name, (B, K, cfg["vocab"]), 0.0, std, "f32")


def make_ctx_lens(B, lo, hi, seed=0, name="ctx_lens"):
    """Context lengths uniform on [lo, hi] (inclusive)."""
    g = stream(seed, name)
    return g.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)


def make_paged_layout(tokens_per_req, page_size, seed=0, shuffle=True, extra_pages=0,
                      name="page_perm"):
    """Page table for requests holding tokens_per_req[b] cache slots.

    Returns (page_table [B, max_pages] int32, num_pages).  Page ids are a seeded
    permutation of the pool when shuffle is set, else consecutive.  Unused
    table entries hold -1."""
    tokens_per_req = np.asarray(tokens_per_req, dtype=np.int64)
    need = (tokens_per_req + page_size - 1) // page_size
    need = np.maximum(need, 1)
    total = int(need.sum()) + int(extra_pages)
    maxp = int(need.max())
    ids = np.arange(total, dtype=np.int64)
    if shuffle:
        ids = stream(seed, name).permutation(total)
    table = np.full((len(need), maxp), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        table[b, :n] = ids[o:o + n]
        o += n
    return table, total
