"""Pins of the CPU oracle against things other than itself: library routines,
closed forms, hand-worked fixtures (tests/golden), brute force and invariants.
CPU only."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dflash as od
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _num(v):
    if isinstance(v, str):
        return float(eval(v, {"ln3": math.log(3.0)}))  # fixture expressions like "0.75*ln3"
    return float(v)


def _arr(a):
    return np.array([[_num(v) for v in row] for row in a]) if isinstance(a[0], list) else \
        np.array([_num(v) for v in a])


# ---------------------------------------------------------------- rounding

def test_round_bf16_matches_torch_on_f32_values():
    g = np.random.default_rng(1)
    x = (g.standard_normal(20000) * np.exp(g.uniform(-20, 20, 20000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(x.astype(np.float64)), ref)


def test_round_bf16_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: the even neighbour is 1
    assert oracle.round_bf16(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: the even one is 1 + 2^-6
    assert oracle.round_bf16(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert oracle.round_bf16(-(1.0 + 2.0 ** -8)) == -1.0


# ---------------------------------------------------------------- rmsnorm

def test_rmsnorm_closed_form():
    y = oracle.rmsnorm(np.array([3.0, 4.0]), np.ones(2), 0.0)
    r = math.sqrt((9 + 16) / 2)
    np.testing.assert_allclose(y, [3 / r, 4 / r], rtol=1e-15)


def test_rmsnorm_matches_torch():
    g = np.random.default_rng(2)
    x = g.standard_normal((5, 96))
    w = 1 + 0.1 * g.standard_normal(96)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-6)
    np.testing.assert_allclose(oracle.rmsnorm(x, w, 1e-6), ref.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- RoPE

def test_rope_theta_zero_is_identity():
    x = np.random.default_rng(3).standard_normal((6, 8))
    np.testing.assert_array_equal(oracle.rope(x, np.arange(6), 0), x)


def test_rope_hand_values_rotate_half_pairing():
    # d=4, theta=10000: frequencies 1 and 0.01; pairs (0,2) and (1,3)
    x = np.array([[1.0, 2.0, 3.0, 4.0]])
    p = 7.0
    c0, s0, c1, s1 = math.cos(p), math.sin(p), math.cos(0.01 * p), math.sin(0.01 * p)
    want = [1 * c0 - 3 * s0, 2 * c1 - 4 * s1, 3 * c0 + 1 * s0, 4 * c1 + 2 * s1]
    np.testing.assert_allclose(oracle.rope(x, [p], 10000.0)[0], want, rtol=1e-14)


def test_rope_relative_position_and_norm():
    g = np.random.default_rng(4)
    q, k = g.standard_normal((1, 64)), g.standard_normal((1, 64))
    th = 1e6
    d1 = oracle.rope(q, [100], th) @ oracle.rope(k, [37], th).T
    d2 = oracle.rope(q, [5100], th) @ oracle.rope(k, [5037], th).T
    np.testing.assert_allclose(d1, d2, rtol=1e-9)
    np.testing.assert_allclose(np.linalg.norm(oracle.rope(q, [999], th)), np.linalg.norm(q), rtol=1e-13)


# ---------------------------------------------------------------- conv

def test_conv_two_tap_hand_fixtures():
    fx = json.load(open(os.path.join(GOLD, "conv_two_tap_hand.json")))
    for case in fx["cases"]:
        u = _arr(case["u"])
        y = oracle.conv_two_tap(u, u, _arr(case["G"]), _arr(case["base"]), case["group"])
        np.testing.assert_allclose(y, _arr(case["expected"]), rtol=1e-13, atol=1e-15,
                                   err_msg=case["name"])


def test_conv_group_equivalence():
    # g=16 equals g=1 when the g=1 map repeats each group row 16 times
    g = np.random.default_rng(5)
    D, grp = 64, 16
    u = g.standard_normal((5, D))
    G16 = g.standard_normal((2 * D // grp, D)) * 0.1
    base = g.standard_normal(2 * D)
    G1 = np.repeat(G16, grp, axis=0)
    np.testing.assert_allclose(oracle.conv_two_tap(u, u, G16, base, grp),
                               oracle.conv_two_tap(u, u, G1, base, 1), rtol=1e-13)


def test_conv_saturated_gates_bypass():
    g = np.random.default_rng(6)
    D = 32
    u = g.standard_normal((4, D))
    base = np.concatenate([np.full(D, 60.0), np.full(D, -60.0)])   # a -> 1, b -> 0
    y = oracle.conv_two_tap(u, u, np.zeros((2 * D, D)), base, 1)
    np.testing.assert_allclose(y, u, rtol=1e-12)


# ---------------------------------------------------------------- attention

def _sdpa_gqa(q, k, v):
    """torch SDPA in float64 with kv heads repeated for the query groups."""
    K, Hq, d = q.shape
    grp = Hq // k.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]
    kt = torch.from_numpy(k).repeat_interleave(grp, dim=1).permute(1, 0, 2)[None]
    vt = torch.from_numpy(v).repeat_interleave(grp, dim=1).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=False)
    return o[0].permute(1, 0, 2).numpy()


def test_attention_matches_torch_sdpa():
    g = np.random.default_rng(7)
    q = g.standard_normal((8, 8, 64))
    k = g.standard_normal((40, 2, 64))
    v = g.standard_normal((40, 2, 64))
    np.testing.assert_allclose(oracle.block_attention(q, k, v, 32), _sdpa_gqa(q, k, v),
                               rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    g = np.random.default_rng(8)
    q = g.standard_normal((3, 2, 16))
    k = np.tile(g.standard_normal((1, 1, 16)), (10, 1, 1))   # identical keys -> uniform weights
    v = g.standard_normal((10, 1, 16))
    o = oracle.block_attention(q, k, v, 7)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=0)[None], o.shape), rtol=1e-12)
    # one key aligned with the query and scaled far above the rest -> that value
    k2 = g.standard_normal((10, 1, 16)) * 0.01
    k2[4, 0] = q[0, 0] * 1000
    o2 = oracle.block_attention(q[:1, :1], k2, v, 7)
    np.testing.assert_allclose(o2[0, 0], v[4, 0], rtol=1e-9)


# ---------------------------------------------------------------- top-k / logsumexp

def test_topk_logp_vs_stable_sort_and_scipy():
    from scipy.special import logsumexp
    g = np.random.default_rng(9)
    z = np.round(g.standard_normal(3000) * 4, 1)               # many exact ties
    ids, lp, lse = oracle.topk_logp(z, 16)
    want = np.argsort(-z, kind="stable")[:16]                    # ties keep the lower id first
    np.testing.assert_array_equal(ids, want)
    np.testing.assert_allclose(lse, logsumexp(z), rtol=1e-14)
    np.testing.assert_allclose(lp, z[want] - logsumexp(z), rtol=1e-13)


# ---------------------------------------------------------------- selector

def test_viterbi_hand_fixture():
    fx = json.load(open(os.path.join(GOLD, "viterbi_hand.json")))
    path, score, margin = oracle.select_path_request(
        np.array(fx["embed"]), np.array(fx["P_u"]), np.array(fx["P_v"]), fx["anchor"],
        np.array(fx["ids"]), np.array(fx["logp"]), with_margin=True)
    assert list(path) == fx["expected_path"]
    assert score == pytest.approx(fx["expected_score"], abs=1e-14)
    assert margin == pytest.approx(fx["expected_margin"], abs=1e-14)


def _brute_paths(E, Pu, Pv, anchor, ids, logp):
    T, k = ids.shape
    u = lambda t: Pu @ E[t]
    v = lambda t: Pv @ E[t]
    scores = {}
    for ranks in itertools.product(range(k), repeat=T):
        toks = [ids[t][ranks[t]] for t in range(T)]
        s, prev = 0.0, anchor
        for t in range(T):
            s += logp[t][ranks[t]] + u(prev) @ v(toks[t])
            prev = toks[t]
        scores[ranks] = s
    return scores


@pytest.mark.parametrize("T,k,seed", [(3, 4, 0), (4, 3, 1), (2, 16, 2), (4, 4, 3)])
def test_viterbi_equals_brute_force(T, k, seed):
    g = np.random.default_rng(seed)
    V, D, r = 50, 12, 4
    E = g.standard_normal((V, D))
    Pu, Pv = g.standard_normal((r, D)), g.standard_normal((r, D))
    ids = np.stack([g.permutation(V - 1)[:k] for _ in range(T)]).astype(np.int32)
    logp = -np.abs(g.standard_normal((T, k)))
    anchor = int(g.integers(0, V - 1))
    scores = _brute_paths(E, Pu, Pv, anchor, ids, logp)
    ranked = sorted(scores.items(), key=lambda kv: -kv[1])
    best_ranks, best = ranked[0]
    path, score, margin = oracle.select_path_request(E, Pu, Pv, anchor, ids, logp, with_margin=True)
    assert score == pytest.approx(best, rel=1e-12)
    assert list(path) == [ids[t][best_ranks[t]] for t in range(T)]
    assert margin == pytest.approx(best - ranked[1][1], rel=1e-9, abs=1e-12)


def test_viterbi_zero_projection_is_per_position_argmax():
    g = np.random.default_rng(11)
    T, k, V, D, r = 7, 16, 300, 8, 4
    ids = np.stack([g.permutation(V)[:k] for _ in range(T)]).astype(np.int32)
    logp = np.sort(-np.abs(g.standard_normal((T, k))), axis=1)[:, ::-1]
    path, _ = oracle.select_path_request(g.standard_normal((V, D)), np.zeros((r, D)),
                                         np.zeros((r, D)), 3, ids, logp)
    np.testing.assert_array_equal(path, ids[:, 0])


def test_viterbi_invariant_to_per_position_shift():
    # replacing log-probabilities by raw logits shifts every path by the same sum
    g = np.random.default_rng(12)
    T, k, V, D, r = 5, 6, 100, 8, 4
    E = g.standard_normal((V, D))
    Pu, Pv = g.standard_normal((r, D)), g.standard_normal((r, D))
    ids = np.stack([g.permutation(V)[:k] for _ in range(T)]).astype(np.int32)
    logp = -np.abs(g.standard_normal((T, k)))
    shift = g.standard_normal(T)[:, None] * 10
    p1, s1 = oracle.select_path_request(E, Pu, Pv, 1, ids, logp)
    p2, s2 = oracle.select_path_request(E, Pu, Pv, 1, ids, logp + shift)
    np.testing.assert_array_equal(p1, p2)
    assert s2 - s1 == pytest.approx(shift.sum(), rel=1e-10)


# ---------------------------------------------------------------- accept

def test_accept_hand_fixture():
    fx = json.load(open(os.path.join(GOLD, "accept_hand.json")))
    for case in fx["cases"]:
        K = len(case["argmax"])
        T = np.zeros((K, fx["vocab"]))
        for i, a in enumerate(case["argmax"]):
            T[i, a] = 1.0
        n, toks = oracle.accept_greedy_request(np.array(case["path"]), T)
        assert n == case["accept_len"], case["name"]
        assert list(toks) == case["tokens"], case["name"]


def test_accept_argmax_ties_pick_lower_id():
    T = np.array([[0.0, 5.0, 1.0, 5.0], [0.0, 0.0, 0.0, 0.0]])
    n, toks = oracle.accept_greedy_request(np.array([1]), T)
    assert (n, list(toks)) == (2, [1, 0])
    n, toks = oracle.accept_greedy_request(np.array([3]), T)
    assert (n, list(toks)) == (1, [1, -1])


# ---------------------------------------------------------------- injection

def _hand_cfg(theta):
    return dict(d_model=4, d_target=4, n_taps=1, n_layers=1, n_q_heads=1, n_kv_heads=1,
                head_dim=4, rms_eps=1e-12, rope_theta=theta)


def _hand_weights():
    I = np.eye(4)
    return {"fc_norm": np.ones(4), "fc": I, "layers.0.wqkv": np.concatenate([0 * I, I, 2 * I]),
            "layers.0.k_norm": np.ones(4)}


def test_inject_hand_example():
    # fc = identity and rmsnorm make c = h / rms(h); K = rmsnorm(c) = c; V = 2c
    h = np.array([[3.0, 3.0, 3.0, 3.0], [2.0, -2.0, 2.0, -2.0]])
    k, v, c = oracle.inject_context(_hand_cfg(0), _hand_weights(), h, [0, 1], contract="none")
    np.testing.assert_allclose(c, [[1, 1, 1, 1], [1, -1, 1, -1]], rtol=1e-12)
    np.testing.assert_allclose(k[0, :, 0], c, rtol=1e-12)
    np.testing.assert_allclose(v[0, :, 0], 2 * c, rtol=1e-12)
    # with RoPE (d=4, theta=10000): position p rotates pairs (0,2) by p and (1,3) by p/100
    k2, _, _ = oracle.inject_context(_hand_cfg(10000.0), _hand_weights(), h[1:], [5], "none")
    p = 5.0
    want = [math.cos(p) - math.sin(p), -math.cos(p / 100) + math.sin(p / 100),
            math.cos(p) + math.sin(p), -math.cos(p / 100) - math.sin(p / 100)]
    np.testing.assert_allclose(k2[0, 0, 0], want, rtol=1e-12)


def test_inject_rows_independent_and_scale_invariant():
    cfg = synth.preset("tiny", rms_eps=0.0)                    # RMSNorm is scale-free at eps = 0
    W = synth.make_weights(cfg, seed=3)
    h = synth.make_hiddens(cfg, 9, seed=3)
    pos = np.arange(9) + 20
    k, v, _ = oracle.inject_context(cfg, W, h, pos, "none")
    k1, v1, _ = oracle.inject_context(cfg, W, h[:4], pos[:4], "none")
    k2, v2, _ = oracle.inject_context(cfg, W, h[4:].astype(np.float64) * 7.5, pos[4:], "none")
    np.testing.assert_allclose(np.concatenate([k1, k2], 1), k, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(np.concatenate([v1, v2], 1), v, rtol=1e-9, atol=1e-12)


# ---------------------------------------------------------------- the draft pass

def _tiny_setup(seed=0, ctx_len=40, K=8, name="tiny", **over):
    cfg = synth.preset(name, **over)
    W = synth.make_weights(cfg, seed=seed, sel_scale=0.3)
    n = ctx_len
    h = synth.make_hiddens(cfg, n, seed=seed)
    k, v, _ = oracle.inject_context(cfg, W, h, np.arange(n), "none")
    return cfg, W, [k[l] for l in range(cfg["n_layers"])], [v[l] for l in range(cfg["n_layers"])]


def test_draft_window_boundary():
    cfg, W, ck, cv = _tiny_setup(ctx_len=90)                  # window 64: keys 26..89
    base = oracle.draft_block_request(cfg, W, ck, cv, 5, 90, 8, "none")["logits"]
    ck2 = [a.copy() for a in ck]
    for a in ck2:
        a[:26] += 3.0                                          # outside the window
    out = oracle.draft_block_request(cfg, W, ck2, cv, 5, 90, 8, "none")["logits"]
    np.testing.assert_array_equal(out, base)
    ck3 = [a.copy() for a in ck]
    ck3[0][26] += 3.0                                          # first key inside the window
    out3 = oracle.draft_block_request(cfg, W, ck3, cv, 5, 90, 8, "none")["logits"]
    assert np.max(np.abs(out3 - base)) > 1e-6


def test_draft_is_non_causal_inside_the_block():
    cfg, W, ck, cv = _tiny_setup()
    g = np.random.default_rng(0)
    x = g.standard_normal((8, cfg["d_model"])) * 0.02
    h0 = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "none", block_inputs=x)["hidden"]
    x2 = x.copy()
    x2[7] += 0.05                                               # last slot changes
    h1 = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "none", block_inputs=x2)["hidden"]
    assert np.max(np.abs(h1[0] - h0[0])) > 1e-8                  # ... and slot 0 sees it


def test_draft_block_mask_equivariance():
    # with the convs bypassed, permuting block rows with their positions permutes the outputs
    cfg, W, ck, cv = _tiny_setup()
    g = np.random.default_rng(1)
    x = g.standard_normal((8, cfg["d_model"])) * 0.02
    pos = np.arange(8) + 40
    perm = g.permutation(8)
    h = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "none", conv_bypass=True,
                                   block_inputs=x, positions=pos)["hidden"]
    hp = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "none", conv_bypass=True,
                                    block_inputs=x[perm], positions=pos[perm])["hidden"]
    np.testing.assert_allclose(hp, h[perm], rtol=1e-10, atol=1e-12)


def test_draft_position_shift_invariance():
    # RoPE is relative: shifting every context and block position by s changes nothing
    cfg = synth.preset("tiny", window=30)                     # both runs read exactly 30 keys
    W = synth.make_weights(cfg, seed=2)
    h = synth.make_hiddens(cfg, 30, seed=2)
    s = 1000
    k0, v0, _ = oracle.inject_context(cfg, W, h, np.arange(30), "none")
    k1, v1, _ = oracle.inject_context(cfg, W, h, np.arange(30) + s, "none")
    L = cfg["n_layers"]
    a = oracle.draft_block_request(cfg, W, [k0[l] for l in range(L)], [v0[l] for l in range(L)],
                                   7, 30, 8, "none")["logits"]
    pad = lambda t: np.concatenate([np.zeros((s,) + t.shape[1:]), t])
    b = oracle.draft_block_request(cfg, W, [pad(k1[l]) for l in range(L)],
                                   [pad(v1[l]) for l in range(L)], 7, 30 + s, 8, "none")
    np.testing.assert_allclose(b["logits"], a, rtol=1e-7, atol=1e-9)


def test_draft_degenerate_layers_reduce_to_lm_head_of_embedding():
    # all projections zero: attention and MLP add nothing, logits = lm_head(norm(embed(token)))
    cfg, W, ck, cv = _tiny_setup()
    Wz = dict(W)
    for l in range(cfg["n_layers"]):
        for n in ("wo", "w_gate_up"):
            Wz[f"layers.{l}.{n}"] = np.zeros_like(W[f"layers.{l}.{n}"])
    out = oracle.draft_block_request(cfg, Wz, ck, cv, 5, 40, 8, "none")["logits"]
    e = W["embed"][cfg["mask_token_id"]].astype(np.float64)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(e), (e.size,),
                                       torch.from_numpy(W["final_norm"].astype(np.float64)),
                                       eps=cfg["rms_eps"])
    want = W["lm_head"].astype(np.float64) @ ref.numpy()
    assert out.shape == (7, cfg["vocab"])
    for t in range(7):
        np.testing.assert_allclose(out[t], want, rtol=1e-10, atol=1e-12)


def test_draft_contract_rounding_stays_close():
    # the bf16 storage contract perturbs logits only at bf16 resolution
    cfg, W, ck, cv = _tiny_setup(name="tiny_bf16")
    a = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "none")["logits"]
    b = oracle.draft_block_request(cfg, W, ck, cv, 5, 40, 8, "bf16")["logits"]
    rel = np.max(np.abs(a - b), axis=1) / np.max(np.abs(a), axis=1)
    assert rel.max() < 2e-2 and rel.max() > 0


# ---------------------------------------------------------------- one drafter layer, by hand

def _sig(z):
    return 1.0 / (1.0 + math.exp(-z))


def _hand_layer_case(fx, case):
    cfg = dict(fx["common"]["cfg"])
    W = {k: np.array(v, dtype=np.float64) for k, v in fx["common"]["weights"].items()}
    W.update({k: np.array(v, dtype=np.float64) for k, v in case["weights"].items()})
    n = case.get("ctx_len", 0)
    shape = (n, cfg["n_kv_heads"], cfg["head_dim"])
    ck = [np.array(case["ctx_k"], dtype=np.float64).reshape(shape) if n else np.zeros(shape)]
    cv = [np.array(case["ctx_v"], dtype=np.float64).reshape(shape) if n else np.zeros(shape)]
    return cfg, W, ck, cv, n


def test_draft_layer_hand_fixtures():
    """One drafter layer on hand-worked 2-wide cases (tests/golden/draft_layer_hand.json):
    SwiGLU takes the gate rows first and applies SiLU to them, the post-sublayer conv
    sits inside the residual branch with its gate map reading the sublayer output,
    and the pre-sublayer conv follows the RMSNorm."""
    fx = json.load(open(os.path.join(GOLD, "draft_layer_hand.json")))
    K, anchor = fx["common"]["K"], fx["common"]["anchor"]
    for case in fx["cases"]:
        cfg, W, ck, cv, n = _hand_layer_case(fx, case)
        out = oracle.draft_block_request(cfg, W, ck, cv, anchor, n, K, contract="none")
        want = np.array([[float(eval(e, {"s": _sig})) for e in row]
                         for row in case["expected_hidden"]])
        np.testing.assert_allclose(out["hidden"], want, rtol=1e-9, atol=1e-12,
                                   err_msg=case["name"])


def test_accept_argmax_orders_nan_above_numbers():
    # numpy's argmax rule: the first NaN of a row is its argmax
    nan = float("nan")
    T = np.array([[1.0, nan, 5.0, nan], [0.0, 2.0, 2.0, -1.0], [nan, nan, nan, nan]])
    assert [int(np.argmax(r)) for r in T] == [1, 1, 0]
    n, toks = oracle.accept_greedy_request(np.array([1, 1]), T)
    assert (n, list(toks)) == (3, [1, 1, 0])
    n, toks = oracle.accept_greedy_request(np.array([2, 1]), T)
    assert (n, list(toks)) == (1, [1, -1, -1])


# ---------------------------------------------------------------- 4-bit weights

def test_dequantize_hand_fixture():
    """s*q + b rounded once to bf16, one (s, b) per group of 64 input features of
    a row: hand-worked values, including two rounding cases and two ties."""
    fx = json.load(open(os.path.join(GOLD, "q4_hand.json")))
    g = fx["group"]
    s = np.asarray(fx["scale"])
    b = np.asarray(fx["bias"])
    q = np.zeros((s.shape[0], s.shape[1] * g), np.int64)
    for r, c, qq, _, _ in fx["entries"]:
        q[r, c] = qq
    w = oracle.dequantize_affine(q, s, b, g)
    for r, c, qq, want, note in fx["entries"]:
        assert w[r, c] == want, (r, c, qq, w[r, c], note)
    # every other weight is its group's bias (q = 0; the biases are bf16 values)
    rest = q == 0
    want_rest = np.repeat(b, g, axis=1)
    np.testing.assert_array_equal(w[rest], want_rest[rest])


def test_dequantized_product_factors_through_groups():
    """With power-of-two scales and small integer biases every step is exact, so
    x @ W^T must equal the group-factored sum  sum_g [s_g sum_k x_k q_k + b_g sum_k x_k]
    written out with loops: pins which axis the groups run along."""
    rng = np.random.default_rng(5)
    N, K, g = 3, 256, 64
    q = rng.integers(0, 16, (N, K))
    s = 2.0 ** rng.integers(-6, -2, (N, K // g))
    b = rng.integers(-4, 4, (N, K // g)).astype(np.float64)
    x = rng.integers(-8, 8, (2, K)).astype(np.float64)
    y = x @ oracle.dequantize_affine(q, s, b, g).T
    want = np.zeros((2, N))
    for t in range(2):
        for n in range(N):
            for j in range(K // g):
                ks = range(j * g, (j + 1) * g)
                want[t, n] += s[n, j] * sum(x[t, k] * q[n, k] for k in ks) + b[n, j] * sum(x[t, k] for k in ks)
    np.testing.assert_array_equal(y, want)


def test_quantized_weights_replace_only_named_matrices():
    cfg = synth.preset("tiny_bf16")
    W = synth.make_weights(cfg, seed=1)
    Q = synth.make_q4_weights(cfg, seed=1)
    Wq = oracle.quantized_weights(W, Q)
    for name in W:
        if name in Q:
            q, s, b = Q[name]
            assert Wq[name].shape == W[name].shape
            np.testing.assert_array_equal(Wq[name], oracle.dequantize_affine(q, s, b, 64))
        else:
            assert Wq[name] is W[name]
