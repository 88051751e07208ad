"""Pins of the oracle's sampling walk and speculative rejection sampling
(Architecture page, "Problem 1": sampling draws from the same pair scores;
"Speculative Decoding Context": rejection sampling makes the scheme lossless):
hand cases of the inverse-CDF draw, the walk's path probabilities against
their product form, and Monte-Carlo chi-square checks that the committed
tokens follow the target distribution exactly.  CPU only."""

import itertools
import math

import numpy as np
import pytest
from scipy.stats import chi2

import oracle

P_VALUE = 1e-4   # chi-square tests reject only below this p-value (fixed seeds)


def chi2_ok(counts, probs):
    counts = np.asarray(counts, dtype=np.float64)
    n = counts.sum()
    expect = n * np.asarray(probs, dtype=np.float64)
    keep = expect > 0
    assert np.all(counts[~keep] == 0), "mass where the target has none"
    stat = float(np.sum((counts[keep] - expect[keep]) ** 2 / expect[keep]))
    df = int(keep.sum()) - 1
    return stat <= chi2.ppf(1.0 - P_VALUE, df), stat, df


def test_draw_index_hand_cases():
    w = [0.0, 2.0, 0.0, 1.0, 1.0]       # running sums 0, 2, 2, 3, 4
    assert oracle.draw_index(w, 0.0) == 1       # u = 0: the first positive weight
    assert oracle.draw_index(w, 0.49) == 1      # 1.96 < 2
    assert oracle.draw_index(w, 0.5) == 3       # 2.0 is not < 2: next positive weight
    assert oracle.draw_index(w, 0.74) == 3      # 2.96 < 3
    assert oracle.draw_index(w, 0.75) == 4
    assert oracle.draw_index(w, 0.999999) == 4


def _lattice(g, T, k, V, D=5, r=3, scale=1.0):
    E = g.standard_normal((V, D))
    Pu, Pv = g.standard_normal((r, D)) * scale, g.standard_normal((r, D)) * scale
    ids = np.stack([g.permutation(V)[:k] for _ in range(T)]).astype(np.int32)
    logp = np.log(g.dirichlet(np.ones(k), size=T))
    return E, Pu, Pv, ids, logp


def test_walk_path_probabilities_are_the_product_of_its_steps():
    """Sampled path frequencies against prod_t q_t(j_t | j_(t-1)) computed here
    from the pair-score definition, over all k^T paths."""
    g = np.random.default_rng(0)
    T, k, V = 3, 3, 12
    E, Pu, Pv, ids, logp = _lattice(g, T, k, V)
    anchor = 7

    def step(prev, t):
        s = np.array([logp[t][j] + (Pu @ E[prev]) @ (Pv @ E[ids[t][j]]) for j in range(k)])
        e = np.exp(s - s.max())
        return e / e.sum()

    paths = list(itertools.product(range(k), repeat=T))
    probs = []
    for ranks in paths:
        pr, prev = 1.0, anchor
        for t, j in enumerate(ranks):
            pr *= step(prev, t)[j]
            prev = ids[t][j]
        probs.append(pr)
    assert abs(sum(probs) - 1.0) < 1e-12
    index = {tuple(ids[t][j] for t, j in enumerate(rk)): n for n, rk in enumerate(paths)}
    counts = np.zeros(len(paths))
    rng = np.random.default_rng(1)
    for _ in range(60000):
        path, q = oracle.sample_path_request(E, Pu, Pv, anchor, ids, logp, rng.random(T))
        counts[index[tuple(int(x) for x in path)]] += 1
    ok, stat, df = chi2_ok(counts, probs)
    assert ok, (stat, df)
    # and q is the step distribution given the drawn predecessor
    path, q = oracle.sample_path_request(E, Pu, Pv, anchor, ids, logp, [0.3, 0.6, 0.9])
    np.testing.assert_allclose(q[0], step(anchor, 0), rtol=1e-12)
    np.testing.assert_allclose(q[1], step(path[0], 1), rtol=1e-12)


def test_walk_without_pair_term_draws_from_logp():
    """P_u = P_v = 0: every step is softmax(logp_t), independent of the path."""
    g = np.random.default_rng(2)
    T, k, V = 2, 4, 20
    E, _, _, ids, logp = _lattice(g, T, k, V)
    Z = np.zeros((3, 5))
    _, q = oracle.sample_path_request(E, Z, Z, 3, ids, logp, [0.5, 0.5])
    np.testing.assert_allclose(q, np.exp(logp), rtol=1e-12)


def test_accept_when_draft_equals_target():
    """q = p: every draft is accepted (u q < p for every u < 1) and the bonus
    token comes from the last row."""
    V, K = 8, 4
    g = np.random.default_rng(3)
    T = g.standard_normal((K, V))
    p = np.exp(T - T.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    cand = np.tile(np.arange(V), (K - 1, 1))
    path = np.array([2, 5, 1])
    for u0 in (0.0, 0.5, 0.999999):
        u = np.full((K, 2), u0)
        n, toks = oracle.accept_sample_request(path, cand, p[:K - 1], T, u)
        assert n == K and list(toks[:K - 1]) == [2, 5, 1]
        assert toks[K - 1] == oracle.draw_index(p[K - 1], u0)


def test_accept_rejects_tokens_the_target_excludes():
    """p(x) = 0 for the draft token: always rejected, replacement from max(0, p - q)."""
    V, K = 5, 2
    T = np.array([[0.0, -np.inf, 1.0, 0.5, 0.0], [0.0] * 5])
    cand = np.array([[1, 2]])
    q = np.array([[0.7, 0.3]])
    p = np.exp(T[0] - 1.0)
    p /= p.sum()
    r = np.maximum(p - np.array([0, 0.7, 0.3, 0, 0]), 0)
    for uu in (0.0, 0.3, 0.8):
        n, toks = oracle.accept_sample_request(np.array([1]), cand, q, T, np.array([[0.0, uu], [0, 0]]))
        assert n == 1 and toks[0] == oracle.draw_index(r, uu) and toks[1] == -1


def _simulate(M, K, p_pos, lat, anchor, n, seed):
    """Generate M positions by repeated draft cycles of block K: each cycle walks
    the lattice of the next K-1 positions from the last committed token, the
    target rows are those positions' (prefix-independent) logits, and the
    accepted tokens are committed.  Returns counts[M][V] of committed tokens."""
    E, Pu, Pv, ids, logp, logits = lat
    V = logits.shape[1]
    rng = np.random.default_rng(seed)
    counts = np.zeros((M, V))
    for _ in range(n):
        pos, prev = 0, anchor
        while pos < M:
            rows = [min(pos + i, M - 1 + K) for i in range(K)]
            path, q = oracle.sample_path_request(E, Pu, Pv, prev, ids[rows[:K - 1]],
                                                 logp[rows[:K - 1]], rng.random(K - 1))
            acc, toks = oracle.accept_sample_request(path, ids[rows[:K - 1]], q, logits[rows],
                                                     rng.random((K, 2)))
            for i in range(acc):
                if pos + i < M:
                    counts[pos + i, toks[i]] += 1
            prev = int(toks[acc - 1])
            pos += acc
    return counts


@pytest.mark.parametrize("K,seed", [(3, 0), (4, 1)])
def test_rejection_sampling_is_lossless(K, seed):
    """Monte Carlo: the committed token at every position follows the target's
    distribution softmax(logits_pos), whatever the drafter proposed."""
    g = np.random.default_rng(100 + seed)
    M, k, V = 3, 3, 6
    rows = M + K
    E, Pu, Pv, ids, logp = _lattice(g, rows, k, V, scale=1.5)
    logits = g.standard_normal((rows, V)) * 1.5
    counts = _simulate(M, K, None, (E, Pu, Pv, ids, logp, logits), anchor=2, n=40000, seed=seed)
    for m in range(M):
        p = np.exp(logits[m] - logits[m].max())
        p /= p.sum()
        ok, stat, df = chi2_ok(counts[m], p)
        assert ok, (m, stat, df)


def test_lossless_check_detects_a_biased_sampler(monkeypatch):
    """The Monte-Carlo check fails when the replacement is drawn from p instead of
    max(0, p - q) (a plausible mistake), so it has the power to pin the rule."""
    orig = oracle.dflash.accept_sample_request

    def biased(path, cand_ids, q, T, u):
        T = np.asarray(T, dtype=np.float64)
        K = T.shape[0]
        toks = np.full(K, -1, dtype=np.int32)
        for i in range(K - 1):
            p = np.exp(T[i] - T[i].max())
            p /= p.sum()
            x = int(path[i])
            qx = float(q[i][list(cand_ids[i]).index(x)])
            if u[i][0] * qx < p[x]:
                toks[i] = x
                continue
            toks[i] = oracle.draw_index(p, u[i][1])
            return i + 1, toks
        p = np.exp(T[K - 1] - T[K - 1].max())
        toks[K - 1] = oracle.draw_index(p / p.sum(), u[K - 1][1])
        return K, toks

    monkeypatch.setattr(oracle, "accept_sample_request", biased)
    g = np.random.default_rng(100)
    M, K, k, V = 3, 3, 3, 6
    E, Pu, Pv, ids, logp = _lattice(g, M + K, k, V, scale=1.5)
    logits = g.standard_normal((M + K, V)) * 1.5
    counts = _simulate(M, K, None, (E, Pu, Pv, ids, logp, logits), anchor=2, n=40000, seed=0)
    p = np.exp(logits[0] - logits[0].max())
    p /= p.sum()
    assert not chi2_ok(counts[0], p)[0]
    monkeypatch.setattr(oracle, "accept_sample_request", orig)


# ---------------------------------------------------------------- context-gated greedy selector

def test_gated_greedy_hand_fixture():
    import json
    import os
    fx = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "selector_gate_hand.json")))
    path, score, margin = oracle.select_greedy_request(
        np.array(fx["embed"]), np.array(fx["P_u"]), np.array(fx["P_v"]), np.array(fx["W_H"]),
        np.array(fx["hidden"]), fx["anchor"], np.array(fx["ids"]), np.array(fx["logp"]),
        with_margin=True)
    assert list(path) == fx["expected_path"]
    assert score == pytest.approx(fx["expected_score"], abs=1e-12)
    assert margin == pytest.approx(fx["expected_margin"], abs=1e-12)


def test_gated_greedy_single_step_equals_viterbi_with_open_gate():
    """One draft position and a gate saturated open: the greedy step is the
    best path, which the brute-force-pinned Viterbi finds."""
    g = np.random.default_rng(8)
    for trial in range(20):
        E, Pu, Pv, ids, logp = _lattice(g, 1, 16, 40, D=6, r=4)
        Wh = np.full((4, 6), 0.0)
        Wh[:, 0] = 80.0
        h = np.zeros((1, 6))
        h[0, 0] = 1.0
        pg, sg = oracle.select_greedy_request(E, Pu, Pv, Wh, h, 5, ids, logp)
        pv, sv = oracle.select_path_request(E, Pu, Pv, 5, ids, logp)
        assert list(pg) == list(pv) and sg == pytest.approx(sv, rel=1e-12, abs=1e-12)


def test_gated_greedy_without_pair_term_is_per_position_argmax():
    g = np.random.default_rng(9)
    E, _, _, ids, logp = _lattice(g, 5, 8, 60, D=6, r=4)
    Z = np.zeros((4, 6))
    path, _ = oracle.select_greedy_request(E, Z, Z, g.standard_normal((4, 6)),
                                           g.standard_normal((5, 6)), 3, ids, logp)
    np.testing.assert_array_equal(path, [ids[t][int(np.argmax(logp[t]))] for t in range(5)])


def test_gated_greedy_never_beats_viterbi_with_open_gate():
    """Viterbi maximises the summed pair scores; the greedy walk's total can only
    match or trail it (gate saturated open, so both score the same function)."""
    g = np.random.default_rng(10)
    for trial in range(20):
        E, Pu, Pv, ids, logp = _lattice(g, 4, 4, 30, D=6, r=4)
        Wh = np.zeros((4, 6))
        Wh[:, 0] = 80.0
        h = np.zeros((4, 6))
        h[:, 0] = 1.0
        _, sg = oracle.select_greedy_request(E, Pu, Pv, Wh, h, 1, ids, logp)
        _, sv = oracle.select_path_request(E, Pu, Pv, 1, ids, logp)
        assert sg <= sv + 1e-12
