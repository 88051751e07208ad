"""GPU parity of the sampling walk and the speculative rejection sampler
(dflash_sample_path, dflash_accept_sample) against the oracle on the same
inputs and the same uniforms, and a Monte-Carlo check on the device that the
first committed token follows the target's distribution.

Decisions depend on where a uniform falls against running sums of
probabilities, which the device forms in float32 and the oracle in float64:
they are compared bit-exactly where the oracle's margin exceeds 1e-4 (relative
to the total being cut), and a walk is compared up to its first step inside
that margin.  Proposal probabilities q agree within 1e-5."""

import numpy as np
import pytest
from scipy.stats import chi2

import oracle
import synth
from _cases import Case

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

MARGIN = 1e-4


def draw_margin(weights, u):
    """Distance of u*W from the nearest running-sum boundary, relative to W."""
    c = np.cumsum(np.asarray(weights, dtype=np.float64))
    x = u * c[-1]
    return float(np.min(np.abs(np.concatenate([[0.0], c]) - x)) / c[-1])


def _uniforms(shape, seed):
    return np.random.default_rng(seed).random(shape).astype(np.float32).astype(np.float64)


@pytest.mark.parametrize("name,B,K,table", [("tiny_bf16", 3, 8, False), ("small", 2, 16, True),
                                             ("small", 4, 8, False), ("tiny", 2, 8, False)])
def test_sample_path_matches_oracle(name, B, K, table):
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case(name, B, K, [40 + 13 * b for b in range(B)], seed=30 + B + K).device()
    if table:
        dfl.prepare_selector(c.cfg, c.Wd, c.cyc.ws)
    o = c.oracle()
    k = c.cfg["top_k"]
    uw = _uniforms((B, K - 1), seed=K)
    path_o, q_o = oracle.sample_path(c.cfg, c.W, c.anchor, o["ids"], o["logp"], uw)
    path = torch.zeros((B, K - 1), dtype=torch.int32, device="cuda")
    pq = torch.zeros((B, K - 1, k), dtype=torch.float32, device="cuda")
    dfl.sample_path(c.cfg, c.Wd, c.d_anchor, torch.from_numpy(o["ids"]).cuda(),
                    torch.from_numpy(o["logp"].astype(np.float32)).cuda(), K,
                    torch.from_numpy(uw.astype(np.float32)).cuda(), c.cyc.ws, path, pq)
    torch.cuda.synchronize()
    assert dfl.read_device_status(c.cyc.ws) == 0
    path, pq = path.cpu().numpy(), pq.cpu().numpy()
    compared = 0
    for b in range(B):
        for t in range(K - 1):
            np.testing.assert_allclose(pq[b, t], q_o[b, t], atol=1e-5, err_msg=f"{b} {t}")
            if draw_margin(q_o[b, t], uw[b, t]) <= MARGIN:
                break                          # later steps follow another predecessor
            assert path[b, t] == path_o[b, t], (b, t)
            compared += 1
    assert compared >= B


def _accept_inputs(c, K, seed):
    """The oracle's sampled path and proposals, and target logits in which the
    drafted tokens are likely up to a per-request length (so that acceptance,
    rejection and the bonus draw all occur)."""
    o = c.oracle()
    B = c.B
    uw = _uniforms((B, K - 1), seed=seed)
    path, q = oracle.sample_path(c.cfg, c.W, c.anchor, o["ids"], o["logp"], uw)
    g = np.random.default_rng(seed)
    T = synth.make_target_logits(c.cfg, B, K, seed=seed).astype(np.float64)
    lens = g.integers(1, K + 1, size=B)
    for b in range(B):
        for i in range(lens[b] - 1):
            T[b, i, path[b, i]] = T[b, i].max() + 6.0
    return o, path, q, T.astype(np.float32)


def _accept_margins_ok(path, cand, q, T, u):
    """True when every decision the oracle takes for this request lies outside
    the margin (acceptance tests and the final draw)."""
    T = T.astype(np.float64)
    K = T.shape[0]
    for i in range(K - 1):
        p = np.exp(T[i] - T[i].max())
        p /= p.sum()
        qi = np.zeros_like(p)
        for j, cid in enumerate(cand[i]):
            qi[cid] += q[i][j]
        x = path[i]
        a, bnd = u[i, 0] * qi[x], p[x]
        if abs(a - bnd) <= MARGIN * max(a, bnd, 1e-30):
            return False
        if not a < bnd:
            r = np.maximum(p - qi, 0)
            return draw_margin(r if r.sum() > 0 else p, u[i, 1]) > MARGIN
    p = np.exp(T[K - 1] - T[K - 1].max())
    return draw_margin(p / p.sum(), u[K - 1, 1]) > MARGIN


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("name,B,K", [("tiny_bf16", 6, 8), ("small", 4, 16)])
def test_accept_sample_matches_oracle(name, B, K, dtype):
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case(name, B, K, [30 + 7 * b for b in range(B)], seed=50 + B).device()
    o, path, q, T = _accept_inputs(c, K, seed=K + B)
    tt = torch.from_numpy(T).cuda()
    if dtype == "bf16":
        tt = tt.to(torch.bfloat16)
        T = tt.float().cpu().numpy()
    u = _uniforms((B, K, 2), seed=7 + K)
    acc_o, tok_o = oracle.accept_sample(path, o["ids"], q, T, u)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    dfl.accept_sample(torch.from_numpy(path).cuda(), torch.from_numpy(o["ids"]).cuda(),
                      torch.from_numpy(q.astype(np.float32)).cuda(), tt,
                      torch.from_numpy(u.astype(np.float32)).cuda(), c.cyc.ws, acc, tok)
    torch.cuda.synchronize()
    acc, tok = acc.cpu().numpy(), tok.cpu().numpy()
    compared = 0
    for b in range(B):
        if _accept_margins_ok(path[b], o["ids"][b], q[b], T[b], u[b]):
            assert acc[b] == acc_o[b], b
            np.testing.assert_array_equal(tok[b], tok_o[b])
            compared += 1
    assert compared >= B // 2
    assert len(set(acc_o.tolist())) > 1          # several accepted lengths occur


def test_accept_sample_is_lossless_on_device():
    """8192 copies of one request, each with its own uniforms, through the device
    walk and the device rejection sampler: the first committed token must follow
    p_0 = softmax(target row 0) (chi-square over the 40 likeliest tokens and the
    rest, p-value 1e-4), whatever the drafter proposed."""
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case("tiny_bf16", 1, 4, [50], seed=77).device()
    o = c.oracle()
    k, V, K = c.cfg["top_k"], c.cfg["vocab"], 4
    N = 8192
    g = np.random.default_rng(5)
    T = g.standard_normal((K, V)) * 1.0
    for i in range(K - 1):                      # the drafter's candidates are plausible
        T[i, o["ids"][0, i]] += 3.0 + g.random(k)
    ids = np.tile(o["ids"], (N, 1, 1))
    logp = np.tile(o["logp"].astype(np.float32), (N, 1, 1))
    anchor = np.full(N, c.anchor[0], dtype=np.int32)
    ws = dfl.Workspace(c.cfg, N, K, 1)
    path = torch.zeros((N, K - 1), dtype=torch.int32, device="cuda")
    pq = torch.zeros((N, K - 1, k), dtype=torch.float32, device="cuda")
    dfl.sample_path(c.cfg, c.Wd, torch.from_numpy(anchor).cuda(), torch.from_numpy(ids).cuda(),
                    torch.from_numpy(logp).cuda(), K,
                    torch.from_numpy(g.random((N, K - 1)).astype(np.float32)).cuda(), ws, path,
                    pq)
    acc = torch.zeros(N, dtype=torch.int32, device="cuda")
    tok = torch.zeros((N, K), dtype=torch.int32, device="cuda")
    dfl.accept_sample(path, torch.from_numpy(ids).cuda(), pq,
                      torch.from_numpy(np.tile(T.astype(np.float32), (N, 1, 1))).cuda(),
                      torch.from_numpy(g.random((N, K, 2)).astype(np.float32)).cuda(), ws, acc,
                      tok)
    torch.cuda.synchronize()
    assert dfl.read_device_status(ws) == 0
    first = tok[:, 0].cpu().numpy()
    p = np.exp(T[0] - T[0].max())
    p /= p.sum()
    top = np.argsort(-p)[:40]
    counts = np.array([np.sum(first == v) for v in top] + [np.sum(~np.isin(first, top))], float)
    expect = N * np.concatenate([p[top], [1.0 - p[top].sum()]])
    stat = float(np.sum((counts - expect) ** 2 / expect))
    assert stat <= chi2.ppf(1.0 - 1e-4, len(counts) - 1), stat
    a = acc.cpu().numpy()
    assert a.min() == 1 and len(set(a.tolist())) >= 3   # rejections and several accepted lengths


@pytest.mark.parametrize("name,B,K,table", [("tiny_bf16", 3, 8, False), ("small", 2, 16, True),
                                             ("tiny", 2, 8, False), ("small_gqa", 2, 8, True)])
def test_select_greedy_matches_oracle(name, B, K, table):
    """The context-gated greedy walk on the oracle's candidates and hidden states:
    each path bit-exact up to its first step whose gap (best minus runner-up
    score) is 1e-2 or less, and the score within 1e-3 where no step is."""
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case(name, B, K, [40 + 9 * b for b in range(B)], seed=60 + B + K).device()
    if table:
        dfl.prepare_selector(c.cfg, c.Wd, c.cyc.ws)
    o = c.oracle()
    path_o, score_o, margin_o = oracle.select_greedy(c.cfg, c.W, c.anchor, o["ids"], o["logp"],
                                                     o["zf"])
    dt = torch.bfloat16 if c.cfg["dtype"] == "bf16" else torch.float32
    hidden = torch.from_numpy(o["zf"].astype(np.float32)).to(dt).cuda()
    path = torch.zeros((B, K - 1), dtype=torch.int32, device="cuda")
    score = torch.zeros(B, dtype=torch.float32, device="cuda")
    dfl.select_greedy(c.cfg, c.Wd, c.d_anchor, torch.from_numpy(o["ids"]).cuda(),
                      torch.from_numpy(o["logp"].astype(np.float32)).cuda(), hidden, K, c.cyc.ws,
                      path, score)
    torch.cuda.synchronize()
    assert dfl.read_device_status(c.cyc.ws) == 0
    path, score = path.cpu().numpy(), score.cpu().numpy()
    compared = 0
    for b in range(B):
        _, _, gaps = oracle.select_greedy_request(
            c.W["embed"], c.W["sel_pu"], c.W["sel_pv"], c.W["sel_gate"], o["zf"][b], c.anchor[b],
            o["ids"][b], o["logp"][b], with_margin=True, step_margins=True)
        for t in range(K - 1):
            if gaps[t] <= 1e-2:
                break                          # later steps follow another predecessor
            assert path[b, t] == path_o[b, t], (b, t)
            compared += 1
        if np.all(gaps > 1e-2):
            assert abs(score[b] - score_o[b]) < 1e-3 * max(1.0, abs(score_o[b])), b
    assert compared >= B


def test_draft_hidden_is_the_lm_head_input():
    """dflash_draft_hidden: the final-normed rows the draft pass left in the
    workspace match the oracle's (row-max relative, the logits' tolerance)."""
    import block_diffusion_drafter_inject_gb300 as dfl
    from _cases import rowmax_rel
    c = Case("small", 2, 8, [70, 33], seed=12).device()
    c.run_device()
    h = dfl.draft_hidden(c.cfg, c.B, c.K, c.cyc.ws).float().cpu().numpy()
    assert rowmax_rel(h, c.oracle()["zf"]) < 2e-2
