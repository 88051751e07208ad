"""Parity at the full drafter size (width 4096, 5 layers, vocab 151936), in the
launch configurations the benchmark uses: B=1 block 8 with 2048 context (and
with 2100, a window that starts mid-page, on the prepared selector table); B=1
block 16 with 8192 context (target logits built from the oracle's path so every
accepted length 1..16 occurs); B=32 ragged contexts in [512, 8192] on shuffled
64-token pages (oracle on a subset of requests, which the pass treats
independently); and a 4096-token injection sampled row by row.

Tolerances: injected K/V within bf16 resolution as in test_gpu_parity.  Logits,
measured row-max relative (max |g - o| / max |o| per row): at this width the bf16
storage contract is itself 2-3 % of the row maximum away from float64
arithmetic (the oracle alone shows it, request by request), so the device's
logits must lie within 2e-2 of the float64 oracle OR no further from it than
1.25 times the bf16-contract oracle is, for the same request, both row-max
relative and norm-wise per row; against the bf16-contract oracle they must lie
within twice the contract's measured sensitivity element-wise (see below).  Decisions: (a) bit-exact on identical
inputs - the top-k equals a full sort of the device's own logits, the selector
run on the oracle's candidates matches the oracle's path where its margin
exceeds 1e-2, acceptance on given logits matches exactly; (b) against the
oracle's own logits, top-k ranks are compared where the oracle's margin
exceeds twice the bf16 contract's measured sensitivity at this width
(tests/golden/contract_sensitivity.json: the oracle alone moves its logits by
that much when its pre-rounding values move by 1e-6)."""

import json
import os

import numpy as np
import pytest

import oracle
import synth
from _cases import FullCase, exact_logits, rowmax_rel, topk_compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BAND = 2.0 * json.load(open(os.path.join(GOLD, "contract_sensitivity.json")))["shift"]


def _check_request(case, b, kv_rows=64):
    import block_diffusion_drafter_inject_gb300 as dfl
    o = case.oracle()[b]
    k = case.cfg["top_k"]
    gk, gv = case.gpu_kv(b)
    rows = np.linspace(0, gk.shape[1] - 1, min(kv_rows, gk.shape[1])).astype(int)
    assert rowmax_rel(gk[:, rows], o["k"][:, rows]) < 1.6e-2
    assert rowmax_rel(gv[:, rows], o["v"][:, rows]) < 1.6e-2
    g_logits = case.d_logits[b].double().cpu().numpy()
    # full width: per-row norm-wise relative error within 2e-2, and no logit
    # further from the oracle than twice the contract's own sensitivity
    def normwise(a, ref):
        return float(np.max(np.linalg.norm(a - ref, axis=1) / np.linalg.norm(ref, axis=1)))

    rm = rowmax_rel(g_logits, o["logits"])
    rm_x = rowmax_rel(g_logits, o["logits_exact"])             # device vs float64
    rm_cx = rowmax_rel(o["logits"], o["logits_exact"])         # bf16 contract vs float64
    assert rm_x < max(2e-2, 1.25 * rm_cx), (rm_x, rm_cx)
    nw_x = normwise(g_logits, o["logits_exact"])
    nw_cx = normwise(o["logits"], o["logits_exact"])
    assert nw_x < max(2e-2, 1.25 * nw_cx), (nw_x, nw_cx)
    nrel = normwise(g_logits, o["logits"])                     # reported
    assert np.abs(g_logits - o["logits"]).max() < BAND
    g_ids = case.cyc.topk_ids[b].cpu().numpy()
    g_logp = case.cyc.topk_logp[b].cpu().numpy().astype(np.float64)
    # (a) exact: the device top-k is the top-k of its own logits
    for t in range(g_logits.shape[0]):
        ids, lp, _ = oracle.topk_logp(g_logits[t], k)
        np.testing.assert_array_equal(g_ids[t], ids)
        np.testing.assert_allclose(g_logp[t], lp, atol=2e-5)
    # (b) against the oracle's logits, outside the contract's sensitivity band
    compared, bad = topk_compare(g_ids, o["logits"], o["ids"], k, margin=BAND)
    top = np.take_along_axis(g_logits - o["logits"], o["ids"].astype(np.int64), axis=1)
    assert compared > 0
    assert bad == 0, f"{bad} of {compared}; max |err| at the oracle top-{k}: {np.abs(top).max():.2e}"
    # reported, not asserted: agreement where the oracle's margin exceeds 1e-2
    c01, b01 = topk_compare(g_ids, o["logits"], o["ids"], k, margin=1e-2)
    print(f"request {b}: logits row-max rel vs float64 {rm_x:.3e} (bf16 contract vs float64 "
          f"{rm_cx:.3e}), vs the bf16 contract {rm:.3e}; norm-wise vs float64 {nw_x:.3e} (contract "
          f"{nw_cx:.3e}), vs the bf16 contract {nrel:.3e}; top-{k} ranks "
          f"compared {compared} (margin {BAND:.3f}) all equal; at margin 1e-2 {c01 - b01} of {c01} "
          f"equal")
    # the selector on the oracle's candidates (no bf16 storage inside)
    ids = torch.from_numpy(o["ids"][None].astype(np.int32)).cuda()
    lp = torch.from_numpy(o["logp"][None].astype(np.float32)).cuda()
    path = torch.zeros((1, case.K - 1), dtype=torch.int32, device="cuda")
    score = torch.zeros((1,), dtype=torch.float32, device="cuda")
    dfl.select_path(case.cfg, case.Wd, case.d_anchor[b:b + 1], ids, lp, case.K, case.cyc.ws,
                    path, score)
    torch.cuda.synchronize()
    if o["margin"] > 1e-2:
        assert list(path.cpu().numpy()[0]) == list(o["path"])
    assert abs(float(score.cpu()[0]) - o["score"]) < 1e-3 * max(1.0, abs(o["score"]))
    return o


def test_full_b1_k8_ctx2048():
    case = FullCase(1, 8, [2048], seed=0).device()
    assert case.status == 0
    _check_request(case, 0)
    # the serving cycle: the last 8 context rows injected by the pass itself
    case.device(tail=[8])
    assert case.status == 0 and case.n_fused == 8
    _check_request(case, 0)


def test_full_q4_b1_k8_ctx2048():
    """The 4-bit drafter at full size (fc, QKV, O, gate/up, down, lm_head as codes
    with a bf16 scale and bias per 64 inputs): the serving cycle, the last 8
    context rows injected by the pass, against the oracle on the weights the codes
    stand for."""
    case = FullCase(1, 8, [2048], seed=3, q4=True).device(tail=[8])
    assert case.status == 0 and case.n_fused == 8
    _check_request(case, 0)


def test_full_b1_unaligned_window_with_selector_table():
    """Context 2100: the window starts mid-page, so it spans 17 cache pages and
    the last of the 16 key splits takes three tiles (two context pages and the
    block) through the split launch's two-stage ring; the selector reads the
    prepared table of all 151936 rows' projections."""
    case = FullCase(1, 8, [2100], seed=7).device(sel_table=True)
    assert case.status == 0
    _check_request(case, 0)


def test_full_b1_k16_ctx8192_every_accept_length():
    import block_diffusion_drafter_inject_gb300 as dfl
    case = FullCase(1, 16, [8192], seed=1).device()
    assert case.status == 0
    o = _check_request(case, 0)
    # target logits from the oracle's path: accept_len = L for L = 1..16
    K, V = 16, case.cfg["vocab"]
    base = synth.make_target_logits(case.cfg, K, K, seed=1)      # one row set per L
    T = np.zeros((K, K, V), np.float32)
    path = case.cyc.path.cpu().numpy()[0]
    for L in range(1, K + 1):
        t = base[L - 1].copy()
        for i in range(L - 1):
            t[i, path[i]] = t[i].max() + 5.0
        if L < K:
            t[L - 1, path[L - 1]] = t[L - 1].min()
        T[L - 1] = t
    acc_o, tok_o = oracle.accept_greedy(np.tile(path, (K, 1)), T)
    np.testing.assert_array_equal(acc_o, np.arange(1, K + 1))
    acc = torch.zeros(K, dtype=torch.int32, device="cuda")
    tok = torch.zeros((K, K), dtype=torch.int32, device="cuda")
    ws = dfl.Workspace(case.cfg, K, K, 1)
    dfl.accept_greedy(torch.from_numpy(np.tile(path, (K, 1))).cuda(), torch.from_numpy(T).cuda(),
                      ws, acc, tok)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), acc_o)
    np.testing.assert_array_equal(tok.cpu().numpy(), tok_o)
    del o


def test_full_b32_ragged_paged_subset():
    """B=32, the oracle on requests 0 and 19 and on the shortest and longest contexts."""
    ctx = synth.make_ctx_lens(32, 512, 8192, seed=2)
    reqs = sorted({0, 19, int(np.argmin(ctx)), int(np.argmax(ctx))})
    assert len(reqs) == 4
    case = FullCase(32, 8, ctx, seed=2, oracle_requests=reqs).device()
    assert case.status == 0
    for b in reqs:
        _check_request(case, b)
    # the same requests with the last 0..8 rows of each injected by the pass itself
    tail = synth.stream(2, "fused_tail").integers(0, 9, 32)
    tail[reqs[0]] = 0
    tail[reqs[1]] = 8
    case.device(tail=tail)
    assert case.status == 0 and case.n_fused == int(tail.sum())
    for b in reqs:
        _check_request(case, b)


def test_full_inject_4096_rows_sampled():
    import block_diffusion_drafter_inject_gb300 as dfl
    cfg = synth.preset("full")
    W = FullCase(1, 8, [64], seed=0).W                         # shared full weights
    N = 4096
    h = synth.make_hiddens(cfg, N, seed=3, name="inject_hiddens")
    P = cfg["page_size"]
    table = np.arange(N // P, dtype=np.int32)[None, :]
    Wd = dfl.DeviceWeights.from_host(cfg, W, "cuda")
    kv = dfl.PagedKV(cfg, table, N // P, "cuda")
    ws = dfl.Workspace(cfg, 1, 2, N)
    dfl.inject_context(cfg, Wd, kv, torch.from_numpy(h).to(torch.bfloat16).cuda(),
                       torch.zeros(N, dtype=torch.int32, device="cuda"),
                       torch.arange(N, dtype=torch.int32, device="cuda"), ws)
    torch.cuda.synchronize()
    assert dfl.read_device_status(ws) == 0
    rows = np.concatenate([np.random.default_rng(3).choice(N, 14, replace=False), [0, N - 1]])
    k, v, _ = oracle.inject_context(cfg, W, h[rows], rows, "bf16")
    pg = torch.from_numpy(rows // P).cuda()
    sl = torch.from_numpy(rows % P).cuda()
    gk = kv.k.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)      # [L, n, Hkv, d]
    gv = kv.v.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)
    assert rowmax_rel(gk.float().cpu().numpy(), k) < 1.6e-2
    assert rowmax_rel(gv.float().cpu().numpy(), v) < 1.6e-2


class _Config5:
    """8 requests each inject 4096 new target-hidden rows (5 x 5120 bf16) in ONE
    inject call (32768 rows, shuffled 64-token pages), then one block-16 cycle
    runs for all 8 (context 4096, window 1024).  Exposes what _check_request
    reads: the oracle on requests `oracle_requests` (their windows injected by the
    oracle), the device K/V at those windows, logits, top-k and selector."""

    def __init__(self, oracle_requests, B=8, n=4096, K=16):
        import block_diffusion_drafter_inject_gb300 as dfl
        self.cfg = cfg = synth.preset("full")
        self.W = FullCase(1, 8, [64], seed=0).W                # shared full weights
        self.B, self.K, self.n = B, K, n
        P, Wn = cfg["page_size"], cfg["window"]
        TIN = cfg["n_taps"] * cfg["d_target"]
        per = (n + K + P - 1) // P
        self.table = synth.stream(5, "c5_pages").permutation(B * per).astype(np.int32).reshape(B, per)
        self.Wd = dfl.DeviceWeights.from_host(cfg, self.W, "cuda")
        self.kv = dfl.PagedKV(cfg, self.table, B * per, "cuda")
        self.cyc = dfl.DraftCycle(cfg, self.Wd, self.kv, B, K, B * n, "cuda")
        hid = torch.empty((B * n, TIN), dtype=torch.bfloat16, device="cuda")
        self.host = {}
        self.lo = n - Wn
        self.oracle_requests = list(oracle_requests)
        rng = np.random.default_rng(5)
        self.sample_rows = {}
        for b in range(B):
            h = synth.make_hiddens(cfg, n, seed=50 + b, name="c5_hiddens")
            hid[b * n:(b + 1) * n] = torch.from_numpy(h).to(torch.bfloat16)
            rows = np.unique(np.concatenate([[0, n - 1], rng.choice(n, 6, replace=False)]))
            self.sample_rows[b] = (rows, h[rows].copy())
            if b in self.oracle_requests:
                self.host[b] = h[self.lo:].copy()
            del h
        req = torch.arange(B, dtype=torch.int32, device="cuda").repeat_interleave(n)
        pos = torch.arange(n, dtype=torch.int32, device="cuda").repeat(B)
        dfl.inject_context(cfg, self.Wd, self.kv, hid, req, pos, self.cyc.ws)   # one call
        del hid
        self.anchor = synth.make_anchors(cfg, B, seed=5)
        self.d_anchor = torch.from_numpy(self.anchor).cuda()
        self.d_ctx = torch.full((B,), n, dtype=torch.int32, device="cuda")
        self.d_logits = torch.zeros((B, K - 1, cfg["vocab"]), dtype=torch.float32, device="cuda")
        dfl.draft_block(cfg, self.Wd, self.kv, self.d_anchor, self.d_ctx, K, self.cyc.ws,
                        self.cyc.topk_ids, self.cyc.topk_logp, self.d_logits)
        dfl.select_path(cfg, self.Wd, self.d_anchor, self.cyc.topk_ids, self.cyc.topk_logp, K,
                        self.cyc.ws, self.cyc.path, self.cyc.score)
        torch.cuda.synchronize()
        self.status = dfl.read_device_status(self.cyc.ws)
        self._o = None

    def _gather(self, b, p):
        P = self.cfg["page_size"]
        pg = torch.from_numpy(self.table[b, p // P].astype(np.int64)).cuda()
        sl = torch.from_numpy((p % P).astype(np.int64)).cuda()
        k = self.kv.k.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)
        v = self.kv.v.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)
        return k.float().cpu().numpy(), v.float().cpu().numpy()

    def gpu_kv(self, b):
        return self._gather(b, np.arange(self.lo, self.n))

    def oracle(self):
        if self._o is None:
            cfg, L, K, n = self.cfg, self.cfg["n_layers"], self.K, self.n
            res = {}
            for b in self.oracle_requests:
                p = np.arange(self.lo, n)
                k, v, _ = oracle.inject_context(cfg, self.W, self.host[b], p, "bf16")
                shape = (n, cfg["n_kv_heads"], cfg["head_dim"])
                ck, cv = [], []
                for l in range(L):
                    a = np.zeros(shape)
                    a[p] = k[l]
                    ck.append(a)
                    a = np.zeros(shape)
                    a[p] = v[l]
                    cv.append(a)
                d = oracle.draft_block(cfg, self.W, [ck], [cv], self.anchor[b:b + 1], [n], K,
                                       "bf16")
                pth, sc, mg = oracle.select_path(cfg, self.W, self.anchor[b:b + 1], d["ids"],
                                                 d["logp"], with_margin=True)
                res[b] = dict(k=k, v=v, logits=d["logits"][0], ids=d["ids"][0],
                              logp=d["logp"][0], path=pth[0], score=sc[0], margin=mg[0],
                              logits_exact=exact_logits(cfg, self.W, self.host[b], p, n,
                                                        self.anchor[b], K))
            self._o = res
        return self._o


def test_full_inject_8x4096_rows_then_block16_cycle():
    """Context capture at scale: one inject call of 32768 rows for 8 requests, checked
    on sampled rows of every request; then one block-16 cycle for all 8, whose
    windows, logits, top-16 and selector match the oracle on two requests."""
    case = _Config5(oracle_requests=[0, 5])
    assert case.status == 0
    for b in range(case.B):
        rows, h = case.sample_rows[b]
        k, v, _ = oracle.inject_context(case.cfg, case.W, h, rows, "bf16")
        gk, gv = case._gather(b, rows)
        assert rowmax_rel(gk, k) < 1.6e-2, b
        assert rowmax_rel(gv, v) < 1.6e-2, b
    for b in case.oracle_requests:
        _check_request(case, b)
