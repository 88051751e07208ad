"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.

Tolerances (written here, derived from the storage contract): logits within
2e-2 of the row maximum for bf16 storage, 1e-3 for the float32 configuration,
against both the oracle that rounds at the same storage points and the one
that rounds nowhere; top-k ids, selected paths and accepted lengths bit-exact
wherever the oracle's decision margin exceeds 1e-2."""

import numpy as np
import pytest

import oracle
import synth
from _cases import Case, rowmax_rel, topk_compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = {"bf16": 2e-2, "f32": 1e-3}
KV_TOL = {"bf16": 1.6e-2, "f32": 1e-4}

CASES = [
    # name, B, K, ctx lengths, preset overrides
    ("tiny", 1, 8, [64], {}),
    ("tiny_bf16", 1, 8, [64], {}),
    ("tiny_bf16", 3, 8, [5, 90, 64], {}),
    ("small", 2, 16, [130, 7], {}),
    ("small_gqa", 2, 8, [200, 129], {}),
    ("tiny_bf16", 1, 32, [1], {}),
    ("small", 1, 2, [96], {}),
    ("tiny_bf16", 9, 8, [70, 3, 64, 0, 200, 17, 64, 65, 9], {}),   # two 64-row conv tiles
    ("tiny_bf16", 2, 12, [40, 77], {}),                            # K does not divide 64
    # one channel per conv gate correction (a full 2D x D gate linear): the fused
    # conv (8 rows), the GEMM + row-kernel conv (24 rows), the float32 conv
    ("tiny_bf16", 1, 8, [64], {"conv_group": 1}),
    ("tiny_bf16", 3, 8, [5, 90, 64], {"conv_group": 1}),
    ("tiny", 1, 8, [64], {"conv_group": 1}),
    # 256 channels a conv CTA at 16 rows: the post conv writes no sums of squares and
    # the pre conv forms its own through the cluster
    ("small_gqa", 2, 8, [200, 129], {"conv_group": 128}),
    # 80 requests (640 block rows): one key split per (request, kv head), the attention's
    # single-split form; ragged contexts 5..403 around the 128-token window; the lm_head
    # over 560 draft rows on two-SM tiles with an odd weight-tile count (71: the last
    # pair's second tile is a phantom)
    ("small_gqa", 80, 8, [5 + (37 * i) % 400 for i in range(80)], {}),
    # 140 draft rows: the lm_head on two-SM tiles, 40 weight tiles with a partial last one
    ("small", 20, 8, [3 + (29 * i) % 150 for i in range(20)], {}),
    # 129 draft rows, the fewest that take the two-SM lm_head (one 256-token tile, one real
    # row in its second half)
    ("tiny_bf16", 43, 4, [(11 * i) % 70 for i in range(43)], {}),
]


def _case_id(c):
    name, B, K, _, over = c
    return f"{name}-B{B}-K{K}" + "".join(f"-{k}{v}" for k, v in over.items())


_made = {}


# Every case runs the cycle both ways: the injection inside the draft pass
# (draft_block_inject: each layer's QKV projection also forms the injected rows'
# K/V) and as two calls (inject_context, then draft_block).  The oracle is the
# same for both.
@pytest.fixture(scope="module", params=[(c, f) for c in CASES for f in (True, False)],
                ids=lambda p: _case_id(p[0]) + ("-fused" if p[1] else "-two_calls"))
def case(request):
    spec, fused = request.param
    name, B, K, ctx, over = spec
    key = _case_id(spec)
    if key not in _made:
        _made.clear()
        _made[key] = Case(name, B, K, ctx, seed=len(ctx) + K, **over)
    c = _made[key].device()
    c.g = c.run_device(fused=fused)
    return c


def test_device_status_clean(case):
    assert case.g["status"] == 0


def test_inject_kv_matches_oracle(case):
    ok, ov = case.oracle()["ck"], case.oracle()["cv"]
    gk, gv = case.gpu_kv_dense()
    tol = KV_TOL[case.cfg["dtype"]]
    for b in range(case.B):
        for l in range(case.cfg["n_layers"]):
            if case.ctx[b] == 0:
                continue
            assert rowmax_rel(gk[b][l], ok[b][l]) < tol, (b, l)
            assert rowmax_rel(gv[b][l], ov[b][l]) < tol, (b, l)


def test_logits_within_tolerance(case):
    o = case.oracle()
    err = rowmax_rel(case.g["logits"], o["logits"])
    assert err < TOL[case.cfg["dtype"]], err


def test_logits_within_tolerance_of_unrounded_oracle(case):
    """The same tolerance against the oracle that keeps float64 at every storage
    point (the device stores bf16 or float32 there)."""
    err = rowmax_rel(case.g["logits"], case.oracle_pure_logits())
    assert err < TOL[case.cfg["dtype"]], err


def test_topk_bitexact_above_margin(case):
    o = case.oracle()
    compared, bad = topk_compare(case.g["ids"], o["logits"], o["ids"], case.cfg["top_k"])
    assert compared > 0
    assert bad == 0, f"{bad} of {compared} ranks differ"
    # log-probabilities at matching ids
    same = case.g["ids"] == o["ids"]
    assert np.max(np.abs(case.g["logp"] - o["logp"])[same]) < 5e-2


def test_topk_exact_on_own_logits(case):
    """The device top-k is exactly the top-k (larger logit, then lower id) of the
    device's own logits, with logp = z - logsumexp(z)."""
    k = case.cfg["top_k"]
    z = case.g["logits"].reshape(-1, case.cfg["vocab"])
    ids = case.g["ids"].reshape(-1, k)
    lp = case.g["logp"].reshape(-1, k)
    for r in range(z.shape[0]):
        want, wlp, _ = oracle.topk_logp(z[r], k)
        np.testing.assert_array_equal(ids[r], want)
        np.testing.assert_allclose(lp[r], wlp, atol=2e-5)


def test_select_path_on_oracle_candidates(case):
    """The selector alone: the oracle's candidates in, path out."""
    import block_diffusion_drafter_inject_gb300 as dfl
    o = case.oracle()
    ids = torch.from_numpy(o["ids"]).cuda()
    logp = torch.from_numpy(o["logp"].astype(np.float32)).cuda()
    path = torch.zeros((case.B, case.K - 1), dtype=torch.int32, device="cuda")
    score = torch.zeros((case.B,), dtype=torch.float32, device="cuda")
    dfl.select_path(case.cfg, case.Wd, case.d_anchor, ids, logp, case.K, case.cyc.ws, path, score)
    torch.cuda.synchronize()
    path, score = path.cpu().numpy(), score.cpu().numpy()
    for b in range(case.B):
        if o["margin"][b] > 1e-2:
            assert list(path[b]) == list(o["path"][b]), b
        assert abs(score[b] - o["score"][b]) < 1e-3 * max(1.0, abs(o["score"][b])), b


def test_end_to_end_path_and_accept(case):
    o = case.oracle()
    g = case.g
    for b in range(case.B):
        same_lattice = np.array_equal(g["ids"][b], o["ids"][b])
        if same_lattice and o["margin"][b] > 1e-2:
            assert list(g["path"][b]) == list(o["path"][b]), b
    # acceptance on the device's own path equals the oracle's rule on that path
    acc, toks = oracle.accept_greedy(g["path"], case.target)
    np.testing.assert_array_equal(g["acc"], acc)
    np.testing.assert_array_equal(g["toks"], toks)


@pytest.mark.parametrize("pattern", ["all_equal", "five_levels"])
def test_topk_heavy_ties(pattern):
    """Logits with massive ties (lm_head rows zero, or repeating in five classes):
    the device top-k must still be the lowest ids among the largest values."""
    c = Case("small", 1, 8, [40], seed=21)
    V = c.cfg["vocab"]
    if pattern == "all_equal":
        c.W["lm_head"] = np.zeros_like(c.W["lm_head"])
    else:
        rows = c.W["lm_head"][1:6].copy()
        c.W["lm_head"] = rows[np.arange(V) % 5]
    c.device()
    g = c.run_device()
    k = c.cfg["top_k"]
    z = g["logits"].reshape(-1, V)
    for r in range(z.shape[0]):
        want, wlp, _ = oracle.topk_logp(z[r], k)
        np.testing.assert_array_equal(g["ids"].reshape(-1, k)[r], want)
        np.testing.assert_allclose(g["logp"].reshape(-1, k)[r], wlp, atol=2e-5)
    if pattern == "all_equal":
        np.testing.assert_array_equal(g["ids"][0, 0], np.arange(k))


@pytest.mark.parametrize("window", [1050, 1200])
@pytest.mark.parametrize("name", ["tiny", "tiny_bf16"])
def test_long_window_leftover_keys(name, window):
    """A window of more than 16 key tiles: the attention's key splits are capped
    at 16 (one thread-block cluster).  1050 + 8 keys: 16 splits of 64 keys and
    the last also takes the 34 left over; 1200 + 8: more than a split's worth
    would be left over, so the splits widen instead.  Logits still match the
    oracle."""
    c = Case(name, 1, 8, [1300], seed=5, window=window).device()
    g = c.run_device()
    assert g["status"] == 0
    err = rowmax_rel(g["logits"], c.oracle()["logits"])
    assert err < TOL[c.cfg["dtype"]], err


def test_page_size_not_64():
    """Pages of 16 positions: the attention copies key rows in 16-byte chunks
    instead of whole pages; logits still match the oracle."""
    c = Case("small", 2, 8, [150, 37], seed=6, page_size=16).device()
    g = c.run_device()
    assert g["status"] == 0
    err = rowmax_rel(g["logits"], c.oracle()["logits"])
    assert err < TOL["bf16"], err


@pytest.mark.parametrize("name", ["tiny", "tiny_bf16", "small"])
def test_selector_table_is_the_projection_of_every_row(name):
    """dflash_prepare_selector: table[0][v] = P_u e_v and table[1][v] = P_v e_v,
    against the fp64 products of the same stored values (the projections the
    oracle's selector forms), on sampled vocabulary rows including the ends."""
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case(name, 1, 8, [64], seed=11).device()
    tab = dfl.prepare_selector(c.cfg, c.Wd, c.cyc.ws)
    torch.cuda.synchronize()
    assert dfl.read_device_status(c.cyc.ws) == 0
    tab = tab.cpu().numpy().astype(np.float64)
    V = c.cfg["vocab"]
    rows = np.unique(np.concatenate([[0, 1, V - 2, V - 1], np.random.default_rng(3).integers(0, V, 64)]))
    E = c.W["embed"][rows].astype(np.float64)
    for side, P in ((0, c.W["sel_pu"]), (1, c.W["sel_pv"])):
        want = E @ P.astype(np.float64).T
        err = np.abs(tab[side][rows] - want).max() / np.abs(want).max()
        assert err < (1e-5 if c.cfg["dtype"] == "f32" else 1e-4), (side, err)


@pytest.mark.parametrize("B,K", [(1, 8), (3, 8), (2, 16)])
def test_select_path_with_table_on_oracle_candidates(B, K):
    """The selector reading candidate rows from the prepared table: the same
    paths as the oracle wherever its margin exceeds 1e-2, scores within 1e-3."""
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case("small", B, K, [60 + 17 * b for b in range(B)], seed=4 + B).device()
    dfl.prepare_selector(c.cfg, c.Wd, c.cyc.ws)
    o = c.oracle()
    ids = torch.from_numpy(o["ids"]).cuda()
    logp = torch.from_numpy(o["logp"].astype(np.float32)).cuda()
    path = torch.zeros((B, K - 1), dtype=torch.int32, device="cuda")
    score = torch.zeros((B,), dtype=torch.float32, device="cuda")
    dfl.select_path(c.cfg, c.Wd, c.d_anchor, ids, logp, K, c.cyc.ws, path, score)
    torch.cuda.synchronize()
    assert dfl.read_device_status(c.cyc.ws) == 0
    path, score = path.cpu().numpy(), score.cpu().numpy()
    for b in range(B):
        if o["margin"][b] > 1e-2:
            assert list(path[b]) == list(o["path"][b]), b
        assert abs(score[b] - o["score"][b]) < 1e-3 * max(1.0, abs(o["score"][b])), b


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("noalloc", [False, True])
def test_accept_nan_rows(dtype, noalloc):
    """Acceptance on target rows holding NaN: a row's first NaN is its argmax (NaN
    ranks above every number), the rule of the oracle (numpy's argmax)."""
    import block_diffusion_drafter_inject_gb300 as dfl
    B, K, V = 3, 4, 20000
    g = np.random.default_rng(7)
    T = g.standard_normal((B, K, V)).astype(np.float32)
    T[0, 0, 12345] = np.nan                 # a NaN beats the row's maximum
    T[0, 1, :] = np.nan                     # all NaN: id 0
    T[1, 0, 19999] = np.nan                 # NaN in the last chunk
    T[1, 0, 9000] = np.nan                  # ... and an earlier one in another chunk
    T[2, 2, 5] = np.inf                     # +inf is a number, NaN still wins
    T[2, 2, 7] = np.nan
    tt = torch.from_numpy(T).cuda()
    if dtype == "bf16":
        tt = tt.to(torch.bfloat16)
        T = tt.float().cpu().numpy()
    # paths that follow the argmax where it is defined by a NaN
    path = np.stack([[int(np.argmax(T[b, i])) for i in range(K - 1)] for b in range(B)])
    path[2, 2] = 0                          # request 2 stops at its third draft
    want_acc, want_tok = oracle.accept_greedy(path.astype(np.int32), T)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    d_path = torch.from_numpy(path.astype(np.int32)).cuda()
    if noalloc:
        dfl.accept_greedy_noalloc(d_path, tt, acc, tok)
    else:
        cfg = synth.preset("tiny_bf16")
        dfl.accept_greedy(d_path, tt, dfl.Workspace(cfg, B, K, 1), acc, tok)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), want_acc)
    np.testing.assert_array_equal(tok.cpu().numpy(), want_tok)
    assert list(want_tok[0][:2]) == [12345, 0] and want_tok[1][0] == 9000


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("V", [20001, 8199, 8192])
def test_accept_unaligned_rows_and_ties(dtype, V):
    """Acceptance's argmax on rows that are not 16-byte aligned (V not a multiple
    of the 16-byte word: those rows take the element-wise path) and on a ragged
    last chunk, with ties (the lower id wins) and a NaN (it wins), against the
    oracle's rule."""
    import block_diffusion_drafter_inject_gb300 as dfl
    B, K = 2, 5
    g = np.random.default_rng(V)
    T = g.standard_normal((B, K, V)).astype(np.float32)
    T[0, 0, [17, V - 1]] = 9.0               # tie across chunks: id 17
    T[0, 1, [V - 2, V - 1]] = 9.0            # tie inside the ragged tail: V - 2
    T[1, 0, 8191] = 9.0                      # last element of the first chunk
    T[1, 0, 8192 % V] = 9.0                  # ... tied with the next chunk's first (or itself)
    T[1, 3, V // 2] = np.nan
    tt = torch.from_numpy(T).cuda()
    if dtype == "bf16":
        tt = tt.to(torch.bfloat16)
        T = tt.float().cpu().numpy()
    path = np.stack([[int(np.argmax(T[b, i])) for i in range(K - 1)] for b in range(B)])
    path[1, 2] = (path[1, 2] + 1) % V        # request 1 stops at its third draft
    want_acc, want_tok = oracle.accept_greedy(path.astype(np.int32), T)
    acc = torch.zeros(B, dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    cfg = synth.preset("tiny_bf16")
    dfl.accept_greedy(torch.from_numpy(path.astype(np.int32)).cuda(), tt,
                      dfl.Workspace(cfg, B, K, 1), acc, tok)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(acc.cpu().numpy(), want_acc)
    np.testing.assert_array_equal(tok.cpu().numpy(), want_tok)
    assert want_tok[0][0] == 17 and want_acc[1] == 3


@pytest.mark.parametrize("name,ctx,tail", [
    ("tiny_bf16", [70, 5, 130], [7, 0, 3]),
    ("small_gqa", [200, 129], [1, 8]),
    ("tiny_bf16", [40, 64, 9, 100], [8, 8, 8, 8]),
    ("tiny", [64, 33], [8, 2]),     # float32 storage: the two calls in sequence
])
def test_fused_tail_after_prefill(name, ctx, tail):
    """The serving cycle: each request's context up to its last tail[b] rows is
    injected beforehand and those last rows by the draft pass itself
    (draft_block_inject, the rows' K/V formed in each layer's QKV projection and
    attended in the same pass).  Cache rows, logits and top-k as the oracle's,
    which injects every row and then drafts."""
    c = Case(name, len(ctx), 8, ctx, seed=31).device()
    g = c.run_device(fused=True, tail=tail)
    assert g["status"] == 0
    o = c.oracle()
    gk, gv = c.gpu_kv_dense()
    tol = KV_TOL[c.cfg["dtype"]]
    for b in range(c.B):
        for l in range(c.cfg["n_layers"]):
            assert rowmax_rel(gk[b][l], o["ck"][b][l]) < tol, (b, l)
            assert rowmax_rel(gv[b][l], o["cv"][b][l]) < tol, (b, l)
    err = rowmax_rel(g["logits"], o["logits"])
    assert err < TOL[c.cfg["dtype"]], err
    compared, bad = topk_compare(g["ids"], o["logits"], o["ids"], c.cfg["top_k"])
    assert compared > 0 and bad == 0, (compared, bad)


@pytest.mark.parametrize("fused", [True, False])
def test_injected_rows_failing_device_checks_are_skipped(fused):
    """Rows whose request row, position or page fails the device checks set their
    status bits and are skipped; the rest of the cycle is unaffected (logits as the
    oracle's on the valid context)."""
    import block_diffusion_drafter_inject_gb300 as dfl
    c = Case("tiny_bf16", 2, 8, [40, 200], seed=9).device()
    dfl.inject_context(c.cfg, c.Wd, c.kv, c.d_hidden, c.d_req, c.d_pos, c.cyc.ws)
    P = c.cfg["page_size"]
    assert c.table[0, 1] == -1 and c.table.shape[1] == 4
    # request row 2 of 2; position beyond request 0's 4-page table; page entry -1
    req = torch.tensor([2, 0, 0], dtype=torch.int32, device="cuda")
    pos = torch.tensor([10, 4 * P + 3, P + 36], dtype=torch.int32, device="cuda")
    hid = c.d_hidden[:3].clone()
    if fused:
        dfl.draft_block_inject(c.cfg, c.Wd, c.kv, hid, req, pos, c.d_anchor, c.d_ctx, c.K,
                               c.cyc.ws, c.cyc.topk_ids, c.cyc.topk_logp, c.d_logits)
    else:
        dfl.inject_context(c.cfg, c.Wd, c.kv, hid, req, pos, c.cyc.ws)
        dfl.draft_block(c.cfg, c.Wd, c.kv, c.d_anchor, c.d_ctx, c.K, c.cyc.ws, c.cyc.topk_ids,
                        c.cyc.topk_logp, c.d_logits)
    torch.cuda.synchronize()
    want = dfl.DEV_REQ_RANGE | dfl.DEV_POS_RANGE | dfl.DEV_PAGE_RANGE
    assert dfl.read_device_status(c.cyc.ws) == want
    err = rowmax_rel(c.d_logits.cpu().numpy(), c.oracle()["logits"])
    assert err < TOL["bf16"], err
