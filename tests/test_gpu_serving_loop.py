"""A serving loop on the device: consecutive fused cycles in which each cycle's
committed tokens become context (their target hidden states injected by the next
cycle's pass, dflash_draft_block_inject) and the bonus token the next anchor;
acceptance lengths vary per request and cycle.  Every cycle is checked against
the oracle run on the whole context so far (logits within the parity tolerance,
top-k ranks above the 1e-2 margin, acceptance exact on the device's path), and
at the end the paged cache against the oracle's injected K/V.  Covers the
cycle's state across calls: the workspace's tickets and status, the cache rows
written in earlier passes, ragged injections at shifting positions."""

import numpy as np
import pytest

import oracle
import synth
from _cases import rowmax_rel, topk_compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = {"bf16": 2e-2, "f32": 1e-3}
KV_TOL = {"bf16": 1.6e-2, "f32": 1e-4}


def _oracle_state(cfg, W, H, ctx, anchor, K):
    """The oracle's draft for context lengths ctx (rows 0..ctx-1 of H injected)."""
    L = cfg["n_layers"]
    ck, cv = [], []
    for b in range(len(ctx)):
        n = int(ctx[b])
        k, v, _ = oracle.inject_context(cfg, W, H[b][:n], np.arange(n), cfg["dtype"])
        ck.append([k[l] for l in range(L)])
        cv.append([v[l] for l in range(L)])
    d = oracle.draft_block(cfg, W, ck, cv, anchor, ctx, K, cfg["dtype"])
    return d, ck, cv


@pytest.mark.parametrize("name,bits", [("tiny_bf16", 0), ("small", 0), ("tiny", 0),
                                       ("tiny_bf16", 4)])
def test_serving_loop_matches_oracle(name, bits):
    import block_diffusion_drafter_inject_gb300 as dfl
    cfg = synth.preset(name, **({"weight_bits": 4} if bits else {}))
    B, K, cycles = 3, 8, 5
    W = synth.make_weights(cfg, seed=7, sel_scale=0.3)
    Q = None
    if bits:
        Q = synth.make_q4_weights(cfg, seed=7)
        W = oracle.quantized_weights(W, Q)
    ctx = np.array([20, 3, 47], dtype=np.int32)
    max_ctx = ctx + cycles * K
    H = [synth.make_hiddens(cfg, int(max_ctx[b]), seed=100 + b, name="loop_hiddens")
         for b in range(B)]
    table, npages = synth.make_paged_layout(max_ctx + K, cfg["page_size"], seed=7)
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    Wd = dfl.DeviceWeights.from_host(cfg, W, "cuda", q4=Q)
    kv = dfl.PagedKV(cfg, table, npages, "cuda")
    cyc = dfl.DraftCycle(cfg, Wd, kv, B, K, 128, "cuda")
    # prefill: rows 0..ctx-1 of every request, one inject call
    req = np.concatenate([np.full(int(ctx[b]), b, np.int32) for b in range(B)])
    pos = np.concatenate([np.arange(int(ctx[b]), dtype=np.int32) for b in range(B)])
    hid = np.concatenate([H[b][:int(ctx[b])] for b in range(B)])
    dfl.inject_context(cfg, Wd, kv, torch.from_numpy(hid).to(dt).cuda(),
                       torch.from_numpy(req).cuda(), torch.from_numpy(pos).cuda(), cyc.ws)
    rng = np.random.default_rng(11)
    anchor = synth.make_anchors(cfg, B, seed=11)
    pend_req = np.zeros(0, np.int32)
    pend_pos = np.zeros(0, np.int32)
    V = cfg["vocab"]
    logits = torch.zeros((B, K - 1, V), dtype=torch.float32, device="cuda")
    seen = set()
    for c in range(cycles):
        hid_new = (torch.from_numpy(np.stack([H[r][p] for r, p in zip(pend_req, pend_pos)]))
                   .to(dt).cuda() if len(pend_req) else None)
        d_anchor = torch.from_numpy(anchor).cuda()
        d_ctx = torch.from_numpy(ctx).cuda()
        dfl.draft_block_inject(cfg, Wd, kv, hid_new,
                               torch.from_numpy(pend_req).cuda() if len(pend_req) else None,
                               torch.from_numpy(pend_pos).cuda() if len(pend_req) else None,
                               d_anchor, d_ctx, K, cyc.ws, cyc.topk_ids, cyc.topk_logp, logits)
        dfl.select_path(cfg, Wd, d_anchor, cyc.topk_ids, cyc.topk_logp, K, cyc.ws, cyc.path,
                        cyc.score)
        torch.cuda.synchronize()
        path = cyc.path.cpu().numpy()
        # target logits that accept the first m_b drafts of request b
        T = synth.make_target_logits(cfg, B, K, seed=200 + c)
        m = rng.integers(0, K, size=B)
        for b in range(B):
            for i in range(K - 1):
                if i < m[b]:
                    T[b, i, path[b, i]] = T[b, i].max() + 5.0
                elif i == m[b]:
                    T[b, i, path[b, i]] = T[b, i].min() - 1.0
        dfl.accept_greedy(cyc.path, torch.from_numpy(T).cuda(), cyc.ws, cyc.accept_len,
                          cyc.tokens)
        torch.cuda.synchronize()
        assert dfl.read_device_status(cyc.ws) == 0
        acc, toks = cyc.accept_len.cpu().numpy(), cyc.tokens.cpu().numpy()
        acc_o, toks_o = oracle.accept_greedy(path, T)
        np.testing.assert_array_equal(acc, acc_o)
        np.testing.assert_array_equal(toks, toks_o)
        np.testing.assert_array_equal(acc, m + 1)
        seen.update(acc.tolist())
        # this cycle's pass against the oracle on the context so far
        d, ck, cv = _oracle_state(cfg, W, H, ctx, anchor, K)
        g_logits = logits.cpu().numpy().astype(np.float64)
        err = rowmax_rel(g_logits, d["logits"])
        assert err < TOL[cfg["dtype"]], (c, err)
        compared, bad = topk_compare(cyc.topk_ids.cpu().numpy(), d["logits"], d["ids"],
                                     cfg["top_k"])
        assert bad == 0, (c, bad, compared)
        # the committed tokens become context; the bonus token is the next anchor
        pend_req = np.concatenate([np.full(int(acc[b]), b, np.int32) for b in range(B)])
        pend_pos = np.concatenate([np.arange(int(ctx[b]), int(ctx[b]) + int(acc[b]),
                                             dtype=np.int32) for b in range(B)])
        ctx = ctx + acc.astype(np.int32)
        anchor = np.array([toks[b, acc[b] - 1] for b in range(B)], dtype=np.int32)
    assert len(seen) >= 3  # acceptance lengths varied
    # the cache holds every row injected so far (the last cycle's rows are still pending)
    done = ctx - acc.astype(np.int32)
    _, ck, cv = _oracle_state(cfg, W, H, done, anchor, K)
    k = kv.k.float().cpu().numpy()
    v = kv.v.float().cpu().numpy()
    P = cfg["page_size"]
    for b in range(B):
        p = np.arange(int(done[b]))
        pages = table[b, p // P]
        for l in range(cfg["n_layers"]):
            assert rowmax_rel(k[l][pages, :, p % P, :], ck[b][l]) < KV_TOL[cfg["dtype"]], (b, l)
            assert rowmax_rel(v[l][pages, :, p % P, :], cv[b][l]) < KV_TOL[cfg["dtype"]], (b, l)
