"""Shared set-up for the GPU parity tests: seeded inputs (synth), the oracle's
expected values, and the same inputs on the device through the C ABI."""

import numpy as np

import oracle
import synth


class Case:
    """B requests with context lengths ctx[b], block K, on preset `name`."""

    def __init__(self, name, B, K, ctx, seed=0, sel_scale=0.3, shuffle=True, extra_pages=3,
                 **over):
        self.cfg = synth.preset(name, **over)
        self.B, self.K = B, K
        self.ctx = np.asarray(ctx, dtype=np.int32)
        self.seed = seed
        self.W = synth.make_weights(self.cfg, seed=seed, sel_scale=sel_scale)
        # 4-bit drafter: the device gets the codes, the oracle the weights they stand for
        self.Q = None
        if self.cfg.get("weight_bits", 0) == 4:
            self.Q = synth.make_q4_weights(self.cfg, seed=seed)
            self.W = oracle.quantized_weights(self.W, self.Q)
        self.contract = self.cfg["dtype"]
        ntot = int(self.ctx.sum())
        self.hidden = synth.make_hiddens(self.cfg, max(ntot, 1), seed=seed)[:ntot]
        self.req = np.concatenate([np.full(c, b, np.int32) for b, c in enumerate(self.ctx)])
        self.pos = np.concatenate([np.arange(c, dtype=np.int32) for c in self.ctx])
        self.anchor = synth.make_anchors(self.cfg, B, seed=seed)
        # room for the context plus the block (the block itself is never stored)
        self.table, self.num_pages = synth.make_paged_layout(
            self.ctx + K, self.cfg["page_size"], seed=seed, shuffle=shuffle,
            extra_pages=extra_pages)
        self.target = synth.make_target_logits(self.cfg, B, K, seed=seed)
        self._o = None

    # ---------------------------------------------------------------- oracle
    def oracle_inject(self):
        L = self.cfg["n_layers"]
        ck, cv = [], []
        o = 0
        for b in range(self.B):
            n = int(self.ctx[b])
            k, v, _ = oracle.inject_context(self.cfg, self.W, self.hidden[o:o + n],
                                            np.arange(n), self.contract)
            ck.append([k[l] for l in range(L)])
            cv.append([v[l] for l in range(L)])
            o += n
        return ck, cv

    def oracle(self):
        if self._o is None:
            ck, cv = self.oracle_inject()
            d = oracle.draft_block(self.cfg, self.W, ck, cv, self.anchor, self.ctx, self.K,
                                   self.contract)
            path, score, margin = oracle.select_path(self.cfg, self.W, self.anchor, d["ids"],
                                                     d["logp"], with_margin=True)
            acc, toks = oracle.accept_greedy(path, self.target)
            self._o = dict(ck=ck, cv=cv, path=path, score=score, margin=margin, acc=acc,
                           toks=toks, **d)
        return self._o

    def oracle_pure_logits(self):
        """The oracle's logits with no storage rounding anywhere (contract "none")."""
        L = self.cfg["n_layers"]
        ck, cv = [], []
        o = 0
        for b in range(self.B):
            n = int(self.ctx[b])
            k, v, _ = oracle.inject_context(self.cfg, self.W, self.hidden[o:o + n], np.arange(n),
                                            "none")
            ck.append([k[l] for l in range(L)])
            cv.append([v[l] for l in range(L)])
            o += n
        return oracle.draft_block(self.cfg, self.W, ck, cv, self.anchor, self.ctx, self.K,
                                  "none")["logits"]

    # ---------------------------------------------------------------- device
    def device(self):
        import torch
        import block_diffusion_drafter_inject_gb300 as dfl
        dev = "cuda"
        self.Wd = dfl.DeviceWeights.from_host(self.cfg, self.W, dev, q4=self.Q)
        self.kv = dfl.PagedKV(self.cfg, self.table, self.num_pages, dev)
        dt = torch.bfloat16 if self.cfg["dtype"] == "bf16" else torch.float32
        self.d_hidden = torch.from_numpy(self.hidden).to(dt).to(dev)
        self.d_req = torch.from_numpy(self.req).to(dev)
        self.d_pos = torch.from_numpy(self.pos).to(dev)
        self.d_anchor = torch.from_numpy(self.anchor).to(dev)
        self.d_ctx = torch.from_numpy(self.ctx).to(dev)
        self.d_target = torch.from_numpy(self.target).to(dev)
        self.cyc = dfl.DraftCycle(self.cfg, self.Wd, self.kv, self.B, self.K,
                                  max(int(self.ctx.sum()), 1), dev)
        V = self.cfg["vocab"]
        self.d_logits = torch.zeros((self.B, self.K - 1, V), dtype=torch.float32, device=dev)
        return self

    def run_device(self, fused=True, tail=None):
        """One cycle on the device.  fused: the injection rides in the draft pass
        (draft_block_inject), else inject_context then draft_block.  tail[b]: only
        the last tail[b] context rows of request b go through the cycle call; the
        rest are injected before it (a prefill)."""
        import torch
        import block_diffusion_drafter_inject_gb300 as dfl
        hid, req, pos = self.d_hidden, self.d_req, self.d_pos
        if tail is not None:
            late = np.concatenate([self.pos[self.req == b] >= int(self.ctx[b]) - int(tail[b])
                                   for b in range(self.B)])
            early = torch.from_numpy(np.nonzero(~late)[0]).cuda()
            if len(early):
                dfl.inject_context(self.cfg, self.Wd, self.kv, hid[early], req[early],
                                   pos[early], self.cyc.ws)
            idx = torch.from_numpy(np.nonzero(late)[0]).cuda()
            hid, req, pos = hid[idx], req[idx], pos[idx]
        self.cyc.run(hid, req, pos, self.d_anchor, self.d_ctx, self.d_target,
                     logits=self.d_logits, fused=fused)
        torch.cuda.synchronize()
        status = dfl.read_device_status(self.cyc.ws)
        c = self.cyc
        return dict(ids=c.topk_ids.cpu().numpy(), logp=c.topk_logp.cpu().numpy(),
                    logits=self.d_logits.cpu().numpy().astype(np.float64),
                    path=c.path.cpu().numpy(), score=c.score.cpu().numpy(),
                    acc=c.accept_len.cpu().numpy(), toks=c.tokens.cpu().numpy(), status=status)

    def gpu_kv_dense(self):
        """The device caches gathered back to dense [b][l] arrays for positions 0..ctx-1."""
        k = self.kv.k.float().cpu().numpy()
        v = self.kv.v.float().cpu().numpy()
        P = self.cfg["page_size"]
        outk, outv = [], []
        for b in range(self.B):
            n = int(self.ctx[b])
            p = np.arange(n)
            pages = self.table[b, p // P]
            outk.append([k[l][pages, :, p % P, :] for l in range(self.cfg["n_layers"])])
            outv.append([v[l][pages, :, p % P, :] for l in range(self.cfg["n_layers"])])
        return outk, outv


def exact_logits(cfg, W, hidden, pos, n_ctx, anchor, K):
    """The oracle's logits of one request with no storage rounding anywhere
    (contract "none"): its context rows `hidden` injected at positions `pos`."""
    k, v, _ = oracle.inject_context(cfg, W, hidden, pos, "none")
    shape = (n_ctx, cfg["n_kv_heads"], cfg["head_dim"])
    ck, cv = [], []
    for l in range(cfg["n_layers"]):
        a = np.zeros(shape)
        a[pos] = k[l]
        ck.append(a)
        a = np.zeros(shape)
        a[pos] = v[l]
        cv.append(a)
    return oracle.draft_block(cfg, W, [ck], [cv], [anchor], [n_ctx], K, "none")["logits"][0]


def rowmax_rel(g, o):
    """max over rows of max|g - o| / max|o| (row-max relative error)."""
    g = np.asarray(g, dtype=np.float64).reshape(-1, np.shape(g)[-1])
    o = np.asarray(o, dtype=np.float64).reshape(-1, np.shape(o)[-1])
    return float(np.max(np.max(np.abs(g - o), axis=1) / np.maximum(np.max(np.abs(o), axis=1), 1e-30)))


def topk_compare(g_ids, o_logits, o_ids, k, margin=1e-2):
    """Compare top-k ids where the oracle's decision margin exceeds `margin`.
    Returns (compared, mismatched) counts."""
    rows = o_logits.reshape(-1, o_logits.shape[-1])
    gi = g_ids.reshape(-1, k)
    oi = o_ids.reshape(-1, k)
    compared = bad = 0
    for r in range(rows.shape[0]):
        z = np.sort(rows[r])[::-1][:k + 1]
        for j in range(k):
            lo = z[j] - z[j + 1] if j + 1 < len(z) else np.inf
            hi = z[j - 1] - z[j] if j > 0 else np.inf
            if min(lo, hi) > margin:
                compared += 1
                bad += int(gi[r, j] != oi[r, j])
    return compared, bad


def sets_equal(g_ids, o_ids):
    return np.array_equal(np.sort(g_ids, axis=-1), np.sort(o_ids, axis=-1))


class FullCase:
    """Full-size drafter case with window-only injection: for request b only the
    positions [max(0, ctx-W), ctx) are injected (the only ones a pass reads),
    on the device and in the oracle.  The oracle runs a subset of requests."""

    _weights = {}

    def __init__(self, B, K, ctx, seed=0, oracle_requests=None, sel_scale=0.3, wseed=0,
                 q4=False):
        self.cfg = synth.preset("full", **({"weight_bits": 4} if q4 else {}))
        self.B, self.K = B, K
        self.ctx = np.asarray(ctx, dtype=np.int32)
        self.seed = seed
        key = (wseed, sel_scale, q4)
        if key not in FullCase._weights:
            FullCase._weights.clear()
            W = synth.make_weights(self.cfg, seed=wseed, sel_scale=sel_scale)
            Q = None
            if q4:
                # the oracle reads the weights the codes stand for (bf16 values, kept
                # as float32 like the other weights)
                Q = synth.make_q4_weights(self.cfg, seed=wseed)
                for n, (q, sc, b) in Q.items():
                    W[n] = oracle.dequantize_affine(q, sc, b, 64).astype(np.float32)
            FullCase._weights[key] = (W, Q)
        self.W, self.Q = FullCase._weights[key]
        Wn, P = self.cfg["window"], self.cfg["page_size"]
        self.lo = np.maximum(0, self.ctx - Wn)
        self.req = np.concatenate([np.full(c - l, b, np.int32)
                                   for b, (c, l) in enumerate(zip(self.ctx, self.lo))])
        self.pos = np.concatenate([np.arange(l, c, dtype=np.int32) for c, l in zip(self.ctx, self.lo)])
        self.hidden = synth.make_hiddens(self.cfg, len(self.req), seed=seed, name="window_hiddens")
        self.anchor = synth.make_anchors(self.cfg, B, seed=seed)
        # pages only for the positions a pass touches
        maxp = int(max((c + K + P - 1) // P for c in self.ctx))
        need = [list(range(l // P, (c + K - 1) // P + 1)) for c, l in zip(self.ctx, self.lo)]
        total = sum(len(n) for n in need)
        perm = synth.stream(seed, "page_perm").permutation(total)
        self.table = np.full((B, maxp), -1, dtype=np.int32)
        o = 0
        for b, pages in enumerate(need):
            for pi in pages:
                self.table[b, pi] = perm[o]
                o += 1
        self.num_pages = total
        self.oracle_requests = list(range(B)) if oracle_requests is None else list(oracle_requests)
        self._o = None

    def oracle(self):
        if self._o is None:
            cfg, L, K = self.cfg, self.cfg["n_layers"], self.K
            res = {}
            for b in self.oracle_requests:
                sel = self.req == b
                n_ctx = int(self.ctx[b])
                k, v, _ = oracle.inject_context(cfg, self.W, self.hidden[sel], self.pos[sel], "bf16")
                shape = (n_ctx, cfg["n_kv_heads"], cfg["head_dim"])
                ck, cv = [], []
                for l in range(L):
                    a = np.zeros(shape)
                    a[self.pos[sel]] = k[l]
                    ck.append(a)
                    a = np.zeros(shape)
                    a[self.pos[sel]] = v[l]
                    cv.append(a)
                d = oracle.draft_block(cfg, self.W, [ck], [cv], self.anchor[b:b + 1], [n_ctx], K,
                                       "bf16")
                p, s, m = oracle.select_path(cfg, self.W, self.anchor[b:b + 1], d["ids"], d["logp"],
                                             with_margin=True)
                res[b] = dict(k=k, v=v, logits=d["logits"][0], ids=d["ids"][0], logp=d["logp"][0],
                              path=p[0], score=s[0], margin=m[0],
                              logits_exact=exact_logits(cfg, self.W, self.hidden[sel],
                                                        self.pos[sel], n_ctx, self.anchor[b], K))
            self._o = res
        return self._o

    def device(self, max_inject=4096, sel_table=False, tail=None):
        """Upload, inject the windows, run draft_block and select_path; with
        sel_table, the selector reads the prepared table of every row's projections.
        tail[b]: the last tail[b] window rows of request b are injected by the pass
        itself (draft_block_inject) instead of beforehand."""
        import torch
        import block_diffusion_drafter_inject_gb300 as dfl
        self.Wd = None
        self.Wd = dfl.DeviceWeights.from_host(self.cfg, self.W, "cuda", q4=self.Q)
        self.kv = dfl.PagedKV(self.cfg, self.table, self.num_pages, "cuda")
        self.cyc = dfl.DraftCycle(self.cfg, self.Wd, self.kv, self.B, self.K, max_inject, "cuda")
        if sel_table:
            dfl.prepare_selector(self.cfg, self.Wd, self.cyc.ws)
        late = np.zeros(len(self.req), bool)
        if tail is not None:
            late = self.pos >= self.ctx[self.req] - np.asarray(tail)[self.req]
        early = np.nonzero(~late)[0]
        hid = torch.from_numpy(self.hidden[early]).to(torch.bfloat16).cuda()
        req = torch.from_numpy(self.req[early]).cuda()
        pos = torch.from_numpy(self.pos[early]).cuda()
        for o in range(0, len(early), max_inject):
            sl = slice(o, o + max_inject)
            dfl.inject_context(self.cfg, self.Wd, self.kv, hid[sl], req[sl], pos[sl], self.cyc.ws)
        self.d_anchor = torch.from_numpy(self.anchor).cuda()
        self.d_ctx = torch.from_numpy(self.ctx).cuda()
        self.d_logits = torch.zeros((self.B, self.K - 1, self.cfg["vocab"]), dtype=torch.float32,
                                    device="cuda")
        if tail is None:
            dfl.draft_block(self.cfg, self.Wd, self.kv, self.d_anchor, self.d_ctx, self.K,
                            self.cyc.ws, self.cyc.topk_ids, self.cyc.topk_logp, self.d_logits)
        else:
            lt = np.nonzero(late)[0]
            self.n_fused = len(lt)
            dfl.draft_block_inject(
                self.cfg, self.Wd, self.kv,
                torch.from_numpy(self.hidden[lt]).to(torch.bfloat16).cuda(),
                torch.from_numpy(self.req[lt]).cuda(), torch.from_numpy(self.pos[lt]).cuda(),
                self.d_anchor, self.d_ctx, self.K, self.cyc.ws, self.cyc.topk_ids,
                self.cyc.topk_logp, self.d_logits)
        dfl.select_path(self.cfg, self.Wd, self.d_anchor, self.cyc.topk_ids, self.cyc.topk_logp,
                        self.K, self.cyc.ws, self.cyc.path, self.cyc.score)
        torch.cuda.synchronize()
        self.status = dfl.read_device_status(self.cyc.ws)
        return self

    def gpu_kv(self, b):
        """Device K/V of request b at its injected positions: [L, n, Hkv, d]."""
        P = self.cfg["page_size"]
        sel = self.req == b
        p = self.pos[sel]
        pages = self.table[b, p // P]
        import torch
        pg = torch.from_numpy(pages.astype(np.int64)).cuda()
        sl = torch.from_numpy((p % P).astype(np.int64)).cuda()
        # [pages, P, L, Hkv, d] -> rows (page, slot) -> [L, n, Hkv, d]
        k = self.kv.k.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)
        v = self.kv.v.permute(1, 3, 0, 2, 4)[pg, sl].permute(1, 0, 2, 3)
        return k.float().cpu().numpy(), v.float().cpu().numpy()
