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

    # ---------------------------------------------------------------- device
    def device(self):
        import torch
        import block_diffusion_drafter_inject_gb300 as dfl
        dev = "cuda"
        self.Wd = dfl.DeviceWeights.from_host(self.cfg, self.W, dev)
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

    def run_device(self):
        import torch
        self.cyc.run(self.d_hidden, self.d_req, self.d_pos, self.d_anchor, self.d_ctx,
                     self.d_target, logits=self.d_logits)
        torch.cuda.synchronize()
        import block_diffusion_drafter_inject_gb300 as dfl
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
