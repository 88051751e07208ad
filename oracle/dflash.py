"""The DFlash 2 draft cycle, written out in float64.

Page names used in citations:
  "KV-injection post"  = llms.blog, "Z Lab releases DFlash 2 ... with target KV injection"
  "Model-card summary" = paperfeed.app, "z-lab/Qwen3.8-27B-DFlash2"
  "Architecture page"  = kb.ekarisky.com, "DFlash 2 / Architecture"

Storage contract.  The CUDA path stores some intermediates in the weight dtype
(bf16): GEMM operands, the KV cache, the attention output.  `contract`
selects how this oracle treats those storage points:
  "none" - keep float64 everywhere (weights still hold their stored values);
  "bf16" - round to bfloat16 (nearest, ties to even) at the same points;
  "f32"  - round to float32 at the same points (the float32 configuration).
"""

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------

def round_bf16(x):
    """Nearest bfloat16 value (8 significant bits, ties to even) of float64 x."""
    x = np.asarray(x, dtype=F64)
    m, e = np.frexp(x)                 # x = m * 2**e, 0.5 <= |m| < 1
    m = np.rint(m * 256.0) / 256.0     # keep 8 significant bits, ties to even
    return np.ldexp(m, e)


def storage_round(x, contract):
    if contract == "bf16":
        return round_bf16(x)
    if contract == "f32":
        return np.asarray(x, dtype=np.float32).astype(F64)
    return np.asarray(x, dtype=F64)


# ----------------------------------------------------------------------------
# 4-bit drafter weights
# ----------------------------------------------------------------------------

def dequantize_affine(q, scale, bias, group):
    """Weights of a drafter kept in 4 bits (README mirror, MLX section: the
    example runs target and draft with 4-bit weights through a quantized matmul).
    Each row of an [N, K] matrix is cut into groups of `group` consecutive input
    features, each with its own scale s and bias b; the weight the product uses is
    s*q + b rounded once to bfloat16, q in 0..15.

    q [N, K] integers; scale, bias [N, K/group].  Returns [N, K] float64."""
    q = np.asarray(q, dtype=F64)
    s = np.repeat(np.asarray(scale, dtype=F64), group, axis=1)
    b = np.repeat(np.asarray(bias, dtype=F64), group, axis=1)
    return round_bf16(s * q + b)


def quantized_weights(W, Q, group=64):
    """The weight set W with every matrix named in Q (name -> (q, scale, bias))
    replaced by its dequantized values; the rest of the drafter is unchanged."""
    out = dict(W)
    for name, (q, s, b) in Q.items():
        out[name] = dequantize_affine(q, s, b, group)
    return out


# ----------------------------------------------------------------------------
# building blocks
# ----------------------------------------------------------------------------

def rmsnorm(x, gain, eps):
    """RMSNorm over the last axis: gain * x / sqrt(mean(x^2) + eps).

    KV-injection post, "Persistent Conditioning Through Target KV Injection"
    (the concatenated target features are normalised with RMSNorm); the same
    form is used for the drafter's pre-norms, q/k head norms and final norm."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gain, dtype=F64)


def rope(x, pos, theta):
    """Rotary position embedding, rotate-half pairing, on x [..., n, d] at
    absolute positions pos [n].  theta == 0 disables it (identity).

    Architecture page, "Internals Worth Knowing": the injected projection is
    post-processed by a norm + RoPE step; the pairing and base are a reading
    of this build (rotate-half, base 1e6)."""
    x = np.asarray(x, dtype=F64)
    if theta == 0:
        return x.copy()
    d = x.shape[-1]
    half = d // 2
    inv = theta ** (-np.arange(half, dtype=F64) * 2.0 / d)          # [half]
    ang = np.asarray(pos, dtype=F64)[:, None] * inv[None, :]          # [n, half]
    lead = [1] * (x.ndim - 2)                                         # broadcast over axes before n
    c = np.cos(ang).reshape(lead + [ang.shape[0], half])
    s = np.sin(ang).reshape(lead + [ang.shape[0], half])
    lo = x[..., :half]
    hi = x[..., half:]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def rope_heads(x, pos, theta):
    """RoPE on x [n, H, d] (heads between position and feature axes)."""
    x = np.asarray(x, dtype=F64)
    return np.stack([rope(x[:, h, :], pos, theta) for h in range(x.shape[1])], axis=1)


def sigmoid(t):
    return 1.0 / (1.0 + np.exp(-t))


def conv_two_tap(u, gate_in, G, base, group):
    """Two-tap dynamic depthwise convolution over one block.

    Architecture page, "Problem 2 - Suffix decay is local", eq. Conv_k:
    y_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, each coefficient a learned base
    kernel plus a correction computed from the current hidden state and
    shared by `group` channels.  The coefficients are sigmoid gates from one
    linear map G = [G_a; G_b] of the current position:
        a_c(t) = sigmoid(base[c]     + (G gate_in_t)[c // group])
        b_c(t) = sigmoid(base[D + c] + (G gate_in_t)[D/group + c // group])
    The block is read on its own: the tap before slot 0 is zero.

    u        [K, D] conv input values
    gate_in  [K, D] input of the gate linear (u, or u rounded for storage)
    G        [2D/group, D]; base [2D]."""
    u = np.asarray(u, dtype=F64)
    K, D = u.shape
    s = np.asarray(gate_in, dtype=F64) @ np.asarray(G, dtype=F64).T   # [K, 2D/group]
    grp = np.arange(D) // group
    a = sigmoid(np.asarray(base[:D], dtype=F64)[None, :] + s[:, grp])
    b = sigmoid(np.asarray(base[D:], dtype=F64)[None, :] + s[:, D // group + grp])
    y = np.zeros_like(u)
    for t in range(K):
        y[t] = a[t] * u[t]
        if t > 0:
            y[t] += b[t] * u[t - 1]
    return y


def block_attention(q, k, v, n_ctx_keys):
    """Non-causal block attention for one request.

    q [K, Hq, d]; k, v [n_ctx_keys + K, Hkv, d] (context window first, then
    the K block slots).  Every block query attends to every key, with no mask
    inside the block (KV-injection post, "Block Diffusion vs. Autoregressive
    Drafting": non-causal mask over the draft slots; Architecture page,
    Component Breakdown, "Block attention mask").  Scale 1/sqrt(d); query head
    h reads kv head h // (Hq/Hkv)."""
    q = np.asarray(q, dtype=F64)
    k = np.asarray(k, dtype=F64)
    v = np.asarray(v, dtype=F64)
    K, Hq, d = q.shape
    Hkv = k.shape[1]
    grp = Hq // Hkv
    o = np.zeros((K, Hq, d))
    for h in range(Hq):
        kh = k[:, h // grp, :]
        vh = v[:, h // grp, :]
        for i in range(K):
            s = (kh @ q[i, h]) / np.sqrt(d)
            p = np.exp(s - s.max())
            p /= p.sum()
            o[i, h] = p @ vh
    del n_ctx_keys
    return o


# ----------------------------------------------------------------------------
# target-KV injection
# ----------------------------------------------------------------------------

def inject_context(cfg, W, hidden, pos, contract="bf16"):
    """Project target hidden states into every draft layer's K/V.

    KV-injection post, "Persistent Conditioning Through Target KV Injection":
    the hidden states of the tapped target layers are concatenated, RMSNorm'd
    and projected (fc) to the draft width, then passed through each draft
    layer's own K and V projections into that layer's cache (also Architecture
    page, Component Breakdown, "KV injection path").  Injected K gets the
    per-head k-norm and RoPE at the token's absolute position (Architecture
    page, "Internals Worth Knowing": norm + RoPE post-processing).

    hidden [N, n_taps*d_target]; pos [N].  Returns (k, v) each [L, N, Hkv, d]
    with storage rounding applied, and c [N, D]."""
    R = lambda t: storage_round(t, contract)
    eps = cfg["rms_eps"]
    Hq, Hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    g = np.asarray(hidden, dtype=F64)
    gn = R(rmsnorm(g, W["fc_norm"], eps))
    c = R(gn @ np.asarray(W["fc"], dtype=F64).T)                       # [N, D]
    N = g.shape[0]
    L = cfg["n_layers"]
    ks = np.zeros((L, N, Hkv, dh))
    vs = np.zeros((L, N, Hkv, dh))
    for l in range(L):
        wqkv = np.asarray(W[f"layers.{l}.wqkv"], dtype=F64)
        wk = wqkv[Hq * dh:(Hq + Hkv) * dh]
        wv = wqkv[(Hq + Hkv) * dh:]
        kk = (c @ wk.T).reshape(N, Hkv, dh)
        kk = rmsnorm(kk, W[f"layers.{l}.k_norm"], eps)
        kk = rope_heads(kk, pos, cfg["rope_theta"])
        ks[l] = R(kk)
        vs[l] = R((c @ wv.T).reshape(N, Hkv, dh))
    return ks, vs, c


# ----------------------------------------------------------------------------
# one non-causal drafter pass over a block
# ----------------------------------------------------------------------------

def topk_logp(z, k):
    """Top-k candidates of one logit row and their log-probabilities.

    Model-card summary, "The idea" (keep the top candidates at each position);
    Architecture page, Component Breakdown (top-16 per position).  Order: larger
    logit first, equal logits by lower token id.  logp = z - logsumexp(z)."""
    z = np.asarray(z, dtype=F64)
    order = np.lexsort((np.arange(z.size), -z))[:k]
    m = z.max()
    lse = m + np.log(np.sum(np.exp(z - m)))
    return order.astype(np.int32), z[order] - lse, lse


def draft_block_request(cfg, W, ctx_k, ctx_v, anchor, ctx_len, K, contract="bf16",
                        conv_bypass=False, block_inputs=None, positions=None):
    """One drafter pass for one request.

    Block construction: slot 0 holds the anchor (last verified token), slots
    1..K-1 hold the mask token (Architecture page, Component Breakdown, "Block
    attention mask"; Model-card summary, "The idea": one pass predicts every
    slot).  Each layer is pre-norm attention then pre-norm SwiGLU MLP, with the
    two-tap conv before and after each sublayer (Architecture page, "Problem 2";
    Draft-Verify Cycle figure).  The shared lm_head gives logits for slots
    1..K-1 (Architecture page, Component Breakdown, shared lm_head).

    ctx_k, ctx_v: per layer, [n, Hkv, d] arrays of injected K/V for absolute
    positions 0..n-1 (n >= ctx_len).  Keys are the last min(window, ctx_len)
    context positions plus all K block slots (sliding window 1024: Architecture
    page, Component Breakdown, drafter backbone).

    conv_bypass: every conv is the identity (a = 1, b = 0); used by the
    block-mask invariance pin.  block_inputs: optional [K, D] replacement for
    the embedded block; positions: optional [K] replacement for the block's
    absolute positions.

    Returns dict(logits [K-1, V], hidden [K, D] (final residual))."""
    R = lambda t: storage_round(t, contract)
    eps = cfg["rms_eps"]
    D = cfg["d_model"]
    Hq, Hkv, dh = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    F = cfg["d_ff"]
    grp = cfg["conv_group"]
    theta = cfg["rope_theta"]
    Wn = cfg["window"]
    E = W["embed"]
    if block_inputs is None:
        toks = [int(anchor)] + [cfg["mask_token_id"]] * (K - 1)
        x = np.stack([np.asarray(E[t], dtype=F64) for t in toks])         # [K, D]
    else:
        x = np.asarray(block_inputs, dtype=F64).copy()
    pos = np.arange(K) + ctx_len if positions is None else np.asarray(positions)
    lo = max(0, ctx_len - Wn)

    def conv(u, gate_in, l, i):
        if conv_bypass:
            return np.asarray(u, dtype=F64)
        return conv_two_tap(u, gate_in, W[f"layers.{l}.conv_w.{i}"],
                            W[f"layers.{l}.conv_base.{i}"], grp)

    for l in range(cfg["n_layers"]):
        p = f"layers.{l}."
        # attention sublayer
        u = R(rmsnorm(x, W[p + "attn_norm"], eps))
        u = R(conv(u, u, l, 0))
        qkv = u @ np.asarray(W[p + "wqkv"], dtype=F64).T
        q = qkv[:, :Hq * dh].reshape(K, Hq, dh)
        k = qkv[:, Hq * dh:(Hq + Hkv) * dh].reshape(K, Hkv, dh)
        v = qkv[:, (Hq + Hkv) * dh:].reshape(K, Hkv, dh)
        q = R(rope_heads(rmsnorm(q, W[p + "q_norm"], eps), pos, theta))
        k = R(rope_heads(rmsnorm(k, W[p + "k_norm"], eps), pos, theta))
        v = R(v)
        keys = np.concatenate([np.asarray(ctx_k[l][lo:ctx_len], dtype=F64), k], axis=0)
        vals = np.concatenate([np.asarray(ctx_v[l][lo:ctx_len], dtype=F64), v], axis=0)
        o = R(block_attention(q, keys, vals, ctx_len - lo).reshape(K, Hq * dh))
        r = o @ np.asarray(W[p + "wo"], dtype=F64).T
        x = x + conv(r, R(r), l, 1)
        # MLP sublayer
        u = R(rmsnorm(x, W[p + "mlp_norm"], eps))
        u = R(conv(u, u, l, 2))
        gu = u @ np.asarray(W[p + "w_gate_up"], dtype=F64).T
        gt, up = gu[:, :F], gu[:, F:]
        h = R(gt * sigmoid(gt) * up)
        r = h @ np.asarray(W[p + "w_down"], dtype=F64).T
        x = x + conv(r, R(r), l, 3)
    zf = R(rmsnorm(x[1:], W["final_norm"], eps))
    logits = zf @ np.asarray(W["lm_head"], dtype=F64).T
    del D
    return dict(logits=logits, hidden=x, zf=zf)


def draft_block(cfg, W, ctx_k, ctx_v, anchors, ctx_lens, K, contract="bf16"):
    """Drafter pass + per-position top-k for a batch of independent requests.

    ctx_k[b][l], ctx_v[b][l]: dense injected K/V of request b.
    Returns dict(logits [B, K-1, V], ids [B, K-1, k], logp [B, K-1, k],
    lse [B, K-1], zf [B, K-1, D]: the final-normed hidden states of slots
    1..K-1, the input of the lm_head)."""
    B = len(anchors)
    k = cfg["top_k"]
    V = cfg["vocab"]
    logits = np.zeros((B, K - 1, V))
    ids = np.zeros((B, K - 1, k), dtype=np.int32)
    logp = np.zeros((B, K - 1, k))
    lse = np.zeros((B, K - 1))
    zf = np.zeros((B, K - 1, cfg["d_model"]))
    for b in range(B):
        out = draft_block_request(cfg, W, ctx_k[b], ctx_v[b], anchors[b], int(ctx_lens[b]), K,
                                  contract)
        logits[b] = out["logits"]
        zf[b] = out["zf"]
        for t in range(K - 1):
            ids[b, t], logp[b, t], lse[b, t] = topk_logp(logits[b, t], k)
    return dict(logits=logits, ids=ids, logp=logp, lse=lse, zf=zf)


# ----------------------------------------------------------------------------
# candidate-path selector
# ----------------------------------------------------------------------------

def select_path_request(E, Pu, Pv, anchor, ids, logp, with_margin=False):
    """Viterbi over the top-k candidate lattice of one request.

    Architecture page, "Problem 1 - Independent picks are incoherent", eq. S_t:
    every adjacent pair of candidates is scored by the drafter's own score of
    the later candidate plus a low-rank bilinear match of compact token
    embeddings of the two.  Here the match is (P_u e_a) . (P_v e_b), e = row of
    the embedding table, and the per-candidate score is the log-probability;
    the path maximising the summed pair scores from the anchor (last verified
    token) is found by max-sum dynamic programming.

        delta_1(j) = logp_1(j) + u(anchor) . v(c_1j)
        delta_t(j) = logp_t(j) + max_i [delta_{t-1}(i) + u(c_{t-1,i}) . v(c_tj)]

    Ties go to the lower candidate rank, both inside the max and at the end.
    ids, logp: [T, k] with T = K-1 draft slots.  Returns (path [T], score) and,
    with with_margin, the gap between the best and second-best path score."""
    E = np.asarray(E)
    Pu = np.asarray(Pu, dtype=F64)
    Pv = np.asarray(Pv, dtype=F64)
    T, k = ids.shape
    emb = lambda t: np.asarray(E[t], dtype=F64)
    u_prev = (Pu @ emb(int(anchor)))[None, :]                           # [1, r]
    delta = None
    bps = []
    # second-best bookkeeping: best two scores per state (list Viterbi, N = 2)
    top2 = None
    for t in range(T):
        vt = np.stack([Pv @ emb(int(c)) for c in ids[t]])              # [k, r]
        pair = u_prev @ vt.T                                            # [n_prev, k]
        lp = np.asarray(logp[t], dtype=F64)
        if t == 0:
            delta = lp + pair[0]
            bp = np.zeros(k, dtype=np.int64)
            top2 = [sorted([(delta[j], 0, 0)], key=lambda e: -e[0]) for j in range(k)]
        else:
            cand = delta[:, None] + pair                                 # [k_prev, k]
            bp = np.argmax(cand, axis=0)                                 # first max = lowest rank
            new_delta = lp + cand[bp, np.arange(k)]
            new_top2 = []
            for j in range(k):
                entries = []
                for i in range(k):
                    for rank, e in enumerate(top2[i]):
                        entries.append((e[0] + pair[i, j] + lp[j], i, rank))
                entries.sort(key=lambda e: -e[0])
                new_top2.append(entries[:2])
            delta = new_delta
            top2 = new_top2
        bps.append(bp)
        u_prev = np.stack([Pu @ emb(int(c)) for c in ids[t]])           # [k, r]
    last = int(np.argmax(delta))
    score = float(delta[last])
    path_rank = [last]
    for t in range(T - 1, 0, -1):
        path_rank.append(int(bps[t][path_rank[-1]]))
    path_rank.reverse()
    path = np.array([ids[t][path_rank[t]] for t in range(T)], dtype=np.int32)
    if not with_margin:
        return path, score
    finals = sorted([e[0] for j in range(k) for e in top2[j]], reverse=True)
    margin = finals[0] - finals[1] if len(finals) > 1 else np.inf
    return path, score, margin


def select_path(cfg, W, anchors, ids, logp, with_margin=False):
    """Batch of independent requests; returns path [B, K-1], score [B] (and margin [B])."""
    B = len(anchors)
    T = ids.shape[1]
    path = np.zeros((B, T), dtype=np.int32)
    score = np.zeros(B)
    margin = np.zeros(B)
    for b in range(B):
        out = select_path_request(W["embed"], W["sel_pu"], W["sel_pv"], anchors[b], ids[b],
                                  logp[b], with_margin=True)
        path[b], score[b], margin[b] = out
    if with_margin:
        return path, score, margin
    return path, score


# ----------------------------------------------------------------------------
# greedy acceptance
# ----------------------------------------------------------------------------

def accept_greedy_request(path, T):
    """Longest accepted prefix plus one bonus token (greedy verification).

    Architecture page, "Speculative Decoding Context" (the target accepts the
    longest valid prefix) and "One Cycle, Step by Step" (accepted prefix + 1
    bonus token); at temperature 0 the output equals the target's own greedy
    output (Model-card summary, "The idea").  Row i of T is the target's
    prediction for the token after block slot i; the draft token of slot i+1
    is accepted while it equals that row's argmax (lower id on ties; a NaN
    counts as larger than every number, so a row's first NaN is its argmax,
    which is numpy's argmax rule).

    Returns (accept_len in 1..K, tokens [K] with -1 after the bonus token)."""
    T = np.asarray(T)
    K = T.shape[0]
    tgt = [int(np.argmax(T[i])) for i in range(K)]
    m = 0
    while m < K - 1 and int(path[m]) == tgt[m]:
        m += 1
    tokens = np.full(K, -1, dtype=np.int32)
    tokens[:m] = path[:m]
    tokens[m] = tgt[m]
    return m + 1, tokens


def accept_greedy(path, T):
    B, K = T.shape[0], T.shape[1]
    acc = np.zeros(B, dtype=np.int32)
    toks = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        acc[b], toks[b] = accept_greedy_request(path[b], T[b])
    return acc, toks


# ----------------------------------------------------------------------------
# sampling walk and lossless rejection sampling
# ----------------------------------------------------------------------------

def draw_index(weights, u):
    """Inverse-CDF draw from non-negative weights (not necessarily normalised)
    with one uniform u in [0, 1): the smallest index j with u * W < C_j, where
    C_j is the running sum of the weights in index order and W = C_last."""
    w = np.asarray(weights, dtype=F64)
    c = np.cumsum(w)
    j = int(np.searchsorted(c, u * c[-1], side="right"))
    return min(j, int(np.flatnonzero(w > 0)[-1]))


def sample_path_request(E, Pu, Pv, anchor, ids, logp, u_walk):
    """Temperature-1 sampling walk over the candidate lattice of one request.

    Architecture page, "Problem 1 - Independent picks are incoherent": the
    walk over the precomputed pair scores is the only sequential part, and
    sampling draws from the same scores as the greedy walk.  From the anchor
    (last verified token), position t draws its candidate j with probability
        q_t(j) = softmax_j( logp_t(j) + (P_u e_a) . (P_v e_{c_tj}) )
    where a is the token drawn at t-1 (the anchor at t = 1), by inverse CDF
    over the candidate ranks with the uniform u_walk[t] (draw_index).
    ids, logp [T, k]; u_walk [T].  Returns (path [T], q [T, k]): the drawn
    tokens and, per position, the proposal distribution they were drawn from."""
    E = np.asarray(E)
    Pu = np.asarray(Pu, dtype=F64)
    Pv = np.asarray(Pv, dtype=F64)
    T, k = ids.shape
    emb = lambda t: np.asarray(E[int(t)], dtype=F64)
    prev = int(anchor)
    path = np.zeros(T, dtype=np.int32)
    q = np.zeros((T, k))
    for t in range(T):
        u_prev = Pu @ emb(prev)
        s = np.array([float(logp[t][j]) + u_prev @ (Pv @ emb(ids[t][j])) for j in range(k)])
        e = np.exp(s - s.max())
        q[t] = e / e.sum()
        j = draw_index(e, float(u_walk[t]))
        path[t] = ids[t][j]
        prev = int(path[t])
    return path, q


def accept_sample_request(path, cand_ids, q, T, u):
    """Speculative rejection sampling of one request's drafted block (lossless).

    Architecture page, "Speculative Decoding Context" (rejection sampling makes
    the scheme lossless) and "Problem 1" (rejection sampling restores the
    exact target distribution).  Row i of T is the target's logits for the
    token after block slot i; p_i = softmax(T[i]) at temperature 1.  The draft
    token x = path[i] came from the proposal q_i (q[i][j] for candidate
    cand_ids[i][j], 0 for every other token).  For i = 0, 1, ...: x is accepted
    when u[i, 0] * q_i(x) < p_i(x) (probability min(1, p/q)); at the first
    rejection the replacement is drawn from max(0, p_i - q_i) with u[i, 1] and
    the block ends; when every draft is accepted a bonus token is drawn from
    p_{K-1} with u[K-1, 1].  Draws use draw_index over token ids.
    path [K-1]; cand_ids, q [K-1, k]; T [K, V]; u [K, 2].
    Returns (accept_len in 1..K, tokens [K], -1 after the last token)."""
    T = np.asarray(T, dtype=F64)
    K = T.shape[0]
    tokens = np.full(K, -1, dtype=np.int32)

    def probs(i):
        z = T[i]
        e = np.exp(z - z.max())
        return e / e.sum()

    for i in range(K - 1):
        p = probs(i)
        x = int(path[i])
        qi = np.zeros_like(p)
        for j, c in enumerate(cand_ids[i]):
            qi[int(c)] += float(q[i][j])
        if float(u[i][0]) * qi[x] < p[x]:
            tokens[i] = x
            continue
        r = np.maximum(p - qi, 0.0)
        # r sums to zero only if p = q, where no draft is ever rejected; p then
        # stands in (a measure-zero case kept defined)
        tokens[i] = draw_index(r if r.sum() > 0 else p, float(u[i][1]))
        return i + 1, tokens
    tokens[K - 1] = draw_index(probs(K - 1), float(u[K - 1][1]))
    return K, tokens


def sample_path(cfg, W, anchors, ids, logp, u_walk):
    """Batch form: path [B, K-1], q [B, K-1, k]."""
    B, T, k = ids.shape
    path = np.zeros((B, T), dtype=np.int32)
    q = np.zeros((B, T, k))
    for b in range(B):
        path[b], q[b] = sample_path_request(W["embed"], W["sel_pu"], W["sel_pv"], anchors[b],
                                            ids[b], logp[b], u_walk[b])
    return path, q


def accept_sample(path, cand_ids, q, T, u):
    """Batch form: accept_len [B], tokens [B, K]."""
    B, K = T.shape[0], T.shape[1]
    acc = np.zeros(B, dtype=np.int32)
    toks = np.zeros((B, K), dtype=np.int32)
    for b in range(B):
        acc[b], toks[b] = accept_sample_request(path[b], cand_ids[b], q[b], T[b], u[b])
    return acc, toks


# ----------------------------------------------------------------------------
# the pages' selector form: context-gated pair scores, greedy walk
# ----------------------------------------------------------------------------

def context_gate(Wh, h):
    """H(h_t) = sigmoid(W_H h_t): the context gate of eq. S_t (Architecture page,
    "Problem 1": H(h_t) decides which parts of the predecessor match count).
    The form of H is a reading of this build (the pages name only its role):
    one linear map of the drafter's hidden state, then per-dimension sigmoid.
    Wh [r, D]; h [T, D]  ->  [T, r]."""
    return sigmoid(np.asarray(h, dtype=F64) @ np.asarray(Wh, dtype=F64).T)


def select_greedy_request(E, Pu, Pv, Wh, h, anchor, ids, logp, with_margin=False,
                          step_margins=False):
    """Greedy walk over the context-gated pair scores of one request.

    Architecture page, "Problem 1", eq. S_t:
        S_t(a, b) = U_t(b) + < A(a) * H(h_t), B(b) >
    with A(a) = P_u e_a, B(b) = P_v e_b (compact r-dim token embeddings), H the
    context gate of the drafter hidden state h_t of position t (context_gate),
    and U_t(b) the drafter's score of candidate b (the log-probability here:
    it differs from the logit by a per-position constant, which moves neither
    the walk nor the comparison of paths).  "Greedy follows the best
    successor": from the anchor, position t takes argmax_b S_t(a_{t-1}, b) over
    its candidates (ties: lower rank).  ids, logp [T, k]; h [T, D].  Returns
    (path [T], score = sum of the chosen S_t) and, with with_margin, the
    smallest gap between the chosen and the runner-up score over the steps
    (with step_margins, the gap of every step [T] instead)."""
    E = np.asarray(E)
    Pu = np.asarray(Pu, dtype=F64)
    Pv = np.asarray(Pv, dtype=F64)
    T, k = ids.shape
    g = context_gate(Wh, h)
    emb = lambda t: np.asarray(E[int(t)], dtype=F64)
    prev = int(anchor)
    path = np.zeros(T, dtype=np.int32)
    score, margin = 0.0, np.inf
    gaps = np.full(T, np.inf)
    for t in range(T):
        ug = (Pu @ emb(prev)) * g[t]
        s = np.array([float(logp[t][j]) + ug @ (Pv @ emb(ids[t][j])) for j in range(k)])
        j = int(np.argmax(s))                      # first maximum = lowest rank
        if k > 1:
            gaps[t] = float(s[j] - np.max(np.delete(s, j)))
            margin = min(margin, gaps[t])
        path[t] = ids[t][j]
        score += float(s[j])
        prev = int(path[t])
    if with_margin:
        return path, score, (gaps if step_margins else margin)
    return path, score


def select_greedy(cfg, W, anchors, ids, logp, hidden):
    """Batch form: hidden [B, K-1, D].  Returns path [B, K-1], score [B], margin [B]."""
    B, T, _ = ids.shape
    path = np.zeros((B, T), dtype=np.int32)
    score = np.zeros(B)
    margin = np.zeros(B)
    for b in range(B):
        path[b], score[b], margin[b] = select_greedy_request(
            W["embed"], W["sel_pu"], W["sel_pv"], W["sel_gate"], hidden[b], anchors[b], ids[b],
            logp[b], with_margin=True)
    return path, score, margin
