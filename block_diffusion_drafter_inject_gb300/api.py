"""Python binding of the DFlash C ABI: argument marshalling only.

Device memory comes from PyTorch (weights, paged KV, workspace, outputs); every
step of the draft cycle runs in the library's CUDA kernels, launched on the
current PyTorch stream.  The names follow include/dflash.h:
inject_context, draft_block, select_path, accept_greedy."""

import ctypes

import torch

from . import _lib
from ._lib import check, lib

_DT = {"f32": _lib.F32, "bf16": _lib.BF16}
_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def make_config(cfg):
    """dflash_config from a dimension dict (the presets' keys)."""
    c = _lib.Config()
    for name, _ in _lib.Config._fields_:
        if name == "dtype":
            c.dtype = _DT[cfg["dtype"]]
        elif name == "mask_token_id":
            c.mask_token_id = int(cfg.get("mask_token_id", cfg["vocab"] - 1))
        elif name == "weight_bits":
            c.weight_bits = int(cfg.get("weight_bits", 0))
        else:
            setattr(c, name, type(getattr(c, name))(cfg[name]))
    return c


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


class DeviceWeights:
    """Drafter weights resident on the GPU and the dflash_weights struct that points at
    them (a weight missing from `tensors` is a NULL pointer: the calls that need it
    refuse with DFLASH_ERR_NULL)."""

    def __init__(self, cfg, tensors):
        self.cfg = cfg
        self.t = tensors
        w = _lib.Weights()
        ptr = lambda n: tensors[n].data_ptr() if n in tensors else None  # absent: NULL
        for n in ("fc_norm", "fc", "embed", "lm_head", "final_norm", "sel_pu", "sel_pv"):
            setattr(w, n, ptr(n))
        for l in range(cfg["n_layers"]):
            L = w.layer[l]
            p = f"layers.{l}."
            for n in ("attn_norm", "mlp_norm", "wqkv", "wo", "q_norm", "k_norm", "w_gate_up",
                      "w_down"):
                setattr(L, n, ptr(p + n))
            for i in range(4):
                L.conv_w[i] = ptr(p + f"conv_w.{i}")
                L.conv_base[i] = ptr(p + f"conv_base.{i}")
        if "sel_gate" in tensors:
            w.sel_gate = tensors["sel_gate"].data_ptr()
        # 4-bit matrices: tensors NAME.q4 (see pack_q4)
        q4 = lambda q, n: setattr(q, "data", ptr(n + ".q4"))
        for n in _lib.Q4_TOP:
            q4(getattr(w, n + "_q4"), n)
        for l in range(cfg["n_layers"]):
            for n in _lib.Q4_LAYER:
                q4(getattr(w.layer[l], n + "_q4"), f"layers.{l}.{n}")
        self.struct = w
        self.sel_table = None  # see prepare_selector

    @classmethod
    def from_host(cls, cfg, host, device="cuda", q4=None):
        """Upload float32 host arrays (holding storage-dtype values) in the config dtype.
        q4: name -> (codes q [N, K] 0..15, scale [N, K/64], bias [N, K/64]) of the
        matrices kept in 4 bits (their storage-dtype arrays in `host` are skipped)."""
        dt = _TORCH_DT[cfg["dtype"]]
        t = {}
        for name, arr in host.items():
            if q4 is not None and name in q4:
                continue
            t[name] = torch.from_numpy(arr).to(dt).to(device).contiguous()
        for name, (q, sc, bias) in (q4 or {}).items():
            t[name + ".q4"] = pack_q4(q, sc, bias).to(device)
        return cls(cfg, t)


def pack_q4(q, scale, bias):
    """The C ABI's 4-bit layout of one matrix (dflash_q4) as a flat uint8 tensor:
    rows padded to a multiple of 128, cut into 64-row blocks; per block and group
    of 64 input features one 2304-byte record: the rows' codes (32 bytes a row,
    the nibbles of features 8j..8j+7 in the order 8j, 8j+2, 8j+4, 8j+6, 8j+1, 8j+3,
    8j+5, 8j+7 from the least significant of their 32-bit word), then their
    (scale, bias) words (bf16 scale bits low, bf16 bias bits high)."""
    q = torch.as_tensor(q).to(torch.uint8)
    N, K = q.shape
    Np = (N + 127) // 128 * 128
    G = K // 64
    g = q.reshape(N, K // 8, 8)
    codes = (g[:, :, [0, 4, 1, 5]] | (g[:, :, [2, 6, 3, 7]] << 4)).reshape(N, K // 2)
    bits = lambda a: torch.as_tensor(a).to(torch.bfloat16).view(torch.int16).to(torch.int32) & 0xFFFF
    words = (bits(scale) | (bits(bias) << 16)).reshape(N, G, 1).view(torch.uint8)  # [N, G, 4]
    rec = torch.zeros((Np, G, 36), dtype=torch.uint8)
    rec[:N, :, :32] = codes.reshape(N, G, 32)
    rec[:N, :, 32:] = words
    # [row block, 64 rows, group, 36] -> [row block, group, 64 rows x 32 | 64 rows x 4]
    rec = rec.reshape(Np // 64, 64, G, 36).permute(0, 2, 1, 3)
    out = torch.cat([rec[..., :32].reshape(Np // 64, G, 2048),
                     rec[..., 32:].reshape(Np // 64, G, 256)], dim=2)
    return out.reshape(-1).contiguous()


def linear_q4(data, N_out, X, out, splits=1, stream=None):
    """dflash_linear_q4: out[s] = the s-th K slice of X W^T with W [N_out, K] in 4 bits
    (data from pack_q4)."""
    w = _lib.Q4()
    w.data = data.data_ptr()
    check(lib().dflash_linear_q4(w, int(N_out), int(X.shape[1]), _ptr(X), int(X.shape[0]),
                                 int(splits), _ptr(out), _stream(stream)), "dflash_linear_q4")


class PagedKV:
    """Per-layer paged K and V caches [L][num_pages][Hkv][page_size][d] and a page table."""

    def __init__(self, cfg, page_table, num_pages, device="cuda"):
        dt = _TORCH_DT[cfg["dtype"]]
        shape = (cfg["n_layers"], int(num_pages), cfg["n_kv_heads"], cfg["page_size"],
                 cfg["head_dim"])
        self.k = torch.zeros(shape, dtype=dt, device=device)
        self.v = torch.zeros(shape, dtype=dt, device=device)
        self.page_table = torch.as_tensor(page_table, dtype=torch.int32).to(device).contiguous()
        s = _lib.KV()
        s.k = self.k.data_ptr()
        s.v = self.v.data_ptr()
        s.page_table = self.page_table.data_ptr()
        s.num_pages = int(num_pages)
        s.max_pages_per_req = int(self.page_table.shape[1])
        s.num_rows = int(self.page_table.shape[0])
        self.struct = s


def workspace_bytes(cfg, B, K, max_inject_tokens):
    c = make_config(cfg)
    n = lib().dflash_workspace_bytes(ctypes.byref(c), B, K, max_inject_tokens)
    if n == 0:
        raise ValueError("invalid configuration or sizes for dflash_workspace_bytes")
    return n


class Workspace:
    """Zero-filled device scratch for up to B requests of block K and max_inject_tokens."""

    def __init__(self, cfg, B, K, max_inject_tokens, device="cuda"):
        self.nbytes = workspace_bytes(cfg, B, K, max_inject_tokens)
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())


def inject_context(cfg, W, kv, hidden, req, pos, ws, stream=None):
    c = make_config(cfg)
    check(lib().dflash_inject_context(ctypes.byref(c), ctypes.byref(W.struct),
                                      ctypes.byref(kv.struct), _ptr(hidden), _ptr(req), _ptr(pos),
                                      int(hidden.shape[0]), ws.ptr, ws.nbytes, _stream(stream)),
          "dflash_inject_context")


def draft_block(cfg, W, kv, anchor, ctx_len, K, ws, topk_ids, topk_logp, logits=None,
                stream=None):
    c = make_config(cfg)
    check(lib().dflash_draft_block(ctypes.byref(c), ctypes.byref(W.struct),
                                   ctypes.byref(kv.struct), _ptr(anchor), _ptr(ctx_len),
                                   int(anchor.shape[0]), int(K), _ptr(topk_ids), _ptr(topk_logp),
                                   _ptr(logits), ws.ptr, ws.nbytes, _stream(stream)),
          "dflash_draft_block")


def draft_block_inject(cfg, W, kv, hidden, req, pos, anchor, ctx_len, K, ws, topk_ids,
                       topk_logp, logits=None, stream=None):
    """inject_context followed by draft_block, in one pass (dflash_draft_block_inject):
    the new rows' K/V come out of each layer's QKV projection."""
    c = make_config(cfg)
    n = 0 if hidden is None else int(hidden.shape[0])
    check(lib().dflash_draft_block_inject(ctypes.byref(c), ctypes.byref(W.struct),
                                          ctypes.byref(kv.struct), _ptr(hidden), _ptr(req),
                                          _ptr(pos), n, _ptr(anchor), _ptr(ctx_len),
                                          int(anchor.shape[0]), int(K), _ptr(topk_ids),
                                          _ptr(topk_logp), _ptr(logits), ws.ptr, ws.nbytes,
                                          _stream(stream)),
          "dflash_draft_block_inject")


def select_path(cfg, W, anchor, topk_ids, topk_logp, K, ws, path, score, stream=None):
    c = make_config(cfg)
    check(lib().dflash_select_path(ctypes.byref(c), ctypes.byref(W.struct), _ptr(anchor),
                                   _ptr(topk_ids), _ptr(topk_logp), int(anchor.shape[0]), int(K),
                                   _ptr(path), _ptr(score), ws.ptr, ws.nbytes, _stream(stream)),
          "dflash_select_path")


def prepare_selector(cfg, W, ws, stream=None):
    """Forms both selector projections of every vocabulary row once
    (dflash_prepare_selector) and points W's weights struct at them, so that
    select_path reads candidate rows from the table instead of projecting them."""
    c = make_config(cfg)
    table = torch.empty((2, cfg["vocab"], cfg["sel_rank"]), dtype=torch.float32,
                        device=W.t["embed"].device)
    check(lib().dflash_prepare_selector(ctypes.byref(c), ctypes.byref(W.struct), _ptr(table),
                                        ws.ptr, ws.nbytes, _stream(stream)),
          "dflash_prepare_selector")
    W.sel_table = table
    W.struct.sel_table = table.data_ptr()
    return table


def accept_greedy(path, target_logits, ws, accept_len, tokens, stream=None):
    B, K, V = target_logits.shape
    dt = _lib.F32 if target_logits.dtype == torch.float32 else _lib.BF16
    check(lib().dflash_accept_greedy(_ptr(path), _ptr(target_logits), dt, B, K, V,
                                     _ptr(accept_len), _ptr(tokens), ws.ptr, ws.nbytes,
                                     _stream(stream)),
          "dflash_accept_greedy")


def accept_greedy_noalloc(path, target_logits, accept_len, tokens, stream=None):
    """dflash_accept_greedy without a workspace (fixed library-owned scratch;
    B * K * ceil(V / 8192) <= 32768; overlapping calls race)."""
    B, K, V = target_logits.shape
    dt = _lib.F32 if target_logits.dtype == torch.float32 else _lib.BF16
    check(lib().dflash_accept_greedy_noalloc(_ptr(path), _ptr(target_logits), dt, B, K, V,
                                             _ptr(accept_len), _ptr(tokens), _stream(stream)),
          "dflash_accept_greedy_noalloc")


def sample_path(cfg, W, anchor, topk_ids, topk_logp, K, uniforms, ws, path, path_q, stream=None):
    """Temperature-1 sampling walk (dflash_sample_path): uniforms [B, K-1] f32 in
    [0, 1); path [B, K-1] int32 and path_q [B, K-1, top_k] f32 out."""
    c = make_config(cfg)
    check(lib().dflash_sample_path(ctypes.byref(c), ctypes.byref(W.struct), _ptr(anchor),
                                   _ptr(topk_ids), _ptr(topk_logp), int(anchor.shape[0]), int(K),
                                   _ptr(uniforms), _ptr(path), _ptr(path_q), ws.ptr, ws.nbytes,
                                   _stream(stream)),
          "dflash_sample_path")


def select_greedy(cfg, W, anchor, topk_ids, topk_logp, hidden, K, ws, path, score, stream=None):
    """The pages' context-gated pair scores, walked greedily (dflash_select_greedy):
    hidden [B, K-1, D] in the config dtype (e.g. draft_hidden after draft_block)."""
    c = make_config(cfg)
    check(lib().dflash_select_greedy(ctypes.byref(c), ctypes.byref(W.struct), _ptr(anchor),
                                     _ptr(topk_ids), _ptr(topk_logp), _ptr(hidden),
                                     int(anchor.shape[0]), int(K), _ptr(path), _ptr(score),
                                     ws.ptr, ws.nbytes, _stream(stream)),
          "dflash_select_greedy")


def draft_hidden(cfg, B, K, ws):
    """The final-normed hidden states [B, K-1, D] that the last draft_block left
    in the workspace (a view of the workspace: valid until its next use)."""
    c = make_config(cfg)
    addr = lib().dflash_draft_hidden(ctypes.byref(c), int(B), int(K), ws.ptr, ws.nbytes)
    if not addr:
        raise ValueError("invalid arguments for dflash_draft_hidden")
    es = 2 if cfg["dtype"] == "bf16" else 4
    off = addr - ws.buf.data_ptr()
    n = B * (K - 1) * cfg["d_model"]
    view = ws.buf[off:off + n * es].view(_TORCH_DT[cfg["dtype"]])
    return view.view(B, K - 1, cfg["d_model"])


def accept_sample(path, topk_ids, path_q, target_logits, uniforms, ws, accept_len, tokens,
                  stream=None):
    """Speculative rejection sampling (dflash_accept_sample): uniforms [B, K, 2] f32."""
    B, K, V = target_logits.shape
    k = topk_ids.shape[-1]
    dt = _lib.F32 if target_logits.dtype == torch.float32 else _lib.BF16
    check(lib().dflash_accept_sample(_ptr(path), _ptr(topk_ids), _ptr(path_q),
                                     _ptr(target_logits), dt, B, K, V, k, _ptr(uniforms),
                                     _ptr(accept_len), _ptr(tokens), ws.ptr, ws.nbytes,
                                     _stream(stream)),
          "dflash_accept_sample")


def linear_splits(N_out, T, K_in):
    return int(lib().dflash_linear_splits(N_out, T, K_in))


def linear(W, X, out, splits, stream=None):
    """out[s] (s < splits) = slice s of X @ W.T; W [N_out, K_in], X [T, K_in] (same dtype)."""
    N, Kin = W.shape
    T = X.shape[0]
    dt = _lib.F32 if W.dtype == torch.float32 else _lib.BF16
    check(lib().dflash_linear(dt, _ptr(W), N, Kin, _ptr(X), T, int(splits), _ptr(out),
                              _stream(stream)), "dflash_linear")


def read_device_status(ws, stream=None):
    r = lib().dflash_read_device_status(ws.ptr, _stream(stream))
    if r < 0:
        check(r, "dflash_read_device_status")
    return r


def clear_device_status(ws, stream=None):
    check(lib().dflash_clear_device_status(ws.ptr, _stream(stream)), "dflash_clear_device_status")


def launch_count(reset=False):
    return int(lib().dflash_launch_count(1 if reset else 0))


class DraftCycle:
    """Buffers and calls of one draft cycle (inject -> draft -> select -> accept) for B
    requests of block K; the shape a serving loop would hold on to."""

    def __init__(self, cfg, W, kv, B, K, max_inject_tokens, device="cuda"):
        self.cfg, self.W, self.kv, self.B, self.K = cfg, W, kv, B, K
        self.ws = Workspace(cfg, B, K, max_inject_tokens, device)
        k = cfg["top_k"]
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        self.topk_ids = torch.zeros((B, K - 1, k), **i32)
        self.topk_logp = torch.zeros((B, K - 1, k), **f32)
        self.path = torch.zeros((B, K - 1), **i32)
        self.score = torch.zeros((B,), **f32)
        self.accept_len = torch.zeros((B,), **i32)
        self.tokens = torch.zeros((B, K), **i32)

    def run(self, hidden, req, pos, anchor, ctx_len, target_logits, logits=None, stream=None,
            fused=True):
        """One cycle.  fused: the injection rides in the draft pass
        (draft_block_inject); else inject_context then draft_block."""
        if fused:
            draft_block_inject(self.cfg, self.W, self.kv, hidden, req, pos, anchor, ctx_len,
                               self.K, self.ws, self.topk_ids, self.topk_logp, logits, stream)
        else:
            if hidden is not None and hidden.shape[0] > 0:
                inject_context(self.cfg, self.W, self.kv, hidden, req, pos, self.ws, stream)
            draft_block(self.cfg, self.W, self.kv, anchor, ctx_len, self.K, self.ws,
                        self.topk_ids, self.topk_logp, logits, stream)
        select_path(self.cfg, self.W, anchor, self.topk_ids, self.topk_logp, self.K, self.ws,
                    self.path, self.score, stream)
        accept_greedy(self.path, target_logits, self.ws, self.accept_len, self.tokens, stream)
