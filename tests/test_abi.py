"""The C-ABI library on the CPU: it loads, exports every symbol include/dflash.h
declares, and its host-side checks return their status codes before anything
is launched (no call here reaches a GPU: every case fails a host check)."""

import ctypes
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dflash.h")


@pytest.fixture(scope="module")
def dfl():
    import block_diffusion_drafter_inject_gb300 as m
    from block_diffusion_drafter_inject_gb300.build import build
    build()
    m.lib()
    return m


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_cycle_calls():
    names = declared_functions()
    for n in ("dflash_inject_context", "dflash_draft_block", "dflash_select_path",
              "dflash_accept_greedy", "dflash_workspace_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(dfl):
    lib = ctypes.CDLL(dfl._lib.LIB)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_declares_every_symbol(dfl):
    assert set(declared_functions()) == set(dfl._lib.EXPORTS)


def test_status_strings(dfl):
    L = dfl.lib()
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, 1, 2, 4, 8, 16):
        s = L.dflash_status_string(code).decode()
        assert s and s != "unknown status", code
    assert L.dflash_status_string(12345).decode() == "unknown status"


def _cfg(dfl, **over):
    c = dfl.make_config(synth.preset("tiny_bf16"))
    for k, v in over.items():
        setattr(c, k, v)
    return c


def test_workspace_bytes_validates(dfl):
    L = dfl.lib()
    good = _cfg(dfl)
    assert L.dflash_workspace_bytes(ctypes.byref(good), 1, 8, 16) > 0
    assert L.dflash_workspace_bytes(None, 1, 8, 16) == 0
    for over in (dict(head_dim=96), dict(d_model=100), dict(n_q_heads=3, n_kv_heads=2),
                 dict(top_k=0), dict(top_k=33), dict(sel_rank=20), dict(dtype=7),
                 dict(conv_group=3), dict(mask_token_id=4096), dict(n_layers=0),
                 dict(n_layers=17), dict(window=0), dict(page_size=0)):
        c = _cfg(dfl, **over)
        assert L.dflash_workspace_bytes(ctypes.byref(c), 1, 8, 16) == 0, over
    for B, K in ((0, 8), (1, 1), (1, 33)):
        assert L.dflash_workspace_bytes(ctypes.byref(good), B, K, 16) == 0, (B, K)


def _fake_weights(dfl, cfg, base=1 << 20):
    """Aligned, never-dereferenced addresses: every case below fails a host
    check before any use of them."""
    w = dfl._lib.Weights()
    a = base
    for n in ("fc_norm", "fc", "embed", "lm_head", "final_norm", "sel_pu", "sel_pv"):
        setattr(w, n, a)
        a += 4096
    for l in range(cfg.n_layers):
        L = w.layer[l]
        for n in ("attn_norm", "mlp_norm", "wqkv", "wo", "q_norm", "k_norm", "w_gate_up",
                  "w_down"):
            setattr(L, n, a)
            a += 4096
        for i in range(4):
            L.conv_w[i] = a
            L.conv_base[i] = a + 1024
            a += 4096
    return w


def _fake_kv(dfl):
    kv = dfl._lib.KV()
    kv.k, kv.v, kv.page_table = 1 << 30, 1 << 31, 1 << 29
    kv.num_pages, kv.max_pages_per_req, kv.num_rows = 4, 2, 2
    return kv


def test_draft_block_host_checks(dfl):
    L = dfl.lib()
    cfg = _cfg(dfl)
    w = _fake_weights(dfl, cfg)
    kv = _fake_kv(dfl)
    P = ctypes.c_void_p
    a = P(1 << 24)
    need = L.dflash_workspace_bytes(ctypes.byref(cfg), 2, 8, 1)

    def call(cfg=cfg, w=w, kv=kv, B=2, K=8, ids=a, lp=a, ws=a, nbytes=need):
        return L.dflash_draft_block(ctypes.byref(cfg) if cfg is not None else None,
                                    ctypes.byref(w) if w is not None else None,
                                    ctypes.byref(kv) if kv is not None else None,
                                    a, a, B, K, ids, lp, None, ws, nbytes, None)

    assert call(cfg=None) == -1
    assert call(K=1) == -3
    assert call(K=33) == -3
    assert call(B=-1) == -3
    assert call(B=0) == 0                       # empty batch: a no-op
    assert call(ids=P(0)) == -1
    assert call(w=None) == -1
    assert call(kv=None) == -1
    assert call(nbytes=need - 1) == -4          # workspace too small, checked before any launch
    assert call(ws=P((1 << 24) + 4)) == -7      # misaligned workspace
    bad = _fake_weights(dfl, cfg)
    bad.layer[1].w_down = (1 << 22) + 2
    assert call(w=bad) == -7                    # misaligned TMA operand
    nul = _fake_weights(dfl, cfg)
    nul.layer[0].conv_w[3] = 0
    assert call(w=nul) == -1
    c2 = _cfg(dfl, head_dim=96)
    assert call(cfg=c2) == -2
    c3 = _cfg(dfl, dtype=5)
    assert call(cfg=c3) == -5


def test_draft_block_inject_host_checks(dfl):
    L = dfl.lib()
    cfg = _cfg(dfl)
    w = _fake_weights(dfl, cfg)
    kv = _fake_kv(dfl)
    P = ctypes.c_void_p
    a = P(1 << 24)
    need = L.dflash_workspace_bytes(ctypes.byref(cfg), 2, 8, 4)

    def call(N=4, hid=a, B=2, K=8, nbytes=need, ws=a):
        return L.dflash_draft_block_inject(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv),
                                           hid, a, a, N, a, a, B, K, a, a, None, ws, nbytes, None)

    assert call(N=-1) == -2
    assert call(K=1) == -3
    assert call(B=0, N=0) == 0                  # nothing to do
    assert call(hid=P(0)) == -1                 # rows without hidden states
    assert call(hid=P((1 << 24) + 2)) == -7     # misaligned hidden states
    assert call(N=5) == -4                      # more rows than the workspace holds
    assert call(nbytes=need - 1) == -4
    assert call(ws=P((1 << 24) + 4)) == -7
    # the workspace of a larger injection capacity holds the pass with rows
    assert L.dflash_workspace_bytes(ctypes.byref(cfg), 2, 8, 64) >= need


def test_inject_select_accept_linear_host_checks(dfl):
    L = dfl.lib()
    cfg = _cfg(dfl)
    w = _fake_weights(dfl, cfg)
    kv = _fake_kv(dfl)
    P = ctypes.c_void_p
    a = P(1 << 24)
    assert L.dflash_inject_context(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), a, a, a,
                                   0, a, 1 << 30, None) == 0          # N = 0: no-op
    assert L.dflash_inject_context(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), a, a, a,
                                   -1, a, 1 << 30, None) == -2
    assert L.dflash_inject_context(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), P(0), a,
                                   a, 4, a, 1 << 30, None) == -1
    need = L.dflash_workspace_bytes(ctypes.byref(cfg), 1, 2, 4)
    assert L.dflash_inject_context(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), a, a, a,
                                   4, a, need - 256, None) == -4
    assert L.dflash_select_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 1, 1, a, a, a,
                                1 << 30, None) == -3
    assert L.dflash_select_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 1, 8, P(0), a, a,
                                1 << 30, None) == -1
    assert L.dflash_accept_greedy(a, a, 3, 1, 8, 100, a, a, a, 1 << 20, None) == -5
    assert L.dflash_accept_greedy(a, a, 0, 1, 40, 100, a, a, a, 1 << 20, None) == -3
    assert L.dflash_accept_greedy(a, a, 0, 1, 8, 100, a, a, a, 16, None) == -4
    assert L.dflash_accept_greedy_noalloc(a, a, 0, 64, 32, 151936, a, a, None) == -4
    assert L.dflash_linear(1, a, 128, 100, a, 8, 1, a, None) == -2      # K_in % 64
    assert L.dflash_linear(1, a, 128, 128, a, 8, 3, a, None) == -2      # splits must divide
    assert L.dflash_linear(1, P((1 << 24) + 8), 128, 128, a, 8, 1, a, None) == -7
    assert L.dflash_linear_splits(4096, 8, 4096) >= 1
    assert L.dflash_read_device_status(None, None) == -1


def test_sampling_host_checks(dfl):
    L = dfl.lib()
    cfg = _cfg(dfl)
    w = _fake_weights(dfl, cfg)
    P = ctypes.c_void_p
    a = P(1 << 24)
    big = 1 << 30
    assert L.dflash_sample_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 0, 8, a, a, a, a,
                                big, None) == 0                       # B = 0: no-op
    assert L.dflash_sample_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 1, 1, a, a, a, a,
                                big, None) == -3                      # K < 2
    assert L.dflash_sample_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 1, 8, P(0), a, a, a,
                                big, None) == -1                      # no uniforms
    assert L.dflash_sample_path(ctypes.byref(cfg), ctypes.byref(w), a, a, a, 1, 8, a, a, a, a,
                                16, None) == -4                       # workspace too small
    assert L.dflash_accept_sample(a, a, a, a, 3, 1, 8, 100, 4, a, a, a, a, big, None) == -5
    assert L.dflash_accept_sample(a, a, a, a, 0, 1, 40, 100, 4, a, a, a, a, big, None) == -3
    assert L.dflash_accept_sample(a, a, a, a, 0, 1, 8, 100, 33, a, a, a, a, big, None) == -2
    assert L.dflash_accept_sample(a, a, a, a, 0, 1, 8, 100, 4, P(0), a, a, a, big, None) == -1
    assert L.dflash_accept_sample(a, a, a, a, 0, 1, 8, 100, 4, a, a, a, a, 16, None) == -4


def test_launch_counter_resets(dfl):
    L = dfl.lib()
    L.dflash_launch_count(1)
    assert L.dflash_launch_count(0) == 0


def test_q4_host_checks(dfl):
    """4-bit weights: the config's weight_bits (0 or 4, bf16 storage only), the
    record pointer of every projection, dflash_linear_q4's shape rules; all
    refused before any launch."""
    L = dfl.lib()
    P = ctypes.c_void_p
    a = P(1 << 24)
    kv = _fake_kv(dfl)
    need = 1 << 40

    def draft(cfg, w):
        return L.dflash_draft_block(ctypes.byref(cfg), ctypes.byref(w), ctypes.byref(kv), a, a,
                                    2, 8, a, a, None, a, need, None)

    cfg = _cfg(dfl, weight_bits=3)
    assert draft(cfg, _fake_weights(dfl, cfg)) == -5
    cfg = _cfg(dfl, weight_bits=4, dtype=0)                 # float32 storage
    assert draft(cfg, _fake_weights(dfl, cfg)) == -5
    cfg = _cfg(dfl, weight_bits=4)
    w = _fake_weights(dfl, cfg)                             # storage-dtype pointers only
    assert draft(cfg, w) == -1
    base = 1 << 26
    for n in dfl._lib.Q4_TOP:
        getattr(w, n + "_q4").data = base
        base += 8192
    for l in range(cfg.n_layers):
        for n in dfl._lib.Q4_LAYER:
            getattr(w.layer[l], n + "_q4").data = base
            base += 8192
    w.layer[1].w_down_q4.data = base + 8                    # misaligned
    assert draft(cfg, w) == -7
    w.layer[1].w_down_q4.data = base
    w.layer[0].wo_q4.data = 0
    assert draft(cfg, w) == -1
    # the 4-bit product
    q = dfl._lib.Q4()
    q.data = 1 << 24
    assert L.dflash_linear_q4(q, 128, 500, a, 8, 1, a, None) == -2     # K % 64
    assert L.dflash_linear_q4(q, 128, 512, a, 8, 3, a, None) == -2     # splits must divide
    assert L.dflash_linear_q4(q, 128, 512, a, 0, 1, a, None) == 0      # no tokens
    assert L.dflash_linear_q4(q, 128, 512, P(0), 8, 1, a, None) == -1
    q.data = (1 << 24) + 4
    assert L.dflash_linear_q4(q, 128, 512, a, 8, 1, a, None) == -7


def test_pack_q4_layout(dfl):
    """The binding's 4-bit packing follows the header: rows padded to 128, one
    2304-byte record per (64-row block, group of 64 inputs), row block major; in
    a record, row i's 32 code bytes then its (scale, bias) word at 2048 + 4i; in
    the word of features 8j..8j+7, (word >> 4k) & 0xF and (word >> (16 + 4k)) & 0xF
    are the codes of features 8j+2k and 8j+2k+1."""
    import numpy as np
    import torch
    g = np.random.default_rng(0)
    N, K = 70, 192
    q = g.integers(0, 16, (N, K)).astype(np.uint8)
    s = torch.tensor(g.uniform(0.001, 1.0, (N, K // 64)), dtype=torch.float32).to(torch.bfloat16)
    b = torch.tensor(g.standard_normal((N, K // 64)), dtype=torch.float32).to(torch.bfloat16)
    data = dfl.pack_q4(q, s.float().numpy(), b.float().numpy()).numpy()
    G = K // 64
    assert data.shape == (2 * G * 2304,)                   # 70 rows -> 128 -> 2 blocks
    sbits = s.view(torch.int16).numpy().astype(np.uint16)
    bbits = b.view(torch.int16).numpy().astype(np.uint16)
    for n in range(N):
        for grp in range(G):
            rec = data[((n // 64) * G + grp) * 2304:][:2304]
            i = n % 64
            words = rec[32 * i:32 * i + 32].view("<u4")
            for j in range(8):
                w = int(words[j])
                for k in range(4):
                    assert (w >> (4 * k)) & 15 == q[n, 64 * grp + 8 * j + 2 * k]
                    assert (w >> (16 + 4 * k)) & 15 == q[n, 64 * grp + 8 * j + 2 * k + 1]
            sw = int(rec[2048 + 4 * i:2052 + 4 * i].view("<u4")[0])
            assert sw & 0xFFFF == sbits[n, grp] and sw >> 16 == bbits[n, grp]
