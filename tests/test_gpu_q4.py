"""GPU parity of the 4-bit drafter (weights w = bf16(s*q + b), one (s, b) per row
and group of 64 input features; README mirror, MLX section): the projection GEMM
alone against the oracle's dequantized product, bit-exact on one-hot inputs
(which read single weights back), and whole cycles against the oracle run on the
dequantized weights, with the tolerances of test_gpu_parity."""

import numpy as np
import pytest

import oracle
import synth
from _cases import Case, rowmax_rel, topk_compare

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TOL = 2e-2
KV_TOL = 1.6e-2


def _q4(N, K, seed):
    g = np.random.default_rng(seed)
    q = g.integers(0, 16, (N, K)).astype(np.uint8)
    s = torch.from_numpy(g.uniform(0.002, 0.006, (N, K // 64)).astype(np.float32))
    s = s.to(torch.bfloat16).float().numpy()
    b = torch.from_numpy((-7.5 * s + 0.002 * g.standard_normal((N, K // 64))).astype(np.float32))
    b = b.to(torch.bfloat16).float().numpy()
    return q, s, b


def _run(q, s, b, X, splits):
    import block_diffusion_drafter_inject_gb300 as dfl
    data = dfl.pack_q4(q, s, b).cuda()
    T = X.shape[0]
    out = torch.zeros((splits, T, q.shape[0]), dtype=torch.float32, device="cuda")
    dfl.linear_q4(data, q.shape[0], X, out, splits)
    torch.cuda.synchronize()
    return out.double().sum(0).cpu().numpy()


@pytest.mark.parametrize("N,K,T,splits", [
    (384, 512, 1, 1), (384, 512, 7, 2), (260, 512, 16, 4), (512, 1024, 33, 2),
    (384, 256, 64, 1), (256, 512, 200, 2), (128, 512, 300, 1), (70, 192, 20, 3),
])
def test_linear_q4_matches_dequantized_product(N, K, T, splits):
    """Token tiles 16..128, K slices, weight tails (260, 70 rows): within fp32
    accumulation of the bf16 products of the oracle's dequantized weights."""
    q, s, b = _q4(N, K, seed=N + K + T)
    Xh = np.random.default_rng(T).standard_normal((T, K)).astype(np.float32)
    X = torch.from_numpy(Xh).to(torch.bfloat16).cuda()
    Xb = X.double().cpu().numpy()
    W = oracle.dequantize_affine(q, s, b, 64)
    want = Xb @ W.T
    got = _run(q, s, b, X, splits)
    scale = np.abs(Xb) @ np.abs(W).T
    assert np.max(np.abs(got - want) / scale) < 1e-5


def test_linear_q4_reads_every_weight_exactly():
    """One-hot rows x_t = e_k return column k of the weights: bit-exact against the
    oracle's bf16(s*q + b) for every input feature of two groups, every row
    (nibble order, swizzled tile, scale and bias of the right group, rounding)."""
    N, K = 256, 512
    q, s, b = _q4(N, K, seed=3)
    ks = np.concatenate([np.arange(0, 64), np.arange(448, 512)])
    Xh = np.zeros((len(ks), K), np.float32)
    Xh[np.arange(len(ks)), ks] = 1.0
    X = torch.from_numpy(Xh).to(torch.bfloat16).cuda()
    got = _run(q, s, b, X, 1)
    W = oracle.dequantize_affine(q, s, b, 64)
    np.testing.assert_array_equal(got, W[:, ks].T)


CASES = [
    ("tiny_bf16", 1, 8, [64]),
    ("tiny_bf16", 3, 8, [5, 90, 64]),
    ("small", 2, 16, [130, 7]),          # SwiGLU width 1344: 21 gate tiles; vocab 5000
    ("small_gqa", 2, 8, [200, 129]),
]


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("name,B,K,ctx", CASES)
def test_q4_cycle_matches_oracle(name, B, K, ctx, fused):
    """A whole cycle with every projection (fc, QKV, O, gate/up, down, lm_head) in
    4 bits: injected K/V, logits (against the contract oracle and the unrounded
    one), top-k and path as the oracle's on the dequantized weights."""
    c = Case(name, B, K, ctx, seed=len(ctx) + K + 40, weight_bits=4).device()
    g = c.run_device(fused=fused)
    assert g["status"] == 0
    o = c.oracle()
    gk, gv = c.gpu_kv_dense()
    for b in range(B):
        if c.ctx[b] == 0:
            continue
        for l in range(c.cfg["n_layers"]):
            assert rowmax_rel(gk[b][l], o["ck"][b][l]) < KV_TOL, (b, l)
            assert rowmax_rel(gv[b][l], o["cv"][b][l]) < KV_TOL, (b, l)
    err = rowmax_rel(g["logits"], o["logits"])
    assert err < TOL, err
    err = rowmax_rel(g["logits"], c.oracle_pure_logits())
    assert err < TOL, err
    compared, bad = topk_compare(g["ids"], o["logits"], o["ids"], c.cfg["top_k"])
    assert compared > 0 and bad == 0, (compared, bad)
    acc, toks = oracle.accept_greedy(g["path"], c.target)
    np.testing.assert_array_equal(g["acc"], acc)
