"""The projection GEMM (dflash_linear) against a float64 matmul of the same
bf16 / f32 operands: ragged shapes across tiles and splits, and the full-size
lm_head (151936 x 4096, 7 tokens) on sampled output rows."""

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _operands(N, K, T, dtype, seed):
    cfg = dict(synth.preset("tiny"), dtype=dtype)
    W = synth.gen._normal(seed, "gemm_w", (N, K), 0.0, 0.05, dtype)
    X = synth.gen._normal(seed, "gemm_x", (T, K), 0.0, 1.0, dtype)
    del cfg
    return W, X


def _run(W, X, S, dtype):
    import block_diffusion_drafter_inject_gb300 as dfl
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    Wd = torch.from_numpy(W).to(td).cuda()
    Xd = torch.from_numpy(X).to(td).cuda()
    out = torch.full((S, X.shape[0], W.shape[0]), float("nan"), device="cuda")
    dfl.linear(Wd, Xd, out, S)
    torch.cuda.synchronize()
    return out.double().sum(0).cpu().numpy()


@pytest.mark.parametrize("N,K,T,S,dtype", [
    (128, 64, 1, 1, "bf16"),
    (300, 256, 7, 2, "bf16"),
    (1000, 512, 16, 4, "bf16"),
    (520, 768, 33, 3, "bf16"),
    (257, 1024, 100, 8, "bf16"),
    (384, 512, 256, 1, "bf16"),
    (200, 320, 300, 5, "bf16"),
    (96, 256, 9, 2, "f32"),
])
def test_linear_matches_float64_matmul(N, K, T, S, dtype):
    W, X = _operands(N, K, T, dtype, seed=N + T)
    got = _run(W, X, S, dtype)
    want = X.astype(np.float64) @ W.astype(np.float64).T
    err = np.max(np.abs(got - want)) / np.max(np.abs(want))
    assert err < 1e-5, err


def test_linear_default_splits_are_valid():
    import block_diffusion_drafter_inject_gb300 as dfl
    for (N, T, K) in [(4096, 8, 14336), (28672, 8, 4096), (6144, 256, 4096), (512, 113, 4096)]:
        S = dfl.linear_splits(N, T, K)
        assert S >= 1 and (K // 64) % S == 0


def test_lm_head_full_size_sampled_rows():
    cfg = synth.preset("full")
    V, D, T = cfg["vocab"], cfg["d_model"], 7
    W = synth.make_weights(cfg, seed=0, names={"lm_head"})["lm_head"]
    X = synth.gen._normal(0, "lm_x", (T, D), 0.0, 1.0, "bf16")
    import block_diffusion_drafter_inject_gb300 as dfl
    S = dfl.linear_splits(V, T, D)
    got = _run(W, X, S, "bf16")
    rows = np.concatenate([np.random.default_rng(0).integers(0, V, 60), np.arange(V - 4, V)])
    want = X.astype(np.float64) @ W[rows].astype(np.float64).T
    err = np.max(np.abs(got[:, rows] - want)) / np.max(np.abs(want))
    assert err < 1e-5, err
