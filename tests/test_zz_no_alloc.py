"""The allocation-free acceptance entry point against the workspace one.

dflash_accept_greedy_noalloc serves callers that cannot hand the library a
workspace (memory planned once at start-up, a binding without a device
allocator, or no cudaMalloc allowed where acceptance runs).  It must return
exactly what dflash_accept_greedy returns.  Two calls in a row also check that
the shared fixed scratch carries nothing from one call into the next.  This
file is collected last so that a failure here stops a -x run only after every
other test has run."""

import ctypes

import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _run_both(lib, path, logits, ws):
    B, K, V = logits.shape
    dt = 0 if logits.dtype == torch.float32 else 1
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    acc_ref = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tok_ref = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    acc_na = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    tok_na = torch.full((B, K), -7, dtype=torch.int32, device="cuda")
    rc = lib.dflash_accept_greedy(_ptr(path), _ptr(logits), dt, B, K, V, _ptr(acc_ref),
                                  _ptr(tok_ref), _ptr(ws), ws.numel(), s)
    assert rc == 0
    rc = lib.dflash_accept_greedy_noalloc(_ptr(path), _ptr(logits), dt, B, K, V, _ptr(acc_na),
                                          _ptr(tok_na), s)
    assert rc == 0
    torch.cuda.synchronize()
    return (acc_ref.cpu().numpy(), tok_ref.cpu().numpy(), acc_na.cpu().numpy(),
            tok_na.cpu().numpy())


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_noalloc_accept_matches_workspace_accept_twice(dtype):
    import block_diffusion_drafter_inject_gb300 as dfl
    lib = dfl.lib()
    cfg = synth.preset("full")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for call, (B, K, seed) in enumerate([(4, 8, 11), (3, 16, 12)]):
        logits = torch.from_numpy(synth.make_target_logits(cfg, B, K, seed=seed)).cuda().to(dtype)
        am = logits.float().argmax(dim=-1).to(torch.int32)          # target argmax per row
        # paths that accept 0..K-1 drafts: follow the argmax for a seeded length
        lens = np.random.default_rng(seed).integers(0, K, size=B)
        path = am[:, :K - 1].clone()
        for b in range(B):
            if lens[b] < K - 1:
                path[b, lens[b]] = (path[b, lens[b]] + 1) % cfg["vocab"]
        acc_ref, tok_ref, acc_na, tok_na = _run_both(lib, path.contiguous(), logits.contiguous(), ws)
        np.testing.assert_array_equal(acc_na, acc_ref, err_msg=f"call {call}")
        np.testing.assert_array_equal(tok_na, tok_ref, err_msg=f"call {call}")
        np.testing.assert_array_equal(acc_ref, np.minimum(lens, K - 1) + 1)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import block_diffusion_drafter_inject_gb300 as dfl
    lib = dfl.lib()
    V, K = 151936, 32
    B = 64                                                     # 64*32*19 > 32768 pairs
    path = torch.zeros((B, K - 1), dtype=torch.int32, device="cuda")
    acc = torch.zeros((B,), dtype=torch.int32, device="cuda")
    tok = torch.zeros((B, K), dtype=torch.int32, device="cuda")
    logits = torch.zeros(16, dtype=torch.float32, device="cuda")  # rejected before any read
    rc = lib.dflash_accept_greedy_noalloc(_ptr(path), _ptr(logits), 0, B, K, V, _ptr(acc),
                                          _ptr(tok), ctypes.c_void_p(0))
    assert rc == -4                                            # DFLASH_ERR_WORKSPACE, nothing launched
