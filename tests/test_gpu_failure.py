"""The GEMM's bounded waits made to run out on the GPU, without a fault: the
tensor-core issuer waits on a barrier that nothing arrives on, with a 20 ms
limit.  The kernel must give up, drain what it issued, report
DFLASH_DEV_TIMEOUT in the status word and return; the context stays usable
and an ordinary launch afterwards is clean and correct."""

import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

TIMEOUT_BIT = 8     # DFLASH_DEV_TIMEOUT


def _call(dfl, W, X, out, ws, stall_us):
    N, Kin = W.shape
    T = X.shape[0]
    rc = dfl.lib().dflash_test_linear_wait(
        ctypes.c_void_p(W.data_ptr()), N, Kin, ctypes.c_void_p(X.data_ptr()), T,
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(), stall_us,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, rc
    torch.cuda.synchronize()
    return int(ws[:4].view(torch.int32).item())


@pytest.mark.parametrize("N,Kin,T", [(256, 64, 8), (384, 4096, 16), (1024, 8192, 40)])
def test_wait_runs_out_then_context_is_clean(N, Kin, T):
    import block_diffusion_drafter_inject_gb300 as dfl
    g = torch.Generator(device="cuda").manual_seed(N + T)
    W = (torch.randn((N, Kin), device="cuda", generator=g) * 0.05).to(torch.bfloat16)
    X = torch.randn((T, Kin), device="cuda", generator=g).to(torch.bfloat16)
    out = torch.zeros((T, N), device="cuda", dtype=torch.float32)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    assert _call(dfl, W, X, out, ws, 20000) & TIMEOUT_BIT          # gave up, reported
    ws.zero_()
    assert _call(dfl, W, X, out, ws, 0) == 0                       # ordinary launch: clean
    ref = X.float() @ W.float().t()
    err = (out - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-4, err           # fp32 sums in another order than torch's
