"""Back-to-back nvfp4_linear calls on one stream and one workspace, each with
a different activation, must each give exactly the Y of the same call made
alone (synchronized before and after).

The calls form a programmatic-dependent launch chain: the next call's
kernels may be resident, and run their set-up, while the previous call's
GEMM still reads the workspace. A kernel that touched the workspace before
its dependency wait would corrupt that GEMM's operand; with one activation
repeated (as in a timing loop) such a race leaves Y unchanged, so every
call here uses its own X. Sizes: the cooperative quantizer with its
barrier counter (prefill and square shapes), the one-cluster and the small
quantizers (decode rows), and the fused decode kernel.
"""
import pytest
import torch

from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


@pytest.mark.parametrize("M,N,K,mode,calls", [
    (4096, 5120, 5120, 0, 6),
    (16384, 16384, 16384, 0, 4),
    (32, 27648, 5120, 0, 6),
    (8, 27648, 5120, 0, 6),
    (8, 27648, 5120, 1, 6),
])
def test_chained_calls_equal_isolated_calls(nv, M, N, K, mode, calls):
    w = workloads.make_w(N, K, seed=N + K, device="cuda")
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w, nv.SF_MMA_128x4)
    del w
    nx = min(calls, 3)  # distinct activations, used in rotation
    xs = [workloads.make_x("outlier" if i % 2 else "token_scaled", M, K, seed=100 + i,
                           device="cuda") for i in range(nx)]
    ws = torch.empty(nv.linear_workspace_bytes(M, N, K, mode), dtype=torch.uint8,
                     device="cuda")
    # isolated: one call at a time
    ref = []
    for i in range(nx):
        torch.cuda.synchronize()
        ref.append(nv.nvfp4_linear(xs[i], Wq, Ws, gw, mode=mode, workspace=ws).clone())
        torch.cuda.synchronize()
    # chained: all calls queued back to back, each with its own output
    ys = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(calls)]
    torch.cuda.synchronize()
    for i in range(calls):
        nv.nvfp4_linear(xs[i % nx], Wq, Ws, gw, mode=mode, Y=ys[i], workspace=ws)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    for i in range(calls):
        assert torch.equal(ys[i].view(torch.int16), ref[i % nx].view(torch.int16)), \
            "chained call %d differs from the same call made alone" % i
