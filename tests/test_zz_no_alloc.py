"""nvfp4_linear_noalloc: the linear layer for callers that cannot allocate
device memory (it keeps its scratch in a fixed array inside the library).

Called through the C ABI twice in a row -- a larger problem, then a smaller
one that lands on the stale contents the first call left in the shared
array -- and checked against nvfp4_linear, the entry point with a
caller-provided workspace. Both run the same kernels on the same inputs, so
the outputs must be bitwise equal (which is also within the GEMM tolerance
the other tests use).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    return nv


def _call_noalloc(lib, X, Wq, Ws, gw, Y):
    st = torch.cuda.current_stream().cuda_stream
    return lib.nvfp4_linear_noalloc(X.data_ptr(), X.shape[0], X.shape[1], X.stride(0),
                                    Wq.data_ptr(), Ws.data_ptr(), gw.data_ptr(), Wq.shape[0],
                                    Y.data_ptr(), Y.stride(0), None, ctypes.c_void_p(st))


@pytest.mark.parametrize("shapes", [((300, 520, 768), (64, 256, 512))])
def test_noalloc_matches_linear_on_two_calls(nv, shapes):
    lib = nv.load_library()
    for i, (M, N, K) in enumerate(shapes):
        X = workloads.make_x("outlier", M, K, seed=900 + i).cuda()
        W = workloads.make_w(N, K, seed=950 + i).cuda()
        Wq, Ws, gw = nv.nvfp4_quantize_weight(W, nv.SF_MMA_128x4)
        y_ref = nv.nvfp4_linear(X, Wq, Ws, gw)
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, X, Wq, Ws, gw, Y) == 0
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), y_ref.view(torch.int16)), \
            "noalloc call %d differs from nvfp4_linear" % (i + 1)
        check_gemm_tolerance(bf16_bits(Y), bf16_bits(y_ref), "noalloc call %d" % (i + 1))
    assert nv.nvfp4_device_error() == 0


def test_noalloc_rejects_sizes_beyond_its_scratch(nv):
    lib = nv.load_library()
    # 8192 x 8192 needs 36 MiB of scratch; rejected before any launch
    st = torch.cuda.current_stream().cuda_stream
    rc = lib.nvfp4_linear_noalloc(0x10000, 8192, 8192, 8192, 0x10000, 0x10000, 0x10000, 256,
                                  0x10000, 256, None, ctypes.c_void_p(st))
    assert rc == 4  # NVFP4_ERR_WORKSPACE_TOO_SMALL
