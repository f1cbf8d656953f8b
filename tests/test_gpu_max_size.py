"""The quantizers and the linear layer at the largest activation the C ABI
accepts: just under 2^28 16-element blocks (262143 x 16384, 8.6 GB of
bfloat16), where every element, vector and block index of the kernels'
32-bit arithmetic is near its top.

The largest |x| is planted at the very last element and a near-largest one
just past element 2^31, so the global scale, checked against its closed form
amax / 2688 (one binary32 division), shows that the reductions reached both.
Sampled rows at the start, around the 2^31-element boundary and at the end
are compared with the oracle: codes and tile-layout scales byte for byte,
Y within the GEMM tolerance.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu

M, K, N = 262143, 16384, 256                      # M * K / 16 = 2^28 - 1024 blocks
ROWS = np.array([0, 1, 4095, 131071, 131072, 131073, M - 129, M - 128, M - 2, M - 1])
AMAX = 1000.0


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


@pytest.fixture(scope="module")
def big_x():
    x = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(77)
    for r0 in range(0, M, 8192):
        r1 = min(M, r0 + 8192)
        x[r0:r1] = torch.randn((r1 - r0, K), generator=g, device="cuda").to(torch.bfloat16)
    x[M - 1, K - 1] = AMAX                        # the largest |x|: the very last element
    x[131072, 5] = -999.0                         # element 2^31 + 5
    torch.cuda.synchronize()
    yield x
    del x
    torch.cuda.empty_cache()


def _g_closed_form() -> float:
    return float(np.float32(AMAX) / np.float32(2688.0))


def _f32_bits(v: float) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


def _tile_offsets(rows, kb_total):
    """Byte offsets of scales (r, 0 .. kb_total - 1) in the 128x4 tile layout."""
    r = rows[:, None].astype(np.int64)
    j = np.arange(kb_total, dtype=np.int64)[None, :]
    return ((r // 128) * (kb_total // 4) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 \
        + j % 4


def _check_rows(oracle_mod, x, q, sf_flat, g, label):
    xr = bf16_bits(x[torch.from_numpy(ROWS).cuda()])
    q_ref, s_ref = oracle_mod.quantize(xr, g)
    q_rows = to_np_u8(q[torch.from_numpy(ROWS).cuda()])
    assert np.array_equal(q_rows, q_ref), label + ": codes"
    offs = torch.from_numpy(_tile_offsets(ROWS, K // 16).ravel()).cuda()
    s_rows = to_np_u8(sf_flat[offs]).reshape(len(ROWS), K // 16)
    assert np.array_equal(s_rows, s_ref), label + ": scales"
    return q_ref, s_ref


def test_global_scale_and_quantize_at_the_block_limit(nv, oracle_mod, big_x):
    g = nv.nvfp4_global_scale(big_x)
    torch.cuda.synchronize()
    assert _f32_bits(g.item()) == _f32_bits(_g_closed_form())
    q, sf = nv.nvfp4_quantize(big_x, g, nv.SF_MMA_128x4)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    _check_rows(oracle_mod, big_x, q, sf.view(-1), _g_closed_form(), "quantize")
    del q, sf


def test_linear_at_the_block_limit(nv, oracle_mod, big_x):
    w = workloads.make_w(N, K, seed=78)
    wb = bf16_bits(w)
    gwo = oracle_mod.global_scale(wb)
    wq, ws = oracle_mod.quantize(wb, gwo)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    wsp = torch.empty(nv.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    y = nv.nvfp4_linear(big_x, Wq, Ws, g_w, workspace=wsp)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    g = _g_closed_form()
    assert _f32_bits(float(wsp[0:4].view(torch.float32).item())) == _f32_bits(g), "g_x"
    header = 8448
    q = wsp[header:header + M * K // 2].view(M, K // 2)
    sf_off = header + (M * K // 2 + 255) // 256 * 256
    sf_flat = wsp[sf_off:sf_off + (M + 127) // 128 * 128 * K // 16]
    xq, xs = _check_rows(oracle_mod, big_x, q, sf_flat, g, "linear workspace")
    y_ref = oracle_mod.gemm_rows(xq, xs, g, wq, ws, gwo)
    y_rows = bf16_bits(y[torch.from_numpy(ROWS).cuda()])
    check_gemm_tolerance(y_rows, y_ref, "linear %dx%dx%d" % (M, N, K))
    del wsp, y
