"""GPU parity of the GEMM for M > 128 on shapes aimed at the tiling: the
CTA-pair kernel (256 x 256 tiles, the partial last wave as 256 x 128
column halves) and the single-CTA kernel (128 x 256 tiles).

Every shape is checked against the oracle within
|y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2, and the two kernels
bitwise against each other (they issue the same K = 64 MMAs in K order; a
column computed by an N = 128 instruction in one and an N = 256 one in the
other gets the same bits). The shapes cover N tails of every width below a
tile, M tails that leave the second CTA of a pair without rows, K of a
single stage, more tiles than CTA pairs (a partial last wave), a strided
output, weight groups, and the bounded-wait timeout of the CTA-pair kernel.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, tile_covering_rows
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu

PAIR, SINGLE = 0, 1


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _select(nv, kernel):
    assert nv.load_library().nvfp4_debug_select_gemm_kernel(kernel) == 0


SHAPES = [  # (M, N, K)
    (260, 100, 512),     # one tile column, 100 of 256 columns valid
    (257, 640, 256),     # 2.5 tile columns, K of one stage
    (513, 1152, 768),    # 4.5 tile columns
    (129, 385, 512),     # one valid column past a whole tile; rank-1 CTAs see only padding rows
    (384, 767, 1280),    # 255 of 256 columns in the last tile
    (1000, 900, 512),    # 132 valid columns in the last tile
    (2048, 3840, 512),   # 120 tiles on 74 pairs: a partial last wave as column halves
    (300, 5120, 1024),   # the prefill column count
]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_pair_kernel_matches_oracle_and_single_cta_kernel(nv, oracle_mod, M, N, K):
    x = workloads.make_x("outlier", M, K, seed=M * 13 + N)
    w = workloads.make_w(N, K, seed=N * 3 + K)
    xd = x.cuda()
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    try:
        y = nv.nvfp4_linear(xd, Wq, Ws, gw)
        _select(nv, SINGLE)
        y_single = nv.nvfp4_linear(xd, Wq, Ws, gw)
    finally:
        _select(nv, PAIR)
    assert nv.nvfp4_device_error() == 0
    assert torch.equal(y.view(torch.int16), y_single.view(torch.int16))
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gwo = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gwo)
    rows = np.arange(M) if M <= 1024 else tile_covering_rows(M, 32)
    y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, ws, gwo, rows)
    check_gemm_tolerance(bf16_bits(y)[rows], y_ref, "pair %dx%dx%d" % (M, N, K))


def test_pair_kernel_on_strided_output(nv, oracle_mod):
    """Y with a leading dimension that is not a multiple of 8 (no TMA
    stores: the direct-store path of the epilogue)."""
    M, N, K = 300, 520, 512
    x = workloads.make_x("normal", M, K, seed=5)
    w = workloads.make_w(N, K, seed=6)
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    big = torch.full((M, N + 3), float("nan"), dtype=torch.bfloat16, device="cuda")
    Y = big[:, 1:N + 1]
    nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, Y=Y)
    y_ref = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw)
    assert torch.equal(Y.contiguous().view(torch.int16), y_ref.view(torch.int16))
    assert torch.isnan(big[:, 0].float()).all() and torch.isnan(big[:, N + 1:].float()).all()


def test_groups_of_mixed_sizes(nv, oracle_mod):
    """Four groups of 256 to 768 columns with their own global scales, each
    equal to its own linear."""
    M, K = 300, 512
    ns = (256, 512, 256, 768)
    ws = [workloads.make_w(n, K, seed=70 + i, std=0.02 + 0.01 * i) for i, n in enumerate(ns)]
    q = [nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4) for w in ws]
    Wq, Ws, g, gn = nv.pack_weight_groups(q)
    x = workloads.make_x("token_scaled", M, K, seed=71).cuda()
    Y = nv.nvfp4_linear_grouped(x, Wq, Ws, g, gn)
    c0 = 0
    for (wq_d, ws_d, gw_d), n in zip(q, ns):
        y_sep = nv.nvfp4_linear(x, wq_d, ws_d, gw_d)
        assert torch.equal(Y[:, c0:c0 + n].view(torch.int16), y_sep.view(torch.int16))
        c0 += n
    assert nv.nvfp4_device_error() == 0


def test_pair_kernel_bounded_wait_timeout(nv, oracle_mod):
    """The producers issue nothing: every wait of the CTA-pair kernel runs
    out, the kernel records a timeout and returns; the next call is correct."""
    M, N, K = 512, 768, 512
    x = workloads.make_x("normal", M, K, seed=1)
    w = workloads.make_w(N, K, seed=2)
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    g = nv.nvfp4_global_scale(x.cuda())
    torch.cuda.synchronize()
    nv.nvfp4_device_error(clear=True)
    try:
        nv.nvfp4_debug_set_fault_injection(1, 20000)  # 20 ms waits
        nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, g_x=g)
        assert nv.nvfp4_device_error(clear=True) == 6  # NVFP4_ERR_TIMEOUT
    finally:
        nv.nvfp4_debug_set_fault_injection(0, 0)
    y = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw)
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gwo = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gwo)
    check_gemm_tolerance(bf16_bits(y), oracle_mod.gemm(xq, xs, gx, wq, ws, gwo), "after timeout")
    assert nv.nvfp4_device_error() == 0
