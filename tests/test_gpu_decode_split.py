"""GPU parity of the decode GEMM (M <= 128) where the weight tiles of a
partial last round are split by K across the two CTAs of a cluster (the
second CTA's FP32 partial added into the first's in shared memory; up to 8
activation rows, whole tiles only beyond).

Tile counts cover a tail of one tile, a tail of exactly half the SMs, a
tail one tile too large to split (whole tiles only) and a weight smaller
than one round (every tile split). Each output is checked against the
oracle within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2, and the
fused mode (X quantized inside the kernel, M <= 8) bitwise against the
unfused one, which runs the same split.
"""
import numpy as np
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
    nv.nvfp4_device_error(clear=True)
    return nv


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count & ~1


def _case(nv, oracle_mod, M, N, K, seed):
    x = workloads.make_x("outlier", M, K, seed=seed)
    w = workloads.make_w(N, K, seed=seed + 1)
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    y = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw)
    if M <= 8:
        y_f = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, mode=nv.LINEAR_FUSED)
        assert torch.equal(y.view(torch.int16), y_f.view(torch.int16))
    assert nv.nvfp4_device_error() == 0
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gwo = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gwo)
    check_gemm_tolerance(bf16_bits(y), oracle_mod.gemm(xq, xs, gx, wq, ws, gwo),
                         "decode %dx%dx%d" % (M, N, K))


@pytest.mark.parametrize("M", [1, 3, 8, 17, 64])
@pytest.mark.parametrize("tail", ["one", "half", "too_many", "all"])
def test_decode_tail_split(nv, oracle_mod, M, tail):
    G = _sms()
    tiles = {"one": G + 1, "half": G + G // 2, "too_many": G + G // 2 + 1, "all": 5}[tail]
    N = tiles * 128 - 40  # a ragged last tile
    _case(nv, oracle_mod, M, N, 1024, seed=M * 7 + tiles)


@pytest.mark.parametrize("K", [2048, 6144])
def test_decode_tail_split_deeper_k(nv, oracle_mod, K):
    _case(nv, oracle_mod, 4, 700, K, seed=K)
