"""GPU parity of the NVFP4 linear layer with a run-time LoRA correction
(down projection computed in the quantization pass, up projection as
bfloat16 tensor-core steps into the GEMM accumulator).

Y must lie within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2 of the
oracle's FP64 sum of the NVFP4 product and the LoRA term on the unquantized
activation, rounded once to bfloat16. With lora_scale = 0 the result equals
nvfp4_linear (so the fused pass wrote the same codes and scales as the
standalone quantizer).
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _run(nv, oracle_mod, M, N, K, r, scale, seed, rows=None, kind="outlier"):
    x = workloads.make_x(kind, M, K, seed=seed)
    w = workloads.make_w(N, K, seed=seed + 1)
    a, b = workloads.make_lora(r, K, N, seed=seed + 2)
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gw)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    assert np.array_equal(to_np_u8(Wq), wq)
    y = nv.nvfp4_linear_lora(x.cuda(), Wq, Ws, g_w, a.cuda(), b.cuda(), scale)
    y_ref = oracle_mod.linear_lora_rows(xq, xs, gx, wq, ws, gw, xb, bf16_bits(a), bf16_bits(b),
                                        scale, rows)
    yb = bf16_bits(y) if rows is None else bf16_bits(y)[rows]
    max_rel, floor_only = check_gemm_tolerance(yb, y_ref, "lora %dx%dx%d r=%d" % (M, N, K, r))
    assert nv.nvfp4_device_error() == 0
    return x, (Wq, Ws, g_w), (a, b), y, max_rel


@pytest.mark.parametrize("M,N,K,r", [(129, 256, 256, 16), (300, 512, 768, 32),
                                     (513, 768, 1024, 64), (256, 384, 512, 48)])
def test_lora_matches_oracle(nv, oracle_mod, M, N, K, r):
    _run(nv, oracle_mod, M, N, K, r, 1.0, seed=M + N + r)


def test_lora_scale_zero_equals_linear(nv, oracle_mod):
    x, (Wq, Ws, g_w), (a, b), y, _ = _run(nv, oracle_mod, 384, 512, 1024, 32, 0.0, seed=7,
                                          kind="token_scaled")
    y_lin = nv.nvfp4_linear(x.cuda(), Wq, Ws, g_w)
    assert torch.equal(y.float(), y_lin.float())


def test_lora_large_correction_and_given_gx(nv, oracle_mod):
    """A correction larger than the NVFP4 product (scale 16) and a given g_x."""
    M, N, K, r = 300, 256, 512, 64
    x = workloads.make_x("normal", M, K, seed=19)
    w = workloads.make_w(N, K, seed=20)
    a, b = workloads.make_lora(r, K, N, seed=21)
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gw)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    y = nv.nvfp4_linear_lora(x.cuda(), Wq, Ws, g_w, a.cuda(), b.cuda(), 16.0,
                             g_x=torch.tensor([gx], dtype=torch.float32, device="cuda"))
    y_ref = oracle_mod.linear_lora_rows(xq, xs, gx, wq, ws, gw, xb, bf16_bits(a), bf16_bits(b),
                                        16.0)
    check_gemm_tolerance(bf16_bits(y), y_ref, "large correction")
    assert nv.nvfp4_device_error() == 0


def test_full_size_prefill_lora(nv, oracle_mod):
    """The 4096 x 5120 x 5120 layer with a rank-32 LoRA, sampled rows."""
    M = 4096
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(9).choice(M, 14, replace=False)]))
    _run(nv, oracle_mod, M, 5120, 5120, 32, 1.0, seed=101, rows=rows)
