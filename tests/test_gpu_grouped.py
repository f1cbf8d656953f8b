"""GPU parity of the grouped projection (several weight groups sharing one
activation, one quantization of X, one GEMM launch, a global scale per
group).

Each group's columns must equal, bit for bit, a separate nvfp4_linear call
on that group (same g_x, same per-element arithmetic), and lie within
|y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2 of the oracle's FP64
contraction with that group's own global scale.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, tile_covering_rows
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _groups(nv, ns, K, seed, std_step=0.01):
    """Weights of different spreads (so the global scales differ)."""
    ws = [workloads.make_w(n, K, seed=seed + i, std=0.02 + std_step * i) for i, n in enumerate(ns)]
    q = [nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4) for w in ws]
    return ws, q


def _check(nv, oracle_mod, M, ns, K, mode, seed, rows=None):
    x = workloads.make_x("outlier", M, K, seed=seed)
    ws, q = _groups(nv, ns, K, seed + 100)
    Wq, Ws, g, gn = nv.pack_weight_groups(q)
    assert len(set(float(t[2].item()) for t in q)) == len(ns)  # distinct scales
    xd = x.cuda()
    Y = nv.nvfp4_linear_grouped(xd, Wq, Ws, g, gn, mode=mode)
    xb = bf16_bits(x)
    gx = oracle_mod.global_scale(xb)
    xq, xs = oracle_mod.quantize(xb, gx)
    c0 = 0
    for (w, (wq_d, ws_d, gw_d)), n in zip(zip(ws, q), ns):
        y_sep = nv.nvfp4_linear(xd, wq_d, ws_d, gw_d, mode=mode)
        assert torch.equal(Y[:, c0:c0 + n].view(torch.int16), y_sep.view(torch.int16)), \
            "group at column %d differs from its separate linear" % c0
        wb = bf16_bits(w)
        gw = oracle_mod.global_scale(wb)
        assert np.float32(gw) == np.float32(gw_d.item())
        wq, wsc = oracle_mod.quantize(wb, gw)
        yb = bf16_bits(Y[:, c0:c0 + n])
        if rows is None:
            y_ref = oracle_mod.gemm(xq, xs, gx, wq, wsc, gw)
        else:
            y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, wsc, gw, rows)
            yb = yb[rows]
        check_gemm_tolerance(yb, y_ref, "group at %d, M=%d" % (c0, M))
        c0 += n
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M", [1, 3, 64, 129, 300])
@pytest.mark.parametrize("mode", [0, 1])
def test_grouped_equals_separate_and_oracle(nv, oracle_mod, M, mode):
    _check(nv, oracle_mod, M, (512, 256, 256), 512, mode, seed=M * 3 + mode)


def test_grouped_one_group_equals_linear(nv, oracle_mod):
    _check(nv, oracle_mod, 257, (768,), 768, 0, seed=9)


def test_grouped_eight_groups(nv, oracle_mod):
    _check(nv, oracle_mod, 200, (256,) * 8, 256, 0, seed=21)


def test_full_size_dit_qkv(nv, oracle_mod):
    """The DiT attention projections: 4096 tokens, 3072 -> 3 x 3072."""
    M = 4096
    rows = tile_covering_rows(M, 128, seed=5)
    _check(nv, oracle_mod, M, (3072, 3072, 3072), 3072, 0, seed=31, rows=rows)
