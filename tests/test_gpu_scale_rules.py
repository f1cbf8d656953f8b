"""GPU parity of the four-over-six and MSE block-scale rules: codes and
scales bit-exact against the oracle (same binary32 steps for the codes,
the same binary64 error sums and tie rule for the choice), in both scale
layouts; a linear layer on MSE-quantized weights within the GEMM tolerance
of the oracle and closer to the unquantized product than absmax."""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, sf_rowmajor_to_mma, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu

RULES = [1, 2]  # four-over-six, MSE


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _special_rows(K):
    """Rows that reach the edge cases: all zero, tiny values (subnormal
    scales), blocks whose maximum saturates the scale, signed zeros, a
    single non-zero value, values exactly on the grid."""
    rows = [np.zeros(K, np.float32),
            np.full(K, 1e-30, np.float32),
            np.linspace(-3e4, 3e4, K).astype(np.float32),
            np.where(np.arange(K) % 2 == 0, -0.0, 0.0).astype(np.float32),
            np.where(np.arange(K) % 16 == 5, 7.0, 0.0).astype(np.float32),
            np.tile(np.array([6, 4, 3, 2, 1.5, 1, .5, 0] * 2, np.float32), K // 16),
            np.full(K, 4.0, np.float32)]
    return np.stack(rows)


@pytest.mark.parametrize("rule", RULES)
@pytest.mark.parametrize("kind", ["normal", "outlier", "token_scaled"])
@pytest.mark.parametrize("layout", [0, 1])
def test_rule_matches_oracle(nv, oracle_mod, rule, kind, layout):
    M, K = 200, 512
    x = workloads.make_x(kind, M, K, seed=rule * 10 + len(kind) + layout).float().numpy()
    x = np.concatenate([x, _special_rows(K)])
    xb = torch.from_numpy(x).to(torch.bfloat16)
    bits = bf16_bits(xb)
    g = oracle_mod.global_scale(bits)
    q_ref, s_ref = oracle_mod.quantize(bits, g, rule)
    gd = torch.tensor([g], dtype=torch.float32, device="cuda")
    q, s = nv.nvfp4_quantize(xb.cuda(), gd, layout, rule=rule)
    assert np.array_equal(to_np_u8(q), q_ref)
    want = s_ref if layout == 0 else sf_rowmajor_to_mma(s_ref)
    assert np.array_equal(to_np_u8(s).reshape(want.shape), want)
    # a given, much larger g: small and subnormal block scales
    g2 = g * 300.0
    q_ref2, s_ref2 = oracle_mod.quantize(bits, float(np.float32(g2)), rule)
    q2, s2 = nv.nvfp4_quantize(xb.cuda(), torch.tensor([g2], dtype=torch.float32,
                                                       device="cuda"), 0, rule=rule)
    assert np.array_equal(to_np_u8(q2), q_ref2) and np.array_equal(to_np_u8(s2), s_ref2)
    assert nv.nvfp4_device_error() == 0


def test_absmax_rule_is_nvfp4_quantize(nv):
    x = workloads.make_x("outlier", 64, 256, seed=3).cuda()
    g = nv.nvfp4_global_scale(x)
    a = nv.nvfp4_quantize(x, g, 1)
    b = nv.nvfp4_quantize(x, g, 1, rule=0)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("rule", RULES)
def test_full_size_weight_sampled_rows(nv, oracle_mod, rule):
    """The 5120 x 5120 prefill weight quantized on the GPU; sampled rows
    (the rule is row-local) against the oracle."""
    w_ = workloads.WORKLOADS["prefill"]
    W = workloads.make_w(5120, w_.K, workloads.w_seed(w_))
    Wq, Ws, gw = nv.nvfp4_quantize_weight(W.cuda(), 0, rule=rule)
    bits = bf16_bits(W)
    g = oracle_mod.global_scale(bits)
    assert np.float32(g) == np.float32(gw.item())
    rows = np.unique(np.concatenate([[0, 5119],
                                     np.random.default_rng(rule).choice(5120, 30, replace=False)]))
    q_ref, s_ref = oracle_mod.quantize(bits[rows], g, rule)
    assert np.array_equal(to_np_u8(Wq)[rows], q_ref)
    assert np.array_equal(to_np_u8(Ws)[rows], s_ref)
    assert nv.nvfp4_device_error() == 0


def test_linear_on_mse_weights(nv, oracle_mod):
    M, N, K = 300, 512, 1024
    x = workloads.make_x("outlier", M, K, seed=61)
    w = workloads.make_w(N, K, seed=62)
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    exact = x.double().numpy() @ w.double().numpy().T
    errs = {}
    for rule in (0, 2):
        wq, ws = oracle_mod.quantize(wb, gw, rule)
        Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4, rule=rule)
        assert np.array_equal(to_np_u8(Wq), wq)
        y = nv.nvfp4_linear(x.cuda(), Wq, Ws, g_w)
        check_gemm_tolerance(bf16_bits(y), oracle_mod.gemm(xq, xs, gx, wq, ws, gw),
                             "rule %d" % rule)
        errs[rule] = float(np.linalg.norm(y.double().cpu().numpy() - exact))
    assert errs[2] < errs[0]
    assert nv.nvfp4_device_error() == 0
