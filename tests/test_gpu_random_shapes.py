"""A seeded sweep of random shapes through the linear entry points, each
checked against the oracle: Y within the GEMM tolerance on every row, and
the quantized activation the call leaves in its workspace (g_x, codes,
tile-layout scales) bit-exact.

The shapes are drawn, not chosen, so that they land where hand-picked cases
might not: any M from 1 to 900 (small, one-cluster and cooperative
quantizers; decode kernel up to 128 rows, with and without the K split of
its partial last round; CTA-pair kernel beyond), any N from 1 to 1300 (a
partial last weight tile of any width), K a multiple of 256 up to 2560,
the dynamic or a given activation scale, and the fused decode mode where it
applies. The dynamic re-quantizing epilogue, the LoRA linear (M > 128, every
rank it supports) and the grouped projections (1 to 4 groups, each group's
columns also bitwise equal to its own linear) get their own draws, and so
does the standalone quantizer (every scale rule, both layouts).
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, sf_rowmajor_to_mma, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu

HEADER = 8448
KINDS = ["outlier", "token_scaled", "normal"]


def _draw(n_cases, seed):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n_cases):
        band = rng.integers(0, 4)
        M = int([rng.integers(1, 9), rng.integers(9, 129), rng.integers(129, 400),
                 rng.integers(400, 901)][band])
        N = int(rng.integers(1, 1301))
        K = int(256 * rng.integers(1, 11))
        given = bool(rng.integers(0, 2))
        fused = bool(M <= 8 and rng.integers(0, 2))
        cases.append((M, N, K, given, fused, KINDS[i % 3], 1000 + i))
    return cases


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _f32_bits(v: float) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


@pytest.mark.parametrize("M,N,K,given,fused,kind,seed", _draw(48, 20261203))
def test_random_linear_matches_oracle(nv, oracle_mod, M, N, K, given, fused, kind, seed):
    x = workloads.make_x(kind, M, K, seed=seed)
    w = workloads.make_w(N, K, seed=seed + 1)
    xb, wb = bf16_bits(x), bf16_bits(w)
    gwo = oracle_mod.global_scale(wb)
    wq, ws = oracle_mod.quantize(wb, gwo)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    assert np.array_equal(to_np_u8(Wq), wq)
    # a given scale deliberately off the tensor's own (some saturation)
    gx = oracle_mod.global_scale(xb) * (0.75 if given else 1.0)
    gx = float(np.float32(gx))
    g_in = torch.tensor([gx], dtype=torch.float32, device="cuda") if given else None
    mode = nv.LINEAR_FUSED if fused else nv.LINEAR_UNFUSED
    wsp = torch.empty(max(nv.linear_workspace_bytes(M, N, K, mode), 1), dtype=torch.uint8,
                      device="cuda")
    y = nv.nvfp4_linear(x.cuda(), Wq, Ws, g_w, g_x=g_in, mode=mode, workspace=wsp)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    xq, xs = oracle_mod.quantize(xb, gx)
    label = "%dx%dx%d given=%s fused=%s" % (M, N, K, given, fused)
    if not fused:
        codes = to_np_u8(wsp[HEADER:HEADER + M * K // 2]).reshape(M, K // 2)
        sf_off = HEADER + (M * K // 2 + 255) // 256 * 256
        rows_pad = (M + 127) // 128 * 128
        sf = to_np_u8(wsp[sf_off:sf_off + rows_pad * K // 16]).reshape(rows_pad, K // 16)
        assert np.array_equal(codes, xq), label + ": workspace codes"
        assert np.array_equal(sf, sf_rowmajor_to_mma(xs)), label + ": workspace scales"
        if not given:
            g_ws = float(wsp[0:4].view(torch.float32).item())
            assert _f32_bits(g_ws) == _f32_bits(gx), label + ": g_x"
    y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, ws, gwo, np.arange(M))
    check_gemm_tolerance(bf16_bits(y), y_ref, label)


def _draw_epi(n_cases, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_cases):
        M = int([rng.integers(1, 65), rng.integers(65, 129), rng.integers(129, 700)][i % 3])
        N = int(256 * rng.integers(1, 5))
        K = int(256 * rng.integers(1, 6))
        out.append((M, N, K, bool(rng.integers(0, 2)), 2000 + i))
    return out


@pytest.mark.parametrize("M,N,K,bias,seed", _draw_epi(15, 7051))
def test_random_dynamic_requant_matches_oracle(nv, oracle_mod, M, N, K, bias, seed):
    x = workloads.make_x("outlier", M, K, seed=seed)
    w = workloads.make_w(N, K, seed=seed + 1)
    b = workloads.make_bias(N, seed=seed + 2) if bias else torch.zeros(N, dtype=torch.bfloat16)
    xb, wb, bb = bf16_bits(x), bf16_bits(w), bf16_bits(b)
    gx, gwo = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gwo)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(
        x.cuda(), Wq, Ws, g_w, bias=b.cuda() if bias else None)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    label = "%dx%dx%d bias=%s" % (M, N, K, bias)
    y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, ws, gwo, np.arange(M),
                                 bias=bb if bias else None)
    check_gemm_tolerance(bf16_bits(Y), y_ref, label)
    y_bits = bf16_bits(Y)
    g_expect = oracle_mod.global_scale(y_bits)
    assert _f32_bits(g_y.item()) == _f32_bits(g_expect), label + ": g_y"
    q_ref, s_ref = oracle_mod.quantize(y_bits, g_expect)
    assert np.array_equal(to_np_u8(Yq), q_ref), label + ": codes"
    assert np.array_equal(to_np_u8(Ys), sf_rowmajor_to_mma(s_ref)), label + ": scales"


def _draw_lora(n_cases, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_cases):
        M = int(rng.integers(129, 900))     # the LoRA entry runs the CTA-pair kernel
        N = int(256 * rng.integers(1, 5))
        K = int(256 * rng.integers(1, 8))
        r = int([16, 32, 48, 64][rng.integers(0, 4)])
        out.append((M, N, K, r, [1.0, 0.5, 16.0][i % 3], KINDS[i % 3], 500 + i))
    return out


@pytest.mark.parametrize("M,N,K,r,scale,kind,seed", _draw_lora(12, 9))
def test_random_lora_matches_oracle(nv, oracle_mod, M, N, K, r, scale, kind, seed):
    import test_gpu_lora
    test_gpu_lora._run(nv, oracle_mod, M, N, K, r, scale, seed=seed, kind=kind)


def _draw_grouped(n_cases, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_cases):
        M = int([rng.integers(1, 9), rng.integers(9, 129), rng.integers(129, 700)][i % 3])
        ns = tuple(int(256 * rng.integers(1, 4)) for _ in range(int(rng.integers(1, 5))))
        out.append((M, ns, int(256 * rng.integers(1, 6)), int(rng.integers(0, 2)), 900 + i))
    return out


@pytest.mark.parametrize("M,ns,K,mode,seed", _draw_grouped(12, 10))
def test_random_grouped_matches_separate_and_oracle(nv, oracle_mod, M, ns, K, mode, seed):
    import test_gpu_grouped
    test_gpu_grouped._check(nv, oracle_mod, M, ns, K, mode, seed=seed)


def _draw_quantize(n_cases, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n_cases):
        rows = int(rng.integers(1, 700))
        layout = int(rng.integers(0, 2))
        K = int((64 if layout else 16) * rng.integers(1, 40))
        out.append((rows, K, int(i % 3), layout, float([1.0, 0.5, 4.0][i % 3]), KINDS[i % 3],
                    3000 + i))
    return out


@pytest.mark.parametrize("rows,K,rule,layout,g_factor,kind,seed", _draw_quantize(15, 11))
def test_random_quantize_matches_oracle(nv, oracle_mod, rows, K, rule, layout, g_factor, kind,
                                        seed):
    """The standalone quantizer under every scale rule, both layouts, ragged
    rows and K (any multiple of 16, of 64 in the tile layout), and a given
    scale off the tensor's own by the drawn factor."""
    x = workloads.make_x(kind, rows, K, seed=seed)
    xb = bf16_bits(x)
    g = float(np.float32(oracle_mod.global_scale(xb) * g_factor))
    q_ref, s_ref = oracle_mod.quantize(xb, g, rule)
    q, s = nv.nvfp4_quantize(x.cuda(), torch.tensor([g], dtype=torch.float32, device="cuda"),
                             layout, rule=rule)
    torch.cuda.synchronize()
    assert nv.nvfp4_device_error() == 0
    label = "%dx%d rule=%d layout=%d" % (rows, K, rule, layout)
    assert np.array_equal(to_np_u8(q), q_ref), label + ": codes"
    want = s_ref if layout == 0 else sf_rowmajor_to_mma(s_ref)
    assert np.array_equal(to_np_u8(s).reshape(want.shape), want), label + ": scales"
