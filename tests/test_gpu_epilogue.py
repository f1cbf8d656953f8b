"""GPU parity of the linear layer's fused epilogue: bias add and the NVFP4
re-quantization of the bfloat16 output for the next layer.

Y is checked against the oracle's FP64 contraction plus bias, rounded once to
bfloat16, within |y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2. The
re-quantized codes and scales must equal, bit for bit, the oracle's
quantization of the GPU's own Y with the same g_y (the rounding decisions are
taken on the same bfloat16 values on both sides).
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, sf_rowmajor_to_mma, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _case(nv, oracle_mod, M, N, K, seed, kind="outlier"):
    x = workloads.make_x(kind, M, K, seed=seed)
    w = workloads.make_w(N, K, seed=seed + 1)
    b = workloads.make_bias(N, seed=seed + 2)
    xb, wb, bb = bf16_bits(x), bf16_bits(w), bf16_bits(b)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gw)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    assert np.array_equal(to_np_u8(Wq), wq)
    return dict(x=x, b=b, bb=bb, ops=(xq, xs, gx, wq, ws, gw), W=(Wq, Ws, g_w))


def _gy(value) -> torch.Tensor:
    return torch.tensor([np.float32(value)], dtype=torch.float32, device="cuda")


def _check_requant(oracle_mod, y_bits, g_y, Yq, Ys, label):
    """GPU (Yq, Ys) == the oracle's quantization of the GPU's Y under g_y."""
    q_ref, s_ref = oracle_mod.quantize(y_bits, float(np.float32(g_y)))
    q = to_np_u8(Yq)
    assert np.array_equal(q, q_ref), "%s: codes differ at %s" % (
        label, np.argwhere(q != q_ref)[:4].tolist())
    s = to_np_u8(Ys)
    s_mma = sf_rowmajor_to_mma(s_ref)
    assert s.shape == s_mma.shape
    assert np.array_equal(s, s_mma), "%s: %d scale bytes differ" % (label, int((s != s_mma).sum()))


EPI_SHAPES = [  # (M, N, K): M > 128; N % 256 == 0; ragged M, several N tiles
    (129, 256, 256), (256, 512, 512), (300, 768, 768), (513, 1024, 1280),
]


@pytest.mark.parametrize("M,N,K", EPI_SHAPES)
def test_bias_and_requant_match_oracle(nv, oracle_mod, M, N, K):
    c = _case(nv, oracle_mod, M, N, K, seed=M * 7 + N + K)
    xq, xs, gx, wq, ws, gw = c["ops"]
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"])
    g_y = oracle_mod.global_scale(y_ref)  # calibrated on the reference output
    Wq, Ws, g_w = c["W"]
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                             bias=c["b"].cuda())
    y_bits = bf16_bits(Y)
    max_rel, floor_only = check_gemm_tolerance(y_bits, y_ref, "bias %dx%dx%d" % (M, N, K))
    _check_requant(oracle_mod, y_bits, g_y, Yq, Ys, "requant %dx%dx%d" % (M, N, K))
    print("bias+requant %dx%dx%d max_rel=%.3g floor_only=%d" % (M, N, K, max_rel, floor_only))
    assert nv.nvfp4_device_error() == 0


def test_requant_only_equals_with_y_and_saturates(nv, oracle_mod):
    """Skipping the bfloat16 store changes nothing else; a g_y calibrated too
    small (amax / (6 * 448) of a quarter of the output) saturates scales at
    448 and codes at 6 on both sides alike."""
    M, N, K = 384, 512, 1024
    c = _case(nv, oracle_mod, M, N, K, seed=99, kind="token_scaled")
    xq, xs, gx, wq, ws, gw = c["ops"]
    Wq, Ws, g_w = c["W"]
    xd, bd = c["x"].cuda(), c["b"].cuda()
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"])
    g_small = oracle_mod.global_scale(y_ref) / 4.0
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(xd, Wq, Ws, g_w, _gy(g_small), bias=bd)
    _check_requant(oracle_mod, bf16_bits(Y), g_small, Yq, Ys, "saturating")
    assert (to_np_u8(Ys) == 0x7E).any()  # 448 in E4M3
    Y2, Yq2, Ys2 = nv.nvfp4_linear_bias_requant(xd, Wq, Ws, g_w, _gy(g_small), bias=bd,
                                                store_y=False)
    assert Y2 is None
    assert torch.equal(Yq2, Yq) and torch.equal(Ys2, Ys)
    assert nv.nvfp4_device_error() == 0


def test_no_bias_no_requant_equals_linear(nv, oracle_mod):
    """With neither step the epilogue kernel writes what nvfp4_linear does."""
    M, N, K = 640, 768, 768
    c = _case(nv, oracle_mod, M, N, K, seed=5)
    Wq, Ws, g_w = c["W"]
    xd = c["x"].cuda()
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(xd, Wq, Ws, g_w, None)
    assert Yq is None and Ys is None
    Y_lin = nv.nvfp4_linear(xd, Wq, Ws, g_w)
    assert torch.equal(Y.view(torch.int16), Y_lin.view(torch.int16))
    # bias only, given g_x: Y matches the oracle with the bias
    xq, xs, gx, wq, ws, gw = c["ops"]
    Yb, _, _ = nv.nvfp4_linear_bias_requant(xd, Wq, Ws, g_w, None, bias=c["b"].cuda(),
                                            g_x=_gy(gx))
    check_gemm_tolerance(bf16_bits(Yb), oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"]),
                         "bias only")
    assert nv.nvfp4_device_error() == 0


def test_chained_layers(nv, oracle_mod):
    """The re-quantized output feeds the next layer's GEMM directly: layer 2
    on (Yq, Ys, g_y) matches the oracle's layer 2 on the oracle's own
    quantization of layer 1's output."""
    M, N1, K, N2 = 257, 1024, 512, 384
    c = _case(nv, oracle_mod, M, N1, K, seed=11)
    Wq, Ws, g_w = c["W"]
    xq, xs, gx, wq, ws, gw = c["ops"]
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"])
    g_y = oracle_mod.global_scale(y_ref)
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                             bias=c["b"].cuda())
    w2 = workloads.make_w(N2, N1, seed=12)
    w2b = bf16_bits(w2)
    gw2 = oracle_mod.global_scale(w2b)
    w2q, w2s = oracle_mod.quantize(w2b, gw2)
    W2q, W2s, g_w2 = nv.nvfp4_quantize_weight(w2.cuda(), nv.SF_MMA_128x4)
    y2 = nv.nvfp4_gemm(Yq, Ys, _gy(g_y), W2q, W2s, g_w2, N1)
    yq_ref, ys_ref = oracle_mod.quantize(bf16_bits(Y), float(np.float32(g_y)))
    y2_ref = oracle_mod.gemm(yq_ref, ys_ref, g_y, w2q, w2s, gw2)
    check_gemm_tolerance(bf16_bits(y2), y2_ref, "chained")
    assert nv.nvfp4_device_error() == 0


def test_full_size_prefill_bias_requant(nv, oracle_mod):
    """The 4096 x 5120 x 5120 layer with both epilogue steps: sampled rows of
    Y against the oracle, every code and scale against the oracle's
    quantization of the GPU's Y."""
    w_ = workloads.WORKLOADS["prefill"]
    M, N, K = 4096, 5120, w_.K
    x = workloads.make_x(w_.x_kind, M, K, workloads.x_seed(w_))
    w = workloads.make_w(N, K, workloads.w_seed(w_))
    b = workloads.make_bias(N, seed=77)
    xb, wb, bb = bf16_bits(x), bf16_bits(w), bf16_bits(b)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gw)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    rows = np.unique(np.concatenate([[0, M - 1],
                                     np.random.default_rng(3).choice(M, 24, replace=False)]))
    y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, ws, gw, rows, bias=bb)
    g_y = oracle_mod.global_scale(y_ref)
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(x.cuda(), Wq, Ws, g_w, _gy(g_y), bias=b.cuda())
    y_bits = bf16_bits(Y)
    check_gemm_tolerance(y_bits[rows], y_ref, "prefill bias")
    _check_requant(oracle_mod, y_bits, g_y, Yq, Ys, "prefill requant")
    assert nv.nvfp4_device_error() == 0


def _f32_bits(v) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


@pytest.mark.parametrize("M,N,K", EPI_SHAPES)
def test_dynamic_requant_matches_oracle(nv, oracle_mod, M, N, K):
    """The output's global scale computed from the output (the epilogue's
    atomic amax): g_y is the oracle's global scale of the GPU's Y, bit for
    bit, and the codes and scales are the oracle's quantization under it."""
    c = _case(nv, oracle_mod, M, N, K, seed=M * 5 + N + 3 * K)
    xq, xs, gx, wq, ws, gw = c["ops"]
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"])
    Wq, Ws, g_w = c["W"]
    g_y = torch.full((1,), 123.0, dtype=torch.float32, device="cuda")  # stale value
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(c["x"].cuda(), Wq, Ws, g_w,
                                                          bias=c["b"].cuda(), g_y=g_y)
    torch.cuda.synchronize()
    y_bits = bf16_bits(Y)
    check_gemm_tolerance(y_bits, y_ref, "dynamic bias %dx%dx%d" % (M, N, K))
    g_expect = oracle_mod.global_scale(y_bits)
    assert _f32_bits(g_y.item()) == _f32_bits(g_expect), "g_y %r vs %r" % (g_y.item(), g_expect)
    _check_requant(oracle_mod, y_bits, g_expect, Yq, Ys, "dynamic requant %dx%dx%d" % (M, N, K))
    assert nv.nvfp4_device_error() == 0


def test_dynamic_requant_equals_unfused_sequence(nv):
    """Bytes equal nvfp4_linear_bias_requant (Y only) + nvfp4_global_scale(Y)
    + nvfp4_quantize(Y), on the prefill shape, twice in a row on one
    workspace (the amax cell is zeroed by every call)."""
    M, N, K = 4096, 5120, 5120
    w = workloads.make_w(N, K, seed=31)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    b = workloads.make_bias(N, seed=32).cuda()
    ws = torch.empty(nv.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    for i, kind in enumerate(["outlier", "token_scaled"]):
        x = workloads.make_x(kind, M, K, seed=40 + i).cuda()
        Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(x, Wq, Ws, g_w, bias=b, workspace=ws)
        Y2, _, _ = nv.nvfp4_linear_bias_requant(x, Wq, Ws, g_w, None, bias=b)
        g2 = nv.nvfp4_global_scale(Y2)
        q2, s2 = nv.nvfp4_quantize(Y2, g2, nv.SF_MMA_128x4)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16)), "call %d: Y" % i
        assert torch.equal(g_y.view(torch.int32), g2.view(torch.int32)), "call %d: g_y" % i
        assert torch.equal(Yq, q2), "call %d: codes" % i
        assert torch.equal(Ys, s2), "call %d: scales" % i
    assert nv.nvfp4_device_error() == 0


def test_dynamic_requant_ignores_padding_rows(nv, oracle_mod):
    """Rows past M of the last tile hold the bias alone and must not enter
    the amax: X >= 0, weight row 0 <= 0 and bias[0] = +1000 make every real
    y[:, 0] smaller than 1000 while a padding row would be exactly 1000."""
    M, N, K = 129, 256, 256
    x = workloads.make_x("normal", M, K, seed=5).abs()
    w = workloads.make_w(N, K, seed=6)
    w[0] = -w[0].abs() - 0.1
    b = torch.zeros(N, dtype=torch.bfloat16)
    b[0] = 1000.0
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(x.cuda(), Wq, Ws, g_w, bias=b.cuda())
    torch.cuda.synchronize()
    y_bits = bf16_bits(Y)
    assert float(Y[:, 0].float().max()) < 1000.0
    g_expect = oracle_mod.global_scale(y_bits)
    assert _f32_bits(g_y.item()) == _f32_bits(g_expect), "g_y %r vs %r" % (g_y.item(), g_expect)
    _check_requant(oracle_mod, y_bits, g_expect, Yq, Ys, "padding rows")
    assert nv.nvfp4_device_error() == 0


def test_dynamic_requant_empty_activation(nv, oracle_mod):
    """M = 0: nothing to multiply; g_y is the global scale of an empty
    tensor (1, as the oracle and nvfp4_global_scale give), written over a
    stale value."""
    N, K = 256, 512
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(workloads.make_w(N, K, seed=7).cuda(),
                                           nv.SF_MMA_128x4)
    x = torch.empty((0, K), dtype=torch.bfloat16, device="cuda")
    g_y = _gy(123.0)
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(x, Wq, Ws, g_w, g_y=g_y)
    torch.cuda.synchronize()
    assert Y.shape == (0, N) and Yq.shape == (0, N // 2) and Ys.numel() == 0
    g_empty = oracle_mod.global_scale(np.zeros((0, K), dtype=np.uint16))
    assert _f32_bits(g_y.item()) == _f32_bits(g_empty) == _f32_bits(1.0)
    assert _f32_bits(nv.nvfp4_global_scale(x).item()) == _f32_bits(1.0)
    assert nv.nvfp4_device_error() == 0


# Decode rows: up to 64 the decode kernel's epilogue (a 16-element block of Y
# spans 16 lanes), 65 .. 128 the CTA-pair kernel; (4, 19200, 1024) has a
# partial last round whose tiles are split by K across a cluster
DECODE_EPI_SHAPES = [(1, 512, 512), (8, 768, 1024), (32, 1024, 512), (64, 512, 768),
                     (100, 512, 512), (4, 19200, 1024)]


@pytest.mark.parametrize("M,N,K", DECODE_EPI_SHAPES)
def test_decode_bias_and_requant_match_oracle(nv, oracle_mod, M, N, K):
    c = _case(nv, oracle_mod, M, N, K, seed=M * 11 + N + K)
    xq, xs, gx, wq, ws, gw = c["ops"]
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"])
    g_y = oracle_mod.global_scale(y_ref)
    Wq, Ws, g_w = c["W"]
    Ys = torch.full(nv.sf_shape(M, N, nv.SF_MMA_128x4), 0xA5, dtype=torch.uint8, device="cuda")
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                             bias=c["b"].cuda(), Ys=Ys)
    y_bits = bf16_bits(Y)
    check_gemm_tolerance(y_bits, y_ref, "decode bias %dx%dx%d" % (M, N, K))
    _check_requant(oracle_mod, y_bits, g_y, Yq, Ys, "decode requant %dx%dx%d" % (M, N, K))
    # Y alone (no re-quantization) and the codes alone (no Y) agree with it
    Y2, _, _ = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, None, bias=c["b"].cuda())
    assert torch.equal(Y2.view(torch.int16), Y.view(torch.int16))
    _, Yq3, Ys3 = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                               bias=c["b"].cuda(), store_y=False)
    assert torch.equal(Yq3, Yq) and torch.equal(Ys3, Ys)
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,N,K", DECODE_EPI_SHAPES)
def test_decode_dynamic_requant_matches_oracle(nv, oracle_mod, M, N, K):
    c = _case(nv, oracle_mod, M, N, K, seed=M * 13 + N + 2 * K)
    Wq, Ws, g_w = c["W"]
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(c["x"].cuda(), Wq, Ws, g_w,
                                                          bias=c["b"].cuda())
    torch.cuda.synchronize()
    y_bits = bf16_bits(Y)
    g_expect = oracle_mod.global_scale(y_bits)
    assert _f32_bits(g_y.item()) == _f32_bits(g_expect), "g_y %r vs %r" % (g_y.item(), g_expect)
    _check_requant(oracle_mod, y_bits, g_expect, Yq, Ys, "decode dynamic %dx%dx%d" % (M, N, K))
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M", [1, 8, 32])
def test_decode_dynamic_requant_equals_unfused_sequence(nv, M):
    """The decode FFN-up shape (5120 -> 27648): all bytes equal the linear
    with the bias, then nvfp4_global_scale(Y) and nvfp4_quantize(Y)."""
    N, K = 27648, 5120
    w = workloads.make_w(N, K, seed=61)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    b = workloads.make_bias(N, seed=62).cuda()
    x = workloads.make_x("outlier", M, K, seed=63 + M).cuda()
    Y, g_y, Yq, Ys = nv.nvfp4_linear_bias_requant_dynamic(x, Wq, Ws, g_w, bias=b)
    Y2, _, _ = nv.nvfp4_linear_bias_requant(x, Wq, Ws, g_w, None, bias=b)
    g2 = nv.nvfp4_global_scale(Y2)
    q2, s2 = nv.nvfp4_quantize(Y2, g2, nv.SF_MMA_128x4)
    torch.cuda.synchronize()
    assert torch.equal(Y.view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(g_y.view(torch.int32), g2.view(torch.int32))
    assert torch.equal(Yq, q2) and torch.equal(Ys, s2)
    assert nv.nvfp4_device_error() == 0


def test_decode_requant_with_unaligned_y(nv, oracle_mod):
    """A Y whose rows are not 16-byte aligned (ldy = N + 1) keeps the
    re-quantization in the decode epilogue; the bytes are the same."""
    M, N, K = 8, 512, 512
    c = _case(nv, oracle_mod, M, N, K, seed=91)
    xq, xs, gx, wq, ws, gw = c["ops"]
    g_y = oracle_mod.global_scale(oracle_mod.gemm(xq, xs, gx, wq, ws, gw, bias=c["bb"]))
    Wq, Ws, g_w = c["W"]
    big = torch.zeros((M, N + 1), dtype=torch.bfloat16, device="cuda")
    Yv = big[:, :N]
    assert Yv.stride(0) == N + 1
    Y, Yq, Ys = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                             bias=c["b"].cuda(), Y=Yv)
    _check_requant(oracle_mod, bf16_bits(Y.contiguous()), g_y, Yq, Ys, "unaligned Y")
    Y2, Yq2, Ys2 = nv.nvfp4_linear_bias_requant(c["x"].cuda(), Wq, Ws, g_w, _gy(g_y),
                                                bias=c["b"].cuda())
    assert torch.equal(Y.contiguous().view(torch.int16), Y2.view(torch.int16))
    assert torch.equal(Yq, Yq2) and torch.equal(Ys, Ys2)
    assert nv.nvfp4_device_error() == 0
