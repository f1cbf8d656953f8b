"""The quantized activation that the linear layers write into their
workspace is the oracle's NVFP4 quantization of X, byte for byte.

nvfp4_linear (and its bias / re-quantization, grouped and LoRA variants)
leaves in the workspace the global scale it used (fp32 at byte 0), X's codes
(M x K/2 at byte 8448) and their tile-layout scales (after the codes,
256-byte aligned). Y alone cannot show that these bytes are right: a code of
-0 and +0, or errors whose products cancel, leave Y unchanged. Each kernel
that writes them is covered here: the cooperative dynamic quantizer
(prefill-sized X), the one-cluster quantizer (medium X), the small-X
quantizer (decode rows), the quantizer with a
given global scale, the LoRA pass, and, through a testing hook, the fused
decode kernel whose operand otherwise stays in shared memory. Every X
carries blocks of signed zeros and of tiny negatives that round to code 0x8.
"""
import ctypes

import numpy as np
import pytest
import torch

from helpers import bf16_bits, sf_rowmajor_to_mma, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu

HEADER = 8448


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _with_special_blocks(x: torch.Tensor) -> torch.Tensor:
    """Plant, in a few rows, a block of signed zeros, a block of tiny
    negatives next to a large value (they round to -0), and a block mixing
    -0.0 with ordinary values."""
    x = x.clone()
    M, K = x.shape
    rows = sorted({0, M // 2, M - 1})
    for i, r in enumerate(rows):
        kb = (5 * i + 1) % (K // 16)
        x[r, kb * 16:(kb + 1) * 16] = -0.0
        kb2 = (kb + 2) % (K // 16)
        blk = torch.full((16,), -1e-6, dtype=torch.float32)
        blk[3] = 40.0
        blk[7] = -0.0
        x[r, kb2 * 16:(kb2 + 1) * 16] = blk.to(torch.bfloat16)
        kb3 = (kb + 4) % (K // 16)
        x[r, kb3 * 16:kb3 * 16 + 8] = -0.0
    return x


def _split_ws(ws: torch.Tensor, M: int, K: int):
    codes = to_np_u8(ws[HEADER:HEADER + M * K // 2]).reshape(M, K // 2)
    sf_off = HEADER + (M * K // 2 + 255) // 256 * 256
    rows_pad = (M + 127) // 128 * 128
    sf = to_np_u8(ws[sf_off:sf_off + rows_pad * K // 16]).reshape(rows_pad, K // 16)
    gx = float(ws[0:4].view(torch.float32).item())
    return codes, sf, gx


def _f32_bits(v: float) -> int:
    return int(np.array([v], np.float32).view(np.uint32)[0])


def _expect(oracle_mod, x, g=None):
    xb = bf16_bits(x)
    if g is None:
        g = oracle_mod.global_scale(xb)
    q, s = oracle_mod.quantize(xb, g)
    return q, sf_rowmajor_to_mma(s), g


def _check(ws, M, K, q_ref, sf_ref, g_ref, check_g=True, label=""):
    codes, sf, gx = _split_ws(ws, M, K)
    if check_g:
        assert _f32_bits(gx) == _f32_bits(g_ref), "%s: g_x %r vs %r" % (label, gx, g_ref)
    bad = np.argwhere(codes != q_ref)
    assert bad.size == 0, "%s: codes differ at %s" % (label, bad[:5].tolist())
    bad = np.argwhere(sf != sf_ref)
    assert bad.size == 0, "%s: scales differ at %s" % (label, bad[:5].tolist())


def _weights(nv, N, K, seed):
    return nv.nvfp4_quantize_weight(workloads.make_w(N, K, seed=seed).cuda(), nv.SF_MMA_128x4)


# (M, K): the cooperative dynamic quantizer for X above 512K elements
# (prefill size included), the one-cluster quantizer from 64K to 512K
# elements (both ends), the small-X quantizer at or below 64K (decode rows)
@pytest.mark.parametrize("M,K,kind", [
    (4096, 5120, "outlier"), (300, 768, "token_scaled"), (1000, 1024, "normal"),
    (32, 5120, "outlier"), (8, 5120, "outlier"), (1, 5120, "outlier"), (64, 1024, "normal"),
    (512, 1024, "outlier"), (513, 1024, "token_scaled"), (65, 1024, "outlier"),
])
def test_linear_workspace_dynamic_scale(nv, oracle_mod, M, K, kind):
    N = 256
    x = _with_special_blocks(workloads.make_x(kind, M, K, seed=M + K))
    Wq, Ws, gw = _weights(nv, N, K, seed=3)
    ws = torch.zeros(nv.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, workspace=ws)
    torch.cuda.synchronize()
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="linear %dx%d" % (M, K))
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,K", [(4096, 5120), (300, 768), (5, 512)])
def test_linear_workspace_given_scale(nv, oracle_mod, M, K):
    N = 256
    x = _with_special_blocks(workloads.make_x("outlier", M, K, seed=2 * M + K))
    Wq, Ws, gw = _weights(nv, N, K, seed=4)
    g_host = 0.75 * oracle_mod.global_scale(bf16_bits(x))  # a smaller scale: saturation
    g = torch.tensor([g_host], dtype=torch.float32, device="cuda")
    ws = torch.zeros(nv.linear_workspace_bytes(M, N, K), dtype=torch.uint8, device="cuda")
    nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, g_x=g, workspace=ws)
    torch.cuda.synchronize()
    q_ref, sf_ref, _ = _expect(oracle_mod, x, g=np.float32(g_host).item())
    _check(ws, M, K, q_ref, sf_ref, None, check_g=False, label="given g %dx%d" % (M, K))


def test_workspace_is_rewritten_over_stale_contents(nv, oracle_mod):
    """The padding rows of the scales and the global scale are written on
    every call, whatever the workspace held before."""
    M, K, N = 200, 1024, 256
    x = _with_special_blocks(workloads.make_x("normal", M, K, seed=9))
    Wq, Ws, gw = _weights(nv, N, K, seed=5)
    ws = torch.full((nv.linear_workspace_bytes(M, N, K),), 0xA5, dtype=torch.uint8,
                    device="cuda")
    nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, workspace=ws)
    torch.cuda.synchronize()
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="stale")


def test_bias_requant_and_grouped_workspace(nv, oracle_mod):
    M, K = 384, 1024
    x = _with_special_blocks(workloads.make_x("token_scaled", M, K, seed=21))
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    xd = x.cuda()
    # bias + re-quantization epilogue
    Wq, Ws, gw = _weights(nv, 512, K, seed=6)
    ws = torch.zeros(nv.linear_workspace_bytes(M, 512, K), dtype=torch.uint8, device="cuda")
    bias = workloads.make_bias(512, seed=1).cuda()
    gy = torch.tensor([0.01], dtype=torch.float32, device="cuda")
    nv.nvfp4_linear_bias_requant(xd, Wq, Ws, gw, bias=bias, g_y=gy, workspace=ws)
    torch.cuda.synchronize()
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="bias_requant")
    # grouped projections
    groups = [_weights(nv, 256, K, seed=30 + i) for i in range(3)]
    Wq3, Ws3, g3, gn3 = nv.pack_weight_groups(groups)
    ws = torch.zeros(nv.linear_workspace_bytes(M, sum(gn3), K), dtype=torch.uint8,
                     device="cuda")
    nv.nvfp4_linear_grouped(xd, Wq3, Ws3, g3, gn3, workspace=ws)
    torch.cuda.synchronize()
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="grouped")
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,K,r", [(4096, 5120, 32), (300, 768, 16)])
def test_lora_pass_workspace(nv, oracle_mod, M, K, r):
    """The LoRA pass quantizes X in the same sweep as the down projection."""
    N = 256
    x = _with_special_blocks(workloads.make_x("outlier", M, K, seed=M + r))
    Wq, Ws, gw = _weights(nv, N, K, seed=7)
    la, lb = workloads.make_lora(r, K, N, seed=8)
    ws = torch.zeros(int(nv.load_library().nvfp4_linear_lora_workspace_bytes(M, N, K, r)),
                     dtype=torch.uint8, device="cuda")
    nv.nvfp4_linear_lora(x.cuda(), Wq, Ws, gw, la.cuda(), lb.cuda(), lora_scale=1.0,
                         workspace=ws)
    torch.cuda.synchronize()
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="lora %dx%d r=%d" % (M, K, r))
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,K", [(1, 5120), (4, 5120), (3, 1280), (2, 6144), (8, 5120), (6, 6144)])
@pytest.mark.parametrize("given", [False, True])
def test_fused_decode_operand(nv, oracle_mod, M, K, given):
    """The fused decode kernel quantizes X in shared memory; the testing hook
    writes that operand out, and it must be the oracle's bytes."""
    lib = nv.load_library()
    N = 384
    x = _with_special_blocks(workloads.make_x("outlier", M, K, seed=40 + M))
    Wq, Ws, gw = _weights(nv, N, K, seed=10)
    g_ref = oracle_mod.global_scale(bf16_bits(x))
    g = torch.tensor([g_ref], dtype=torch.float32, device="cuda") if given else None
    ws = torch.full((nv.linear_workspace_bytes(M, N, K, nv.LINEAR_FUSED),), 0x5A,
                    dtype=torch.uint8, device="cuda")
    assert lib.nvfp4_debug_capture_fused_operand(1) == 0
    try:
        y_f = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, g_x=g, mode=nv.LINEAR_FUSED, workspace=ws)
        torch.cuda.synchronize()
    finally:
        assert lib.nvfp4_debug_capture_fused_operand(0) == 0
    q_ref, sf_ref, _ = _expect(oracle_mod, x, g=g_ref)
    _check(ws, M, K, q_ref, sf_ref, None, check_g=False, label="fused %dx%d" % (M, K))
    y_u = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, g_x=g, mode=nv.LINEAR_UNFUSED)
    assert torch.equal(y_f.view(torch.int16), y_u.view(torch.int16))
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,K", [(8, 1024), (100, 1024), (300, 3072)])
def test_strided_activation_workspace(nv, oracle_mod, M, K):
    """X as a strided view (row pitch K + 64): the small (8 x 1024), the
    one-cluster (100 x 1024) and the cooperative (300 x 3072) dynamic
    quantizers leave the oracle's bytes, and Y equals the contiguous call."""
    N = 256
    x = _with_special_blocks(workloads.make_x("outlier", M, K, seed=80 + M))
    big = torch.zeros((M, K + 64), dtype=torch.bfloat16)
    big[:, 32:32 + K] = x
    xd = big.cuda()[:, 32:32 + K]
    assert xd.stride(0) == K + 64
    Wq, Ws, gw = _weights(nv, N, K, seed=12)
    ws = torch.full((nv.linear_workspace_bytes(M, N, K),), 0x5A, dtype=torch.uint8,
                    device="cuda")
    y_s = nv.nvfp4_linear(xd, Wq, Ws, gw, workspace=ws)
    torch.cuda.synchronize()
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="strided %dx%d" % (M, K))
    y_c = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw)
    assert torch.equal(y_s.view(torch.int16), y_c.view(torch.int16))
    assert nv.nvfp4_device_error() == 0


def test_default_mode_keeps_the_workspace_contract(nv, oracle_mod):
    """With no mode given, a call without a workspace may take the fused
    decode kernel (the same Y bits), while a call with a workspace runs the
    unfused sequence and leaves X's quantized form in it."""
    M, N, K = 4, 1024, 2048
    x = _with_special_blocks(workloads.make_x("outlier", M, K, seed=41))
    Wq, Ws, gw = _weights(nv, N, K, 42)
    y_default = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw)
    y_fused = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, mode=nv.LINEAR_FUSED)
    ws = torch.full((nv.linear_workspace_bytes(M, N, K),), 0xA5, dtype=torch.uint8,
                    device="cuda")
    y_ws = nv.nvfp4_linear(x.cuda(), Wq, Ws, gw, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y_default.view(torch.int16), y_fused.view(torch.int16))
    assert torch.equal(y_default.view(torch.int16), y_ws.view(torch.int16))
    q_ref, sf_ref, g_ref = _expect(oracle_mod, x)
    _check(ws, M, K, q_ref, sf_ref, g_ref, label="default mode with a workspace")
    assert nv.nvfp4_device_error() == 0
