"""GPU parity of the tcgen05 block-scaled FP4 GEMM and the NVFP4 linear layer.

The oracle quantizes X and W itself (bit-exactness of the GPU quantizer is
checked on the way) and computes Y in FP64 from the dequantized operands,
rounded once to bfloat16. GPU Y must be within
|y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m,:]||_2 elementwise.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, check_gemm_tolerance, sf_rowmajor_to_mma, tile_covering_rows, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    nv.nvfp4_device_error(clear=True)
    return nv


def _oracle_operands(oracle_mod, x, w):
    xb, wb = bf16_bits(x), bf16_bits(w)
    gx, gw = oracle_mod.global_scale(xb), oracle_mod.global_scale(wb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq, ws = oracle_mod.quantize(wb, gw)
    return (xq, xs, gx), (wq, ws, gw)


def _run_linear(nv, x, w, mode, given_gx=None):
    xd, wd = x.cuda(), w.cuda()
    Wq, Ws, gw = nv.nvfp4_quantize_weight(wd, nv.SF_MMA_128x4)
    gx = None if given_gx is None else torch.tensor([given_gx], dtype=torch.float32,
                                                    device="cuda")
    y = nv.nvfp4_linear(xd, Wq, Ws, gw, g_x=gx, mode=mode)
    return y, (Wq, Ws, gw)


GEMM_SHAPES = [  # (M, N, K): ragged M/N tails, several K tiles
    (64, 128, 256), (1, 8, 256), (7, 40, 512), (128, 256, 256), (200, 300, 1280),
    (300, 520, 768), (129, 257, 512), (513, 1000, 1024),
]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_linear_matches_oracle(nv, oracle_mod, M, N, K):
    x = workloads.make_x("outlier", M, K, seed=M * 31 + K)
    w = workloads.make_w(N, K, seed=N * 17 + K)
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw)
    y, (Wq, Ws, g_w) = _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
    assert np.array_equal(to_np_u8(Wq), wq)
    assert np.array_equal(to_np_u8(Ws), sf_rowmajor_to_mma(ws))
    max_rel, floor_only = check_gemm_tolerance(bf16_bits(y), y_ref, "linear %dx%dx%d" % (M, N, K))
    print("linear %dx%dx%d max_rel=%.3g floor_only=%d" % (M, N, K, max_rel, floor_only))
    assert nv.nvfp4_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(64, 128, 256), (200, 300, 1280), (513, 1000, 1024)])
def test_gemm_on_oracle_operands(nv, oracle_mod, M, N, K):
    """nvfp4_gemm fed the oracle's own quantized operands."""
    x = workloads.make_x("token_scaled", M, K, seed=M + 3 * K)
    w = workloads.make_w(N, K, seed=N + 5 * K)
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = nv.nvfp4_gemm(dev(xq), dev(sf_rowmajor_to_mma(xs)),
                      torch.tensor([gx], dtype=torch.float32, device="cuda"),
                      dev(wq), dev(sf_rowmajor_to_mma(ws)),
                      torch.tensor([gw], dtype=torch.float32, device="cuda"), K)
    check_gemm_tolerance(bf16_bits(y), y_ref, "gemm %dx%dx%d" % (M, N, K))


def test_linear_given_global_scale_and_fused_equal(nv, oracle_mod):
    M, N, K = 257, 384, 768
    x = workloads.make_x("outlier", M, K, seed=77)
    w = workloads.make_w(N, K, seed=78)
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, gw)
    y_dyn, _ = _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
    y_given, _ = _run_linear(nv, x, w, nv.LINEAR_UNFUSED, given_gx=gx)
    y_fused, _ = _run_linear(nv, x, w, nv.LINEAR_FUSED)
    assert torch.equal(y_dyn, y_given)
    assert torch.equal(y_dyn.view(torch.int16), y_fused.view(torch.int16))
    check_gemm_tolerance(bf16_bits(y_fused), y_ref, "fused")


def test_identity_weight_selects_columns(nv, oracle_mod):
    """W with a single code of 1.0 per row: Y[:, n] = dequantized X[:, n]."""
    M, K = 150, 256
    N = K
    x = workloads.make_x("normal", M, K, seed=12)
    xb = bf16_bits(x)
    gx = oracle_mod.global_scale(xb)
    xq, xs = oracle_mod.quantize(xb, gx)
    wq = np.zeros((N, K // 2), np.uint8)
    for n in range(N):
        wq[n, n // 2] = 0x02 << (4 * (n % 2))
    ws = np.full((N, K // 16), 0x38, np.uint8)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    y = nv.nvfp4_gemm(dev(xq), dev(sf_rowmajor_to_mma(xs)),
                      torch.tensor([gx], dtype=torch.float32, device="cuda"),
                      dev(wq), dev(sf_rowmajor_to_mma(ws)),
                      torch.tensor([1.0], dtype=torch.float32, device="cuda"), K)
    y_ref = oracle_mod.gemm(xq, xs, gx, wq, ws, 1.0)
    assert np.array_equal(bf16_bits(y), y_ref)  # one product per output: exact


def test_gemm_zero_sized_is_noop(nv):
    K = 256
    z = lambda *s: torch.zeros(*s, dtype=torch.uint8, device="cuda")
    g = torch.ones(1, dtype=torch.float32, device="cuda")
    y = nv.nvfp4_gemm(z(0, K // 2), z(0, K // 16), g, z(16, K // 2), z(128, K // 16), g, K)
    assert y.shape == (0, 16)
    torch.cuda.synchronize()


@pytest.mark.parametrize("M", [1, 3, 4, 5, 8, 9, 32])
@pytest.mark.parametrize("N,K", [(8, 256), (200, 768), (1000, 512), (300, 6144), (130, 6400)])
def test_fused_skinny_equals_unfused(nv, oracle_mod, M, N, K):
    """M <= 8, K <= 6144: the fused kernel quantizes X into shared memory;
    its output is bitwise the unfused one's (beyond those limits the fused
    mode runs the unfused sequence), and within tolerance of the oracle."""
    x = workloads.make_x("outlier", M, K, seed=M * 131 + N)
    w = workloads.make_w(N, K, seed=N * 7 + K)
    y_unf, _ = _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
    y_fus, _ = _run_linear(nv, x, w, nv.LINEAR_FUSED)
    assert torch.equal(y_unf.view(torch.int16), y_fus.view(torch.int16))
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    check_gemm_tolerance(bf16_bits(y_fus), oracle_mod.gemm(xq, xs, gx, wq, ws, gw), "fused")
    assert nv.nvfp4_device_error() == 0


def test_fused_skinny_strided_x_and_given_scale(nv, oracle_mod):
    M, N, K = 3, 384, 1024
    big = workloads.make_x("outlier", M, K + 256, seed=3)
    x = big[:, 128:128 + K]
    w = workloads.make_w(N, K, seed=4)
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x.contiguous(), w)
    Wq, Ws, g_w = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    xd = big.cuda()[:, 128:128 + K]
    g = torch.tensor([gx], dtype=torch.float32, device="cuda")
    y_f = nv.nvfp4_linear(xd, Wq, Ws, g_w, g_x=g, mode=nv.LINEAR_FUSED)
    y_u = nv.nvfp4_linear(xd, Wq, Ws, g_w, mode=nv.LINEAR_UNFUSED)
    assert torch.equal(y_f.view(torch.int16), y_u.view(torch.int16))
    check_gemm_tolerance(bf16_bits(y_f), oracle_mod.gemm(xq, xs, gx, wq, ws, gw), "strided")


def _full_size_case(nv, oracle_mod, name, M, Nn, step):
    w_ = workloads.WORKLOADS[name]
    x = workloads.make_x(w_.x_kind, M, w_.K, workloads.x_seed(w_))
    w = workloads.make_w(Nn, w_.K, workloads.w_seed(w_))
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    y, (Wq, Ws, _) = _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
    rows = np.arange(M) if M <= 64 else tile_covering_rows(M, step)
    y_ref = oracle_mod.gemm_rows(xq, xs, gx, wq, ws, gw, rows)
    y_rows = y.index_select(0, torch.from_numpy(rows).cuda())
    max_rel, floor_only = check_gemm_tolerance(bf16_bits(y_rows), y_ref, name)
    if M <= 32:  # the fused mode, in the configurations the benchmark times
        y_f, _ = _run_linear(nv, x, w, nv.LINEAR_FUSED)
        assert torch.equal(y_f.view(torch.int16), y.view(torch.int16))
    print("%s M=%d N=%d: max_rel=%.3g floor_only=%d" % (name, M, Nn, max_rel, floor_only))
    assert np.array_equal(to_np_u8(Wq), wq)
    assert nv.nvfp4_device_error() == 0


def test_full_size_prefill(nv, oracle_mod):
    _full_size_case(nv, oracle_mod, "prefill", 4096, 5120, 32)   # 128 rows, every 32-row band


@pytest.mark.parametrize("Nn", [9216, 12288])
def test_full_size_dit(nv, oracle_mod, Nn):
    _full_size_case(nv, oracle_mod, "dit", 4096, Nn, 32)


@pytest.mark.parametrize("M", [1, 8, 32])
def test_full_size_decode(nv, oracle_mod, M):
    _full_size_case(nv, oracle_mod, "decode", M, 27648, 32)      # every row


def test_full_size_square(nv, oracle_mod):
    _full_size_case(nv, oracle_mod, "square", 16384, 16384, 128)  # 128 rows, every CTA tile


def test_tile_covering_rows_reach_every_tile():
    for M, step in ((4096, 32), (16384, 128), (300, 32), (16384 + 77, 128)):
        rows = tile_covering_rows(M, step)
        assert rows.min() == 0 and rows.max() == M - 1
        assert set(np.unique(rows // 128)) == set(range((M + 127) // 128))


def test_bounded_wait_timeout_is_reported(nv, oracle_mod):
    """The producer is told to issue no loads: the consumers' bounded waits
    run out, the kernel records a timeout and returns; the context stays
    usable and the next GEMM is correct."""
    M, N, K = 128, 256, 512
    x = workloads.make_x("normal", M, K, seed=1)
    w = workloads.make_w(N, K, seed=2)
    nv.nvfp4_device_error(clear=True)
    try:
        nv.nvfp4_debug_set_fault_injection(1, 20000)  # 20 ms waits
        _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
        assert nv.nvfp4_device_error(clear=True) == 6  # NVFP4_ERR_TIMEOUT
    finally:
        nv.nvfp4_debug_set_fault_injection(0, 0)
    (xq, xs, gx), (wq, ws, gw) = _oracle_operands(oracle_mod, x, w)
    y, _ = _run_linear(nv, x, w, nv.LINEAR_UNFUSED)
    check_gemm_tolerance(bf16_bits(y), oracle_mod.gemm(xq, xs, gx, wq, ws, gw), "after timeout")
    assert nv.nvfp4_device_error() == 0
