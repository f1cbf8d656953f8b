"""GPU parity of the global scale and the NVFP4 quantizer against the oracle.

Packed codes and scales must match the oracle bit for bit; the tile-layout
scales must be exactly the row-major ones permuted by the layout's
definition.
"""
import numpy as np
import pytest
import torch

from helpers import bf16_bits, sf_rowmajor_to_mma, to_np_u8
from nvfp4_block_scaled_28_b300 import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import nvfp4_block_scaled_28_b300 as nv
    nv.load_library()
    assert torch.cuda.is_available(), "CUDA device required"
    return nv


def _f32_bits(x: float) -> int:
    return int(np.array([x], np.float32).view(np.uint32)[0])


def _quant_both(nv, oracle_mod, x: torch.Tensor, g_host=None):
    """Quantize x (CPU bf16) on the GPU and in the oracle; return both."""
    bits = bf16_bits(x)
    xd = x.cuda()
    if g_host is None:
        g_host = oracle_mod.global_scale(bits)
        g = nv.nvfp4_global_scale(xd)
        assert _f32_bits(float(g.item())) == _f32_bits(g_host)
    else:
        g = torch.tensor([g_host], dtype=torch.float32, device="cuda")
    q, sf = nv.nvfp4_quantize(xd, g, nv.SF_ROW_MAJOR)
    qo, so = oracle_mod.quantize(bits, g_host)
    return (to_np_u8(q), to_np_u8(sf)), (qo, so), (xd, g)


SHAPES = [(1, 16), (3, 48), (17, 256), (64, 256), (129, 64), (300, 5120), (1000, 160),
          (257, 1024)]


@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("kind", ["normal", "outlier", "token_scaled"])
def test_quantize_bit_exact(nv, oracle_mod, rows, cols, kind):
    x = workloads.make_x(kind, rows, cols, seed=rows * 7919 + cols)
    (q, sf), (qo, so), (xd, g) = _quant_both(nv, oracle_mod, x)
    assert np.array_equal(q, qo), "codes differ at %s" % (np.argwhere(q != qo)[:5],)
    assert np.array_equal(sf, so), "scales differ at %s" % (np.argwhere(sf != so)[:5],)
    if cols % 64 == 0:
        q2, sf2 = nv.nvfp4_quantize(xd, g, nv.SF_MMA_128x4)
        assert np.array_equal(to_np_u8(q2), qo)
        assert np.array_equal(to_np_u8(sf2), sf_rowmajor_to_mma(so))
        perm = nv.nvfp4_sf_to_mma_layout(torch.from_numpy(so).cuda(), rows, cols)
        assert np.array_equal(to_np_u8(perm), sf_rowmajor_to_mma(so))


def _special_rows():
    """Blocks built to sit on rounding boundaries: for each E4M3 scale s,
    the block max 6 s, every grid value and midpoint times s, and the
    bfloat16 neighbours of each midpoint, with mixed signs; plus zeros,
    -0.0 and tiny negatives."""
    grid = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    probes = []
    for a, b in zip(grid, grid[1:]):
        probes += [a, (a + b) / 2]
    probes.append(6.0)
    rows = []
    for S in range(1, 0x7F):
        s = float(torch.tensor([S], dtype=torch.uint8).view(torch.float8_e4m3fn).float())
        if 6 * s > 3e38:
            continue
        vals = [6 * s] + [p * s for p in probes]
        for p in probes[1:-1]:
            v = torch.tensor([p * s], dtype=torch.float32).to(torch.bfloat16)
            b = int(v.view(torch.int16))
            for d in (-1, 1):
                vals.append(float(torch.tensor([b + d], dtype=torch.int16).view(torch.bfloat16).float()))
        vals = (vals + [0.0] * 64)[:64]
        signs = [1.0 if i % 3 else -1.0 for i in range(64)]
        rows.append([v * sg for v, sg in zip(vals, signs)])
    z = [0.0] * 64
    z[3] = -0.0
    z[20] = -1e-30
    z[40] = 1.0
    z[41] = -1e-3
    rows.append(z)
    return torch.tensor(rows, dtype=torch.float32).to(torch.bfloat16)


def test_quantize_rounding_boundaries(nv, oracle_mod):
    x = _special_rows()
    bits = bf16_bits(x)
    bits[-1, 3] = 0x8000  # exact -0.0
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    for g in (1.0, 0.37, 3.0):  # g = 1 puts every block exactly on its scale
        (q, sf), (qo, so), _ = _quant_both(nv, oracle_mod, x, g_host=g)
        assert np.array_equal(sf, so)
        assert np.array_equal(q, qo), np.argwhere(q != qo)[:5]


def test_quantize_saturation_with_small_given_scale(nv, oracle_mod):
    x = workloads.make_x("outlier", 64, 512, seed=5)
    g_true = oracle_mod.global_scale(bf16_bits(x))
    for g in (g_true / 8, g_true / 1000):
        (q, sf), (qo, so), _ = _quant_both(nv, oracle_mod, x, g_host=g)
        assert np.array_equal(sf, so) and np.array_equal(q, qo)
        assert np.any(so == 0x7E)  # some block scales saturate at 448


def test_quantize_all_zero_and_strided(nv, oracle_mod):
    x = torch.zeros(5, 128, dtype=torch.bfloat16)
    (q, sf), (qo, so), _ = _quant_both(nv, oracle_mod, x)
    assert np.array_equal(q, qo) and np.array_equal(sf, so) and not sf.any()
    big = workloads.make_x("normal", 40, 384, seed=9)
    xs = big[:, 64:320]  # row stride 384 > cols 256
    bits = bf16_bits(xs)
    g_host = oracle_mod.global_scale(bits)
    xd = big.cuda()[:, 64:320]
    g = nv.nvfp4_global_scale(xd)
    assert _f32_bits(float(g.item())) == _f32_bits(g_host)
    q, sf = nv.nvfp4_quantize(xd, g)
    qo, so = oracle_mod.quantize(bits, g_host)
    assert np.array_equal(to_np_u8(q), qo) and np.array_equal(to_np_u8(sf), so)


def test_quantize_empty(nv):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = nv.nvfp4_global_scale(x)
    assert float(g.item()) == 1.0
    q, sf = nv.nvfp4_quantize(x, g)
    assert q.shape == (0, 32) and sf.shape == (0, 4)
    torch.cuda.synchronize()


def test_quantize_weight_matches_oracle(nv, oracle_mod):
    w = workloads.make_w(300, 512, seed=3)
    bits = bf16_bits(w)
    Wq, Ws, gw = nv.nvfp4_quantize_weight(w.cuda(), nv.SF_MMA_128x4)
    g_host = oracle_mod.global_scale(bits)
    qo, so = oracle_mod.quantize(bits, g_host)
    assert _f32_bits(float(gw.item())) == _f32_bits(g_host)
    assert np.array_equal(to_np_u8(Wq), qo)
    assert np.array_equal(to_np_u8(Ws), sf_rowmajor_to_mma(so))


def test_quantize_full_size_square_sampled_rows(nv, oracle_mod):
    """16384 x 16384 activation quantize (the standalone quantize workload) in
    the launch configuration the benchmark uses; the oracle checks 192
    sampled rows bit for bit (rows are independent given g)."""
    w = workloads.WORKLOADS["square"]
    x = workloads.make_x(w.x_kind, w.M[0], w.K, workloads.x_seed(w))
    bits_all = bf16_bits(x)
    g_host = oracle_mod.global_scale(bits_all)
    xd = x.cuda()
    g = nv.nvfp4_global_scale(xd)
    assert _f32_bits(float(g.item())) == _f32_bits(g_host)
    q, sf = nv.nvfp4_quantize(xd, g, nv.SF_ROW_MAJOR)
    rows = np.sort(np.random.default_rng(0).choice(w.M[0], 192, replace=False))
    rows = np.concatenate([[0, w.M[0] - 1], rows])
    qo, so = oracle_mod.quantize(bits_all[rows], g_host)
    ridx = torch.from_numpy(rows).cuda()
    assert np.array_equal(to_np_u8(q.index_select(0, ridx)), qo)
    assert np.array_equal(to_np_u8(sf.index_select(0, ridx)), so)
    del xd, q, sf
    torch.cuda.empty_cache()
