"""Host-side checks of the Python binding for the fused-epilogue, grouped
and LoRA entry points (no GPU): malformed operands are refused with a
ValueError before anything reaches the device, and stacking per-group
weights keeps the tensor-core scale layout."""
import numpy as np
import pytest
import torch

import nvfp4_block_scaled_28_b300 as nv
from helpers import sf_rowmajor_to_mma


def _codes(rows, K):
    return torch.zeros(rows, K // 2, dtype=torch.uint8)


def _scales_tile(rows, K, seed):
    rm = np.random.default_rng(seed).integers(0, 0x7F, (rows, K // 16), dtype=np.uint8)
    return rm, torch.from_numpy(sf_rowmajor_to_mma(rm).copy())


def test_stacked_group_scales_are_the_tile_layout_of_the_stacked_weight():
    K = 512
    rm0, t0 = _scales_tile(256, K, 1)
    rm1, t1 = _scales_tile(512, K, 2)
    g = torch.ones(1)
    Wq, Ws, gw, gn = nv.pack_weight_groups([(_codes(256, K), t0, g), (_codes(512, K), t1, g * 2)])
    assert gn == [256, 512] and tuple(Wq.shape) == (768, K // 2)
    assert torch.equal(gw, torch.tensor([1.0, 2.0]))
    want = sf_rowmajor_to_mma(np.concatenate([rm0, rm1]))
    assert np.array_equal(Ws.numpy(), want)


def test_pack_weight_groups_rejects_ragged_groups():
    K = 256
    _, t = _scales_tile(128, K, 3)
    with pytest.raises(ValueError, match="multiple of 256"):
        nv.pack_weight_groups([(_codes(128, K), t, torch.ones(1))])


def test_grouped_needs_one_scale_per_group():
    K = 256
    X = torch.zeros(8, K, dtype=torch.bfloat16)
    _, t = _scales_tile(512, K, 4)
    with pytest.raises(ValueError, match="one scale per group"):
        nv.nvfp4_linear_grouped(X, _codes(512, K), t, torch.ones(1), [256, 256])


def test_lora_factor_shapes_are_checked():
    M, K, N, r = 256, 512, 256, 32
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    _, t = _scales_tile(N, K, 5)
    A = torch.zeros(r, K, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="lora_B"):
        nv.nvfp4_linear_lora(X, _codes(N, K), t, torch.ones(1), A,
                             torch.zeros(r, N, dtype=torch.bfloat16), 1.0)  # transposed B
    with pytest.raises(ValueError, match="lora_A"):
        nv.nvfp4_linear_lora(X, _codes(N, K), t, torch.ones(1), A.float(),
                             torch.zeros(N, r, dtype=torch.bfloat16), 1.0)


def test_bias_must_match_the_output_columns():
    M, K, N = 256, 512, 256
    X = torch.zeros(M, K, dtype=torch.bfloat16)
    _, t = _scales_tile(N, K, 6)
    with pytest.raises(ValueError, match="bias"):
        nv.nvfp4_linear_bias_requant(X, _codes(N, K), t, torch.ones(1), None,
                                     bias=torch.zeros(N + 1, dtype=torch.bfloat16))
