"""Shared helpers for the parity tests (host side only)."""
import numpy as np
import torch

# GEMM tolerance: |y - y_ref| <= 2^-7 |y_ref| + 1e-3 ||Y_ref[m, :]||_2, with
# y_ref the oracle's FP64 contraction of the dequantized operands rounded once
# to bfloat16.
REL_TOL = 2.0 ** -7
ROW_FLOOR = 1e-3


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_np_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").contiguous().view(torch.uint8).numpy()


def sf_rowmajor_to_mma(sf: np.ndarray) -> np.ndarray:
    """Row-major (rows, K/16) scales -> the 128x4 tile layout, written from
    its definition in include/nvfp4.h: scale (r, j) sits in tile
    (r // 128) * (K/64) + j // 4 at byte (r % 32) * 16 + ((r % 128) // 32) * 4
    + j % 4; padding rows are 0."""
    rows, kb = sf.shape
    rows_pad = (rows + 127) // 128 * 128
    out = np.zeros(rows_pad * kb, np.uint8)
    r = np.arange(rows)[:, None]
    j = np.arange(kb)[None, :]
    off = ((r // 128) * (kb // 4) + j // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4
    out[off.ravel()] = sf.ravel()
    return out.reshape(rows_pad, kb)


def check_gemm_tolerance(y_bits: np.ndarray, yref_bits: np.ndarray, label: str = ""):
    """Assert the GEMM tolerance elementwise; returns (max_rel, n_floor_only)."""
    y = bits_to_f64(y_bits)
    yr = bits_to_f64(yref_bits)
    assert y.shape == yr.shape
    assert np.all(np.isfinite(y)), "%s: non-finite outputs" % label
    row_norm = np.sqrt(np.sum(yr * yr, axis=1, keepdims=True))
    err = np.abs(y - yr)
    rel_part = REL_TOL * np.abs(yr)
    bound = rel_part + ROW_FLOOR * row_norm
    bad = err > bound
    if np.any(bad):
        i, j = np.argwhere(bad)[0]
        raise AssertionError("%s: %d elements out of tolerance, first at (%d, %d): y=%r ref=%r "
                             "bound=%r" % (label, int(bad.sum()), i, j, y[i, j], yr[i, j],
                                           bound[i, j]))
    floor_only = int(np.sum(err > rel_part))
    nz = np.abs(yr) > 0
    max_rel = float(np.max(err[nz] / np.abs(yr[nz]))) if np.any(nz) else 0.0
    return max_rel, floor_only


def tile_covering_rows(M: int, step: int, seed: int = 1) -> np.ndarray:
    """One random row in every `step`-row band of [0, M), plus the first and
    last row. With step dividing 128 every CTA's 128 accumulator rows of
    every output tile (whole tiles and the column halves of the partial last
    wave alike, since each sampled row is checked across all N columns) are
    sampled; the offset within a band cycles through the four 32-lane TMEM
    quarters from band to band."""
    rng = np.random.default_rng(seed)
    starts = np.arange(0, M, step)
    quarter = (np.arange(len(starts)) % 4) * 32 if step == 128 else 0
    within = quarter + rng.integers(0, min(step, 32), len(starts))
    rows = np.minimum(starts + within, M - 1)
    return np.unique(np.concatenate([[0, M - 1], rows]))
