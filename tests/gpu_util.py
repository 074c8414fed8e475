"""Test-side helpers for the GPU parity tests.

The scale-factor layout helpers restate the 128x4 blocked layout documented in
include/nvfp4rl.h; they share no code with the CUDA kernels (which write the
layout) or with the oracle (which is layout-free, row-major).
"""

import numpy as np
import pytest
import torch


def require_gpu():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a usable CUDA device")


def sf_index(rows_pad: int, K: int) -> np.ndarray:
    """index[row, kblk] = byte offset of that scale in the blocked buffer."""
    r = np.arange(rows_pad, dtype=np.int64)[:, None]
    kb = np.arange(K // 16, dtype=np.int64)[None, :]
    return ((r // 128) * (K // 64) + kb // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + kb % 4


def unswizzle_sf(sf_flat, rows: int, K: int):
    """Blocked buffer -> (row-major [rows, K/16], padding rows [rows_pad-rows, K/16])."""
    sf_flat = np.asarray(sf_flat).reshape(-1)
    rows_pad = (rows + 127) // 128 * 128
    assert sf_flat.size == rows_pad * (K // 16)
    full = sf_flat[sf_index(rows_pad, K)]
    return full[:rows], full[rows:]


def swizzle_sf(sf_rowmajor, K: int) -> np.ndarray:
    """Row-major [rows, K/16] -> blocked buffer (padding rows 0)."""
    sf_rowmajor = np.asarray(sf_rowmajor, np.uint8)
    rows = sf_rowmajor.shape[0]
    rows_pad = (rows + 127) // 128 * 128
    out = np.zeros(rows_pad * (K // 16), np.uint8)
    idx = sf_index(rows_pad, K)
    out[idx[:rows].reshape(-1)] = sf_rowmajor.reshape(-1)
    return out


def np_(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def assert_gemm_close(y_gpu_bits, y_ref, S, what=""):
    """|y - y_ref| <= 1e-3 * sum_k |a_k b_k| + 2^-8 |y_ref| (bf16 output rounding)."""
    y = bf16_to_f64(y_gpu_bits)
    err = np.abs(y - y_ref)
    tol = 1e-3 * S + 2.0 ** -8 * np.abs(y_ref)
    bad = err > tol
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside tolerance; first at {tuple(i)}:"
                             f" gpu {y[tuple(i)]!r} ref {y_ref[tuple(i)]!r} tol {tol[tuple(i)]!r}")
