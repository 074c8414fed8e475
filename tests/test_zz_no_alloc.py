"""nvfp4_requant_noalloc: the same results as nvfp4_requant with a caller workspace.

Collected last on purpose (the scratch is per device and shared by every call), and
checked both right after other tests and on its own.  The entry point has no
counterpart in the Sol-RL pages; it serves callers that cannot provide scratch.
"""

import ctypes

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
from gpu_util import np_, require_gpu


def _inputs(N, K, seed):
    g = torch.Generator().manual_seed(seed)
    W = (torch.randn(N, K, generator=g) * 0.02).to(torch.bfloat16)
    A = torch.randn(32, K, generator=g) / 32
    B = torch.randn(N, 32, generator=g) * 0.01
    return W.cuda(), A.cuda(), B.cuda()


@pytest.mark.gpu
def test_noalloc_matches_workspace_path_on_two_calls():
    """Two calls with different inputs through each entry point: codes, scales and
    s_t identical, so the shared scratch carries nothing from one call to the next."""
    require_gpu()
    for N, K, seed in [(1024, 3072, 1), (300, 1088, 2)]:
        W, A, B = _inputs(N, K, seed)
        ref = [np_(t) for t in nv.nvfp4_requant(W, A, B, 32.0)]
        got = [np_(t) for t in nv.nvfp4_requant_noalloc(W, A, B, 32.0)]
        torch.cuda.synchronize()
        for r, x, name in zip(ref, got, ["codes", "sf", "s_t"]):
            assert np.array_equal(r.view(np.uint8), x.view(np.uint8)), f"{name} differ at N={N} K={K}"
    assert nv.nvfp4_device_status() == 0


@pytest.mark.gpu
def test_noalloc_without_merge_and_with_fp32_weights():
    """Paths that need no scratch (no LoRA, fp32 weights) go through unchanged."""
    require_gpu()
    W, A, B = _inputs(256, 512, 3)
    for args in [(W, None, None), (W.float(), A, B)]:
        ref = [np_(t) for t in nv.nvfp4_requant(*args, 32.0)]
        got = [np_(t) for t in nv.nvfp4_requant_noalloc(*args, 32.0)]
        for r, x in zip(ref, got):
            assert np.array_equal(r.view(np.uint8), x.view(np.uint8))


def test_noalloc_rejects_sizes_above_its_scratch():
    """A shape whose workspace exceeds the fixed scratch is refused before any CUDA
    call (K = 65536: A' alone is 16 MiB)."""
    lib = nv.library()
    P = ctypes.c_void_p
    A16 = 0x10000
    rc = lib.nvfp4_requant_noalloc(P(A16), 0, P(A16), P(A16), 32, ctypes.c_float(32.0), 64, 65536,
                                   P(A16), P(A16), P(A16), None)
    assert rc == 2  # NVFP4_ERR_SHAPE
