"""Failure detection without a GPU fault.

Every wait inside the library's kernels is bounded.  The test hook launches one
CTA that waits on a barrier nothing completes; it must give up after the given
limit, record NVFP4_ERR_TIMEOUT in the device status word, and leave the context
usable (the next calls succeed and report a clean status).
"""

import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    require_gpu()
    assert nv.nvfp4_device_status(clear=True) in (0, 6)
    nv.nvfp4_test_wait_timeout(50_000_000)  # 50 ms
    assert nv.nvfp4_device_status(clear=True) == 6
    assert nv.nvfp4_device_status(clear=True) == 0
    X = torch.randn(256, 256, device="cuda").to(torch.bfloat16)
    W = torch.randn(512, 256, device="cuda").to(torch.bfloat16)
    y = nv.bf16_gemm(X, W)
    ref = (X.float() @ W.float().T)
    assert torch.allclose(y.float(), ref, rtol=2e-2, atol=2e-2)
    assert nv.nvfp4_device_status(clear=False) == 0
