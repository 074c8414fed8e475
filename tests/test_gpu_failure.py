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


def test_gemm_abort_path_frees_everything_and_the_next_call_is_clean(orc):
    """The NVFP4 GEMM's own abort path: the first CTA pair's even CTA never loads one
    K-stage (test hook), so its MMA issuer, scale writers and epilogue, and the odd
    CTA's roles, all run into their bounded waits (50 ms here).  The status must read
    NVFP4_ERR_TIMEOUT; afterwards the same GEMM, and a larger one that uses every SM
    (each allocates tensor memory again), must match the oracle with a clean status."""
    require_gpu()
    import numpy as np

    import workloads
    from gpu_util import assert_gemm_close, np_, swizzle_sf

    def operand(rows, K, seed, stream):
        c, sf, s = [t.numpy() for t in workloads.random_nvfp4_operand(rows, K, seed, stream)]
        return c, sf, s

    def gpu(c, sf, s, K):
        return (torch.from_numpy(c).cuda(), torch.from_numpy(swizzle_sf(sf, K)).cuda(),
                torch.from_numpy(np.ascontiguousarray(s, np.float32)).cuda())

    assert nv.nvfp4_device_status(clear=True) in (0, 6)
    M, N, K = 256, 256, 1024
    ac, asf, a_s = operand(M, K, 21, 0)
    wc, wsf, w_s = operand(N, K, 22, 1)
    a, w = gpu(ac, asf, a_s, K), gpu(wc, wsf, w_s[:1], K)
    nv.nvfp4_test_gemm_withhold(a, w, withhold_kb=1, timeout_ns=50_000_000)
    assert nv.nvfp4_device_status(clear=True) == 6
    y = nv.nvfp4_gemm(a, w)
    assert nv.nvfp4_device_status(clear=True) == 0
    y_ref, S = orc.gemm_nvfp4(ac, asf, a_s, wc, wsf, w_s[:1])
    assert_gemm_close(np_(y), y_ref, S, "after abort")
    M2, N2 = 8192, 4096
    ac2, asf2, a_s2 = operand(M2, K, 23, 0)
    wc2, wsf2, w_s2 = operand(N2, K, 24, 1)
    y2 = nv.nvfp4_gemm(gpu(ac2, asf2, a_s2, K), gpu(wc2, wsf2, w_s2[:1], K))
    assert nv.nvfp4_device_status(clear=True) == 0
    rows = np.concatenate([np.arange(0, 8192, 61), np.arange(M2 - 8, M2)])
    y_ref2, S2 = orc.gemm_nvfp4(ac2, asf2, a_s2, wc2, wsf2, w_s2[:1], rows=rows)
    assert_gemm_close(np_(y2)[rows], y_ref2, S2, "every SM after abort")


def test_attention_abort_path_frees_everything():
    """The fused attention's own abort path: one K tile of the first CTA pair is never
    loaded (test hook), every wait is bounded by 50 ms.  The pair must record
    NVFP4_ERR_TIMEOUT and exit with its tensor memory freed: the same attention then
    runs correctly, and so does a larger one that puts a CTA pair on every SM."""
    require_gpu()
    import numpy as np

    import oracle as orc
    from gpu_util import np_

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(orc.bf16_rne(a)).view(np.int16)).view(torch.bfloat16).cuda()

    def check(o, qkv, B, S, H, images):
        o, qkv = np_(o), np_(qkv)
        D = qkv.shape[1] // 3
        for b in images:
            rs = slice(b * S, (b + 1) * S)
            ref = orc.attention(qkv[rs], 1, S, H)
            vo, vr = orc.bf16_value(o[rs]), orc.bf16_value(ref)
            assert (o[rs] == ref).mean() > 0.95
            assert np.max(np.abs(vo - vr)) <= 2.0 ** -6 * np.max(np.abs(vr))
        assert o.shape[1] == D

    assert nv.nvfp4_device_status(clear=True) in (0, 6)
    rng = np.random.default_rng(31)
    B, S, D, H = 2, 512, 256, 2
    qkv = bf16(rng.standard_normal((B * S, 3 * D)) * 0.5)
    nv.nvfp4_test_attention_withhold(qkv, B, S, H, withhold_tile=1, timeout_ns=50_000_000)
    assert nv.nvfp4_device_status(clear=True) == 6
    o = nv.nvfp4_dit_attention(qkv, B, S, H)
    assert nv.nvfp4_device_status(clear=True) == 0
    check(o, qkv, B, S, H, range(B))
    B2, S2 = 8, 2048  # 128 items (image-head, 256 query rows): every pair of the persistent grid works
    qkv2 = bf16(rng.standard_normal((B2 * S2, 3 * D)) * 0.5)
    o2 = nv.nvfp4_dit_attention(qkv2, B2, S2, H)
    assert nv.nvfp4_device_status(clear=True) == 0
    check(o2, qkv2, B2, S2, H, [0, B2 - 1])
