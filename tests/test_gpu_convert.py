"""Exhaustive checks of the device E2M1 / E4M3 rounding against the oracle.

Every fp32 bit pattern in the range the quantizers can produce is converted by
the very device functions the quantizers use (through the library's test hooks)
and compared with the oracle's rounding, which follows the format definitions
(OCP Microscaling Formats, FP4 E2M1; OCP 8-bit Floating Point, E4M3).  This
also settles the nibble order of the packed conversion and the sign of zero.
The quotient tests check the reciprocal fast path with its exact-division
fallback against fl32(x / den) rounded by the oracle, on adversarial inputs.
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
from gpu_util import np_, require_gpu

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26


def _sweep(lo_bits: int, hi_bits: int, gpu_fn, orc_fn, negate: bool):
    dev = torch.device("cuda")
    start = lo_bits
    while start < hi_bits:
        n = min(CHUNK, hi_bits - start)
        bits_np = np.arange(start, start + n, dtype=np.uint32)
        if negate:
            bits_np |= np.uint32(0x80000000)
        vals_np = bits_np.view(np.float32)
        g = gpu_fn(torch.from_numpy(vals_np).to(dev)).cpu().numpy()
        o = orc_fn(vals_np)
        if not np.array_equal(g, o):
            i = int(np.argmax(g != o))
            raise AssertionError(f"mismatch at 0x{int(bits_np[i]):08x} ({vals_np[i]!r}): "
                                 f"gpu 0x{int(g[i]):x} oracle 0x{int(o[i]):x}; "
                                 f"{int((g != o).sum())} mismatches in chunk")
        start += n


@pytest.mark.parametrize("negate", [False, True])
def test_e2m1_exhaustive(orc, negate):
    require_gpu()
    # every fp32 with |q| <= 8, then a sample above (beyond 6 everything saturates)
    _sweep(0, 0x41000001, nv.nvfp4_test_e2m1, orc.e2m1_rne, negate)
    big = np.random.default_rng(2).integers(0x41000001, 0x7F800000, 1 << 20).astype(np.uint32)
    big = big | np.uint32(0x80000000 if negate else 0)
    v = big.view(np.float32)
    got = nv.nvfp4_test_e2m1(torch.from_numpy(v).cuda()).cpu().numpy()
    assert np.array_equal(got, orc.e2m1_rne(v))


def test_e4m3_exhaustive(orc):
    require_gpu()
    # every fp32 in [0, 512], then a sample above (beyond 448 everything saturates)
    _sweep(0, 0x44000001, nv.nvfp4_test_e4m3, orc.e4m3_rne, False)
    big = np.random.default_rng(3).integers(0x44000001, 0x7F800000, 1 << 20).astype(np.uint32)
    v = big.view(np.float32)
    got = nv.nvfp4_test_e4m3(torch.from_numpy(v).cuda()).cpu().numpy()
    assert np.array_equal(got, orc.e4m3_rne(v))


def _adversarial_quotients(rng, thresholds, n_random, den_lo, den_hi):
    den = np.exp(rng.uniform(np.log(den_lo), np.log(den_hi), n_random)).astype(np.float32)
    x = (rng.standard_normal(n_random) * 3).astype(np.float32) * den
    xs, ds = [x], [den]
    # x within a few ulps of t * den for every rounding boundary t, both signs
    d2 = np.exp(rng.uniform(np.log(den_lo), np.log(den_hi), 4096)).astype(np.float32)
    for t in thresholds:
        base = (np.float64(t) * d2.astype(np.float64)).astype(np.float32)
        for k in range(-12, 13):
            xk = base.view(np.int32) + k
            xs.append(xk.view(np.float32))
            ds.append(d2)
            xs.append(-xk.view(np.float32))
            ds.append(d2)
    return np.concatenate(xs), np.concatenate(ds)


def test_e2m1_quotient_fast_path(orc):
    require_gpu()
    rng = np.random.default_rng(0)
    x, den = _adversarial_quotients(rng, [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 1.0, 1.5, 3.0],
                                    1 << 20, 1e-30, 1e30)
    # subnormal and extreme denominators take the exact path
    x2 = rng.standard_normal(4096).astype(np.float32) * np.float32(1e-40)
    d2 = np.full(4096, 1e-41, np.float32)
    x = np.concatenate([x, x2, np.array([0.0, -0.0], np.float32)])
    den = np.concatenate([den, d2, np.array([1.0, 1.0], np.float32)])
    keep = np.isfinite(x)
    x, den = x[keep], den[keep]
    with np.errstate(all="ignore"):
        q = (x / den).astype(np.float32)  # IEEE fp32 division
    want = orc.e2m1_rne(q)
    got = nv.nvfp4_test_e2m1_quotient(torch.from_numpy(x).cuda(), torch.from_numpy(den).cuda()).cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} mismatches"


def test_e4m3_quotient_fast_path(orc):
    require_gpu()
    rng = np.random.default_rng(1)
    vals = [orc.e4m3_decode(c) for c in range(127)]
    mids = [(vals[c] + vals[c + 1]) / 2 for c in range(126)]
    x, d = _adversarial_quotients(rng, mids + vals[1:], 1 << 20, 1e-35, 1e35)
    x = np.abs(x)
    keep = np.isfinite(x)
    x, d = x[keep], d[keep]
    with np.errstate(all="ignore"):
        q = (x / d).astype(np.float32)
    want = orc.e4m3_rne(q)
    got = nv.nvfp4_test_e4m3_quotient(torch.from_numpy(x).cuda(), torch.from_numpy(d).cuda()).cpu().numpy()
    assert np.array_equal(got, want), f"{int((got != want).sum())} mismatches"


def test_e4m3_decode_every_scale_code(orc):
    """Every non-negative finite E4M3 code decodes to the oracle's value, bit for bit
    (the quantizers divide by this value)."""
    require_gpu()
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    got = np_(nv.nvfp4_test_e4m3_decode(codes.cuda()))
    want = np.array([orc.e4m3_decode(int(c)) for c in codes], np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
