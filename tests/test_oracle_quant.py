"""Pins for the oracle's LoRA merge and NVFP4 quantizer.

Expected values come from closed forms (exact merges on dyadic inputs, the fused
multiply-add case, tensors built on the NVFP4 grid so that quantize-dequantize
is the identity), the quantizer's error bound, and special cases.  Merge rank 32
follows the AI Trends summary (paragraph on training stability, LoRA rank 32);
re-quantization after each update follows the Sol-RL project page
("Two-Stage Pipeline", Stage 2).
"""

from fractions import Fraction

import numpy as np
import pytest


def _bf16_bits(x):
    """Truncate fp32 values that are exactly bf16-representable to bf16 bits."""
    x = np.ascontiguousarray(x, np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "test input not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def test_merge_closed_form_on_dyadic_inputs(orc):
    """With small dyadic A, B, W every partial sum is exact, so the merge must equal
    W + (alpha/r) * B @ A computed in integers.  N, K, r all differ, so a transposed
    factor or a dropped rank term changes the result."""
    rng = np.random.default_rng(3)
    N, K, r = 48, 80, 32
    Ai = rng.integers(-7, 8, (r, K))
    Bi = rng.integers(-7, 8, (N, r))
    Wi = rng.integers(-500, 501, (N, K))
    A = (Ai * 2.0 ** -4).astype(np.float32)
    B = (Bi * 2.0 ** -3).astype(np.float32)
    W = (Wi * 2.0 ** -7).astype(np.float32)
    alpha = 24.0  # c = 0.75
    got = orc.merge(W, A, B, alpha)
    want = (Wi * 4 + 3 * (Bi @ Ai)) * 2.0 ** -9  # W + 0.75 * B@A * 2^-7, exact
    assert np.array_equal(got.astype(np.float64), want)


def test_merge_is_a_fused_sequential_chain(orc):
    """acc = fmaf(B1, A1, fmaf(B0, A0, 0)).  With B0*A0 = -(1 + 2^-11) and
    B1 = A1 = 1 + 2^-12, a fused chain in index order leaves exactly 2^-24; a
    separate multiply and add, or the reverse order, leaves 0."""
    e = 1.0 + 2.0 ** -12
    A = np.array([[-(1.0 + 2.0 ** -11)], [e]], np.float32)  # [r=2, K=1]
    B = np.array([[1.0, e]], np.float32)                     # [N=1, r=2]
    W = np.zeros((1, 1), np.float32)
    got = orc.merge(W, A, B, alpha=2.0)                       # c = 1
    assert got[0, 0] == np.float32(2.0 ** -24)


def test_merge_without_lora_is_identity(orc):
    rng = np.random.default_rng(4)
    W = rng.standard_normal((16, 64)).astype(np.float32)
    assert np.array_equal(orc.merge(W, None, None, 32.0), W)
    Wb = _bf16_bits((W.view(np.uint32) & 0xFFFF0000).view(np.float32))
    got = orc.merge(Wb, None, None, 32.0)
    assert np.array_equal(got.view(np.uint32) >> 16, Wb.astype(np.uint32))


def _grid_tensor(rows, K, k_exp, scopes_rows, rng):
    """Tensor whose every 16-block is e * 2^-k * g with g on the E2M1 grid,
    max |g| = 6 in every block, and e = 448 in at least one block of each scope."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    e4m3 = [Fraction(x) for x in (0.015625, 0.0625, 0.25, 0.5, 1, 1.125, 1.75, 3, 13, 52, 160, 448)]
    x = np.zeros((rows, K), np.float64)
    scales = np.zeros((rows, K // 16))
    codes = np.zeros((rows, K), np.int64)
    for rr in range(rows):
        for b in range(K // 16):
            e = float(e4m3[rng.integers(len(e4m3))])
            gi = rng.integers(0, 8, 16)
            gi[rng.integers(16)] = 7
            sign = rng.integers(0, 2, 16)
            codes[rr, b * 16:(b + 1) * 16] = gi | (sign << 3)
            scales[rr, b] = e
            x[rr, b * 16:(b + 1) * 16] = np.where(sign == 1, -1, 1) * grid[gi] * e * 2.0 ** -k_exp
    for r0 in scopes_rows:  # force one 448 block per scope
        scales[r0, 0] = 448
        g = np.abs(codes[r0, :16]) & 7
        x[r0, :16] = np.where(codes[r0, :16] >> 3 == 1, -1, 1) * grid[g] * 448 * 2.0 ** -k_exp
    return x.astype(np.float32), codes, scales


@pytest.mark.parametrize("scope", ["tensor", "row"])
def test_quantize_exact_reconstruction(orc, scope):
    rng = np.random.default_rng(5)
    rows, K, k_exp = 6, 128, 10
    x, codes, scales = _grid_tensor(rows, K, k_exp, [0] if scope == "tensor" else range(rows), rng)
    qc, sf, s = orc.quantize(x, scope)
    assert np.all(s == np.float32(2.0 ** -k_exp))
    # scales decode to the construction's scales
    dec_sf = np.vectorize(orc.e4m3_decode)(sf.astype(int))
    assert np.array_equal(dec_sf, scales)
    # nibble order: code of even k in the low nibble
    unpacked = np.stack([qc & 15, qc >> 4], axis=-1).reshape(rows, K).astype(np.int64)
    nonzero = (codes & 7) != 0
    assert np.array_equal(unpacked[nonzero], codes[nonzero])
    assert np.all((unpacked[~nonzero] & 7) == 0)
    xh = orc.dequantize(qc, sf, s, scope)
    assert np.array_equal(xh, x.astype(np.float64))


def test_quantize_nibble_order_single_element(orc):
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = 6.0
    x[0, 3] = -3.0
    qc, sf, s = orc.quantize(x, "row")
    assert sf[0, 0] == 0x7E and s[0] == np.float32(6.0) / np.float32(2688.0)
    assert qc[0, 0] == 0x07 and qc[0, 1] == 0xD0


def _gap_half(mag):
    return np.where(mag <= 2, 0.25, np.where(mag <= 4, 0.5, 1.0))


@pytest.mark.parametrize("scope", ["tensor", "row"])
def test_quantize_error_bound(orc, scope):
    """|x - x_hat| <= (gap/2) * sf * s (+ fp32 slack) for every element whose
    quotient is <= 6; the rest are saturated and bounded by |x| - 6 sf s."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    x[:, [3, 77, 200]] *= 25
    x[5] *= 1e-30
    x[6, :40] = 0
    qc, sf, s = orc.quantize(x, scope)
    xh = orc.dequantize(qc, sf, s, scope)
    sff = np.vectorize(orc.e4m3_decode)(sf.astype(int)).repeat(16, axis=1)
    srow = np.broadcast_to(s.astype(np.float64)[:, None] if scope == "row" else s.astype(np.float64),
                           (64, 1))
    den = sff * srow
    xd = x.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(den > 0, np.abs(xd) / den, 0)
    err = np.abs(xd - xh)
    ok = q <= 6
    bound = (_gap_half(q) + q * 2.0 ** -21) * den
    assert np.all(err[ok & (den > 0)] <= bound[ok & (den > 0)])
    sat = (~ok) & (den > 0)
    assert np.all(err[sat] <= np.abs(xd[sat]) - 6 * den[sat] + 1e-30)
    # zero-scale blocks emit zero codes
    assert np.all(xh[den == 0] == 0)


def test_quantize_amax_block_gets_top_scale(orc):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((32, 512)).astype(np.float32)
    qc, sf, s = orc.quantize(x, "tensor")
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, c // 16] == 0x7E
    code = (qc[r, c // 2] >> (4 * (c % 2))) & 15
    assert code & 7 == 7 and (code >> 3) == int(x[r, c] < 0)


def test_quantize_zero_and_tiny(orc):
    qc, sf, s = orc.quantize(np.zeros((3, 64), np.float32), "tensor")
    assert s[0] == 0 and not sf.any() and not qc.any()
    # amax so small that s rounds to 0: every scale and code is 0 (zero scale)
    x = np.full((2, 32), 1e-45, np.float32)
    qc, sf, s = orc.quantize(x, "row")
    assert np.all(s == 0) and not sf.any() and not qc.any()


def test_row_scope_equals_tensor_scope_of_each_row(orc):
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((9, 96)) * rng.uniform(0.01, 100, (9, 1))).astype(np.float32)
    qc, sf, s = orc.quantize(x, "row")
    for r in range(9):
        qc1, sf1, s1 = orc.quantize(x[r:r + 1], "tensor")
        assert np.array_equal(qc1[0], qc[r]) and np.array_equal(sf1[0], sf[r]) and s1[0] == s[r]


def test_act_quant_reads_bf16_bits(orc):
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 64)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)
    qc, sf, s = orc.act_quant(xb)
    qc2, sf2, s2 = orc.quantize(((xb.astype(np.uint32)) << 16).view(np.float32), "row")
    assert np.array_equal(qc, qc2) and np.array_equal(sf, sf2) and np.array_equal(s, s2)


def _rn32(fr):
    """Round a non-negative exact rational to the nearest fp32 value, ties to even
    (normal range only), by integer arithmetic on the rational itself."""
    assert fr > 0
    e = fr.numerator.bit_length() - fr.denominator.bit_length()
    if Fraction(2) ** e > fr:
        e -= 1
    while Fraction(2) ** (e + 1) <= fr:
        e += 1
    ulp = Fraction(2) ** (e - 23)
    q, rem = divmod(fr, ulp)
    q = int(q)
    if rem * 2 > ulp or (rem * 2 == ulp and q % 2 == 1):
        q += 1
    return q * ulp


def test_quotient_is_one_division_at_e2m1_ties(orc):
    """Reading R1 (q = x / (sf * s), one IEEE division) decides exact ties that the
    reciprocal-multiply and two-step forms resolve the other way
    (tests/golden/quotient_ties.txt).  Exact rationals establish, independently of
    the oracle, that each quotient is exactly the boundary and that the other forms
    are above it; the oracle must return the tie's even code."""
    from conftest import golden_lines
    rows = golden_lines("quotient_ties.txt")
    amax = float(rows[0][1])
    elems = [(float(r[1]), float(r[2]), int(r[3], 16), int(r[4], 16)) for r in rows[1:]]
    a = Fraction(np.float32(amax).item())
    s = _rn32(a / 2688)
    d6 = _rn32(6 * s)
    assert _rn32(a / d6) == 448  # block scale exactly 448: code 0x7E
    den = _rn32(448 * s)
    rec = _rn32(1 / den)
    for x, b, _, _ in elems:
        xf = Fraction(np.float32(x).item())
        assert _rn32(xf / den) == Fraction(b)            # exactly the boundary
        assert _rn32(xf * rec) > Fraction(b)             # reciprocal form: above it
        assert _rn32(_rn32(xf / s) / 448) > Fraction(b)  # two-step form: above it
    x = np.zeros((1, 16), np.float32)
    x[0, 0] = amax
    for i, (v, _, _, _) in enumerate(elems):
        x[0, 1 + i] = v
    codes, sf, st = orc.quantize(x, "tensor")
    assert sf[0, 0] == 0x7E
    assert st[0] == np.float32(float(s))
    nib = [(codes[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
    assert nib[0] == 0x7  # the amax element: 6.0
    for i, (_, _, by_div, by_rec) in enumerate(elems):
        assert by_div != by_rec
        assert nib[1 + i] == by_div, f"element {1 + i}: code {nib[1 + i]:#x}, want {by_div:#x}"
    assert all(n == 0 for n in nib[4:])
