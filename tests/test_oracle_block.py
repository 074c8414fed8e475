"""Pins of the oracle's synthetic DiT block (reading R15 in oracle/oracle.c's header): bf16
rounding, the attention softmax, the GELU (tanh form), the residual add, one
attention head and the block's wiring.  Each is checked against a library routine
(torch's float32 -> bf16 conversion and bf16 addition, scipy's softmax and erf), a
closed form or an identity, not against a retyped formula."""

import numpy as np
import pytest
import torch

import oracle as orc

scipy_special = pytest.importorskip("scipy.special")


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_float32_inputs():
    """Values exactly representable in float32: the direct rounding must equal torch's
    float32 -> bf16 conversion (nearest, ties to even), subnormals and overflow included."""
    rng = np.random.default_rng(0)
    with np.errstate(over="ignore", invalid="ignore"):
        x = np.concatenate([
            (rng.standard_normal(100000) * 10.0 ** rng.integers(-30, 30, 100000)).astype(np.float32),
            np.frombuffer(rng.bytes(4 * 100000), np.uint32).view(np.float32),
            np.array([0.0, -0.0, 1e-45, -1e-45, 1.17e-38, 3.39e38, 3.4e38, -3.4e38], np.float32),
        ])
    assert x.dtype == np.float32
    x = x[np.isfinite(x)]
    want = _bits(torch.from_numpy(x).to(torch.bfloat16))
    got = orc.bf16_rne(x.astype(np.float64))
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


def test_bf16_rne_ties_and_neighbours():
    """Every bf16 value maps to itself; the midpoint of two neighbours goes to the one
    with an even last bit, and any nudge off the midpoint to the nearer one."""
    b = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)  # finite non-negative patterns
    v = orc.bf16_value(b)
    assert np.array_equal(orc.bf16_rne(v), b)
    assert np.array_equal(orc.bf16_rne(-v)[1:], b[1:] | 0x8000)
    lo, hi = v[:-1], v[1:]
    mid = (lo + hi) / 2  # exact in double
    want = np.where(b[:-1] % 2 == 0, b[:-1], b[1:])
    assert np.array_equal(orc.bf16_rne(mid), want)
    eps = (hi - lo) * 2.0 ** -20
    assert np.array_equal(orc.bf16_rne(mid - eps), b[:-1])
    assert np.array_equal(orc.bf16_rne(mid + eps), b[1:])


def test_softmax_matches_scipy_and_closed_forms():
    rng = np.random.default_rng(1)
    L = _bits(torch.from_numpy(rng.standard_normal((64, 300)).astype(np.float32) * 4).to(torch.bfloat16))
    scale = 1 / np.sqrt(128)
    P = orc.softmax_bf16(L, scale)
    ref = scipy_special.softmax(orc.bf16_value(L) * scale, axis=1)
    # Equal after rounding, except where the reference is within 1e-9 (relative) of a
    # bf16 midpoint, where the two double evaluations may round apart.
    r = orc.bf16_rne(ref)
    near = np.abs(ref - orc.bf16_value(r)) > orc.bf16_value(r) * (2.0 ** -9 - 1e-9)
    assert np.array_equal(P[~near], r[~near])
    # A constant row: every probability is bf16(1 / cols).
    assert np.all(orc.softmax_bf16(np.full((2, 256), 0x4040, np.uint16), 0.3) == orc.bf16_rne(1 / 256))
    # One logit far above the rest takes all the mass.
    L2 = np.zeros((1, 100), np.uint16)
    L2[0, 37] = orc.bf16_rne(1e4)
    P2 = orc.bf16_value(orc.softmax_bf16(L2, 1.0))
    assert P2[0, 37] == 1.0 and P2.sum() == 1.0
    # Shifting a row of integers by an integer leaves it unchanged.
    ints = rng.integers(-8, 8, (4, 64)).astype(np.float64)
    assert np.array_equal(orc.softmax_bf16(orc.bf16_rne(ints), 0.5), orc.softmax_bf16(orc.bf16_rne(ints + 3), 0.5))


def test_gelu_identity_and_erf_form():
    x = np.linspace(-12, 12, 48001)
    g = orc.gelu_f64(x)
    gn = orc.gelu_f64(-x)
    # The tanh form satisfies g(x) - g(-x) = x exactly in real arithmetic.
    assert np.all(np.abs(g - gn - x) <= 4e-16 * (1 + np.abs(x)))
    assert orc.gelu_f64(np.array([0.0]))[0] == 0.0
    # Within the known gap of the tanh approximation to x Phi(x) (about 2e-4).
    exact = 0.5 * x * (1 + scipy_special.erf(x / np.sqrt(2)))
    assert np.max(np.abs(g - exact)) < 5e-4
    assert np.max(np.abs(g - exact)[np.abs(x) > 6]) < 1e-7
    # The bf16 version is the rounded double version on bf16 inputs.
    xb = orc.bf16_rne(x)
    assert np.array_equal(orc.gelu_bf16(xb), orc.bf16_rne(orc.gelu_f64(orc.bf16_value(xb))))


def test_gelu_tail_against_high_precision():
    """The tanh form evaluated at 60 digits by mpmath, across the range where 1 + tanh(t)
    cancels (x down to -11, where g(x) is about -1e-48): the double result keeps its
    relative accuracy there, and the bf16 result is the high-precision value rounded
    (subnormal bf16 values included)."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    k = mpmath.sqrt(2 / mpmath.pi)
    x = np.concatenate([np.linspace(-11, -3, 801), np.linspace(-3, 3, 301), np.array([5.0, 9.0])])
    hp = [0.5 * mpmath.mpf(v) * (1 + mpmath.tanh(k * (mpmath.mpf(v) + mpmath.mpf("0.044715") * mpmath.mpf(v) ** 3)))
          for v in x]
    g = orc.gelu_f64(x)
    rel = np.array([abs((mpmath.mpf(gi) - h) / h) if h != 0 else abs(gi) for gi, h in zip(g, hp)], np.float64)
    assert rel.max() < 1e-13
    xb = orc.bf16_rne(x)
    xv = orc.bf16_value(xb)
    hb = np.array([float(0.5 * mpmath.mpf(v) * (1 + mpmath.tanh(k * (mpmath.mpf(v) + mpmath.mpf("0.044715") * mpmath.mpf(v) ** 3))))
                   for v in xv])
    assert np.array_equal(orc.gelu_bf16(xb), orc.bf16_rne(hb))
    assert (orc.bf16_value(orc.gelu_bf16(xb)) < 0).sum() > 700  # the negative tail does not flush to zero


def test_add_matches_torch_bf16_addition():
    rng = np.random.default_rng(2)
    a = torch.from_numpy((rng.standard_normal(200000) * 10.0 ** rng.integers(-6, 6, 200000)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy((rng.standard_normal(200000) * 10.0 ** rng.integers(-6, 6, 200000)).astype(np.float32)).to(torch.bfloat16)
    assert np.array_equal(orc.add_bf16(_bits(a), _bits(b)), _bits(a + b))


def test_attention_head_closed_forms():
    rng = np.random.default_rng(3)
    S, dh = 256, 128
    v = orc.bf16_rne(rng.standard_normal((S, dh)))
    k = orc.bf16_rne(rng.standard_normal((S, dh)))
    # q = 0: uniform probabilities 1/256 (exact in bf16), O = bf16(mean of the rows of v).
    o = orc.attention_head(np.zeros((S, dh), np.uint16), k, v)
    assert np.array_equal(o, orc.bf16_rne(orc.bf16_value(v).mean(axis=0))[None, :].repeat(S, 0))
    # Every query aligned with one key only, far above the others: O = that key's value row.
    q = np.zeros((S, dh), np.uint16)
    k2 = np.zeros((S, dh), np.uint16)
    q[:, 5] = orc.bf16_rne(64.0)
    k2[77, 5] = orc.bf16_rne(64.0)
    o2 = orc.attention_head(q, k2, v)
    assert np.array_equal(o2, v[77][None, :].repeat(S, 0))


def test_block_residual_wiring():
    """With zero output projections (and zero biases) the block returns its input,
    whatever the other weights: both residual connections carry x through."""
    rng = np.random.default_rng(4)
    B, S, H, dh = 2, 64, 2, 128
    D = H * dh
    x = orc.bf16_rne(rng.standard_normal((B * S, D)))
    def weight(n, k, scale):
        return orc.requant(orc.bf16_rne(rng.standard_normal((n, k)) * scale), None, None, 32.0)
    zero = lambda n, k: orc.requant(np.zeros((n, k), np.uint16), None, None, 32.0)
    w = {"qkv": weight(3 * D, D, 0.05), "o": zero(D, D), "up": weight(4 * D, D, 0.05), "dn": zero(D, 4 * D)}
    r = orc.dit_block(x, w, {}, B, S, H)
    assert r["qkv"].shape == (B * S, 3 * D) and r["u"].shape == (B * S, 4 * D)
    assert np.array_equal(r["h1"], x) and np.array_equal(r["out"], x)
    # Zero everywhere: the attention output is zero too (uniform weights over zero values).
    wz = {"qkv": zero(3 * D, D), "o": zero(D, D), "up": zero(4 * D, D), "dn": zero(D, 4 * D)}
    rz = orc.dit_block(x, wz, {}, B, S, H)
    assert not orc.bf16_value(rz["o"]).any() and np.array_equal(rz["out"], x)


def test_block_rows_equals_whole_block():
    """The row-restricted block (for inputs too large to run whole) reproduces the whole
    block's output bit for bit on the chosen rows, rows of the first and last image
    included, with biases on every linear."""
    rng = np.random.default_rng(6)
    B, S, H, dh = 3, 64, 2, 64
    D = H * dh
    x = orc.bf16_rne(rng.standard_normal((B * S, D)))
    shapes = {"qkv": (3 * D, D), "o": (D, D), "up": (4 * D, D), "dn": (D, 4 * D)}
    w = {k: orc.requant(orc.bf16_rne(rng.standard_normal(sh) * 0.05), None, None, 32.0) for k, sh in shapes.items()}
    bias = {k: orc.bf16_rne(rng.standard_normal(sh[0]) * 0.02) for k, sh in shapes.items()}
    full = orc.dit_block(x, w, bias, B, S, H)["out"]
    rows = np.array([0, 5, 63, 2 * S, 2 * S + 17, 3 * S - 1])
    assert np.array_equal(orc.dit_block_rows(x, w, bias, B, S, H, rows), full[rows])


def _grid_weight(rng, N, K):
    """A bf16 weight that per-tensor NVFP4 represents exactly: tensor amax 2688 * 2^-12
    (so s = 2^-12), every 16-block c * sf * s with c on the E2M1 grid and sf an E4M3
    value, one element of each block at |c| = 6 (so the block scale is sf itself)."""
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    sfs = np.array([448.0, 224.0, 112.0, 96.0, 56.0, 40.0, 13.0, 1.5, 0.25])
    c = grid[rng.integers(0, 8, (N, K))] * rng.choice([-1.0, 1.0], (N, K))
    c.reshape(N, K // 16, 16)[:, :, 0] = 6.0 * rng.choice([-1.0, 1.0], (N, K // 16))
    sf = sfs[rng.integers(0, len(sfs), (N, K // 16))]
    sf[0, 0] = 448.0
    W = c * np.repeat(sf, 16, axis=1) * 2.0 ** -12
    bits = orc.bf16_rne(W)
    assert np.array_equal(orc.bf16_value(bits), W)
    return bits


def test_linear_unquantized_is_the_bf16_product_on_grid_weights():
    """On a weight that NVFP4 represents exactly, the unquantized-activation linear is
    the plain product of the bf16 activations with that weight: it must equal the
    oracle's bf16 GEMM (rounded to bf16), bias included, bit for bit."""
    rng = np.random.default_rng(8)
    N, K, T = 96, 256, 40
    w_bits = _grid_weight(rng, N, K)
    w = orc.requant(w_bits, None, None, 32.0)
    assert np.float32(np.asarray(w[2]).reshape(-1)[0]) == np.float32(2.0 ** -12)
    assert np.array_equal(orc.dequantize(w[0], w[1], w[2], "tensor"), orc.bf16_value(w_bits))
    x = orc.bf16_rne(rng.standard_normal((T, K)))
    b = orc.bf16_rne(rng.standard_normal(N) * 0.1)
    ref = orc.bf16_rne(orc.gemm_bf16(x, w_bits, b)[0])
    assert np.array_equal(orc.linear_unquantized(x, w, b), ref)
    # The quantized linear on the same weight differs (the activations are quantized).
    assert not np.array_equal(orc.nvfp4_linear(x, w, b), ref)


def test_block_rows_unquantized_mode():
    """quantize_activations=False changes only the linears: with zero output
    projections the block is still the identity, and otherwise it stays close to the
    NVFP4 block (their gap is the activation quantization's, a few percent)."""
    rng = np.random.default_rng(9)
    B, S, H, dh = 2, 64, 2, 64
    D = H * dh
    x = orc.bf16_rne(rng.standard_normal((B * S, D)))
    shapes = {"qkv": (3 * D, D), "o": (D, D), "up": (4 * D, D), "dn": (D, 4 * D)}
    w = {k: orc.requant(orc.bf16_rne(rng.standard_normal(sh) * 0.05), None, None, 32.0) for k, sh in shapes.items()}
    rows = np.array([1, 70, 127])
    wz = dict(w, o=orc.requant(np.zeros(shapes["o"], np.uint16), None, None, 32.0),
              dn=orc.requant(np.zeros(shapes["dn"], np.uint16), None, None, 32.0))
    assert np.array_equal(orc.dit_block_rows(x, wz, {}, B, S, H, rows, quantize_activations=False), x[rows])
    q = orc.bf16_value(orc.dit_block_rows(x, w, {}, B, S, H, rows))
    u = orc.bf16_value(orc.dit_block_rows(x, w, {}, B, S, H, rows, quantize_activations=False))
    gap = np.linalg.norm(q - u) / np.linalg.norm(u)
    assert 1e-3 < gap < 0.2


def test_attention_head_applies_the_scale():
    """Two keys whose logits differ by a: P = (1/(1 + e^(-a s)), 1/(1 + e^(a s))) with s =
    1/sqrt(dh) (dh = 64: s = 1/8 exactly, dh = 128: the fp32 value of 1/sqrt(128)); v
    picks each probability out into its own column of O.  A missing or different scale
    (none, 1/dh, sqrt(dh)) changes P by far more than a bf16 step."""
    for dh in (64, 128):
        s = float(np.float32(1.0) / np.sqrt(np.float32(dh)))
        for a in (1.0, 4.0, 10.0, -7.5):
            q = np.zeros((2, dh), np.uint16)
            k = np.zeros((2, dh), np.uint16)
            v = np.zeros((2, dh), np.uint16)
            q[:, 0] = orc.bf16_rne(a)
            k[0, 0] = orc.bf16_rne(1.0)  # logits: a for key 0, 0 for key 1 (exact in bf16)
            v[0, 1] = orc.bf16_rne(1.0)
            v[1, 2] = orc.bf16_rne(1.0)
            o = orc.bf16_value(orc.attention_head(q, k, v))
            p0 = 1.0 / (1.0 + np.exp(-a * s))
            p1 = 1.0 / (1.0 + np.exp(a * s))
            for col, p in ((1, p0), (2, p1)):
                # P is rounded to bf16, then O = bf16(P * 1): two roundings of p
                assert np.all(o[:, col] == orc.bf16_value(orc.bf16_rne(orc.bf16_value(orc.bf16_rne(p)))))
            for wrong in (1.0, 1.0 / dh, np.sqrt(dh)):
                pw = 1.0 / (1.0 + np.exp(-a * wrong))
                assert abs(pw - p0) > 2.0 ** -7 * max(p0, 1e-30)
