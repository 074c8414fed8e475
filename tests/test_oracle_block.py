"""Pins of the oracle's synthetic DiT block (reading R11 in oracle/oracle.c): bf16
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
