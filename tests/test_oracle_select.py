"""Pins for the oracle's contrastive filter and reward transform.

Filter: Sol-RL project page, "Two-Stage Pipeline" (Stage 1 keeps the top/bottom
seeds out of N = 96; K = 24 are regenerated), with the AI Trends summary's split
into top K/2 and bottom K/2.  Transform: "DiffusionNFT" (VeRL-Omni
documentation), "Algorithm": r = 1/2 + 1/2 clip((r_raw - mean) / Z, -1, 1),
global standard deviation by default.

The filter is checked against Python's sorted() and an O(N^2) rank count; the
transform against a hand-worked example and its invariants.
"""

import math

import numpy as np
import pytest

from conftest import golden_lines


def test_selection_golden_ties(orc):
    lines = golden_lines("selection_ties.txt")
    rewards = np.array([[float(v) for v in lines[0][1:]]], np.float32)
    for ln in lines[1:]:
        K = int(ln[0][1:])
        idx, _ = orc.select_contrastive(rewards, K, with_transform=False)
        assert list(idx[0]) == [int(v) for v in ln[1:]]


def _ref_by_sort(v, K):
    n = len(v)
    top = sorted(range(n), key=lambda i: (-float(v[i]), i))[:K // 2]
    bot = sorted(range(n), key=lambda i: (float(v[i]), i))[:K // 2]
    return top + bot


def _ref_by_rank(v, K):
    n = len(v)
    h = K // 2
    out = [None] * K
    for i in range(n):
        rt = sum(1 for j in range(n) if v[j] > v[i] or (v[j] == v[i] and j < i))
        rb = sum(1 for j in range(n) if v[j] < v[i] or (v[j] == v[i] and j < i))
        if rt < h:
            out[rt] = i
        if rb < h:
            out[h + rb] = i
    return out


@pytest.mark.parametrize("P,N,K", [(1, 96, 24), (5, 96, 24), (3, 10, 10), (4, 17, 2), (2, 64, 40)])
def test_selection_matches_full_sort_and_rank_count(orc, P, N, K):
    rng = np.random.default_rng(P * 100 + N)
    v = np.round(rng.standard_normal((P, N)) * 2) / 2  # many ties
    v[v == 0] = np.where(rng.random((v == 0).sum()) < 0.5, -0.0, 0.0)
    v = v.astype(np.float32)
    idx, _ = orc.select_contrastive(v, K, with_transform=False)
    for p in range(P):
        assert list(idx[p]) == _ref_by_sort(v[p], K) == _ref_by_rank(list(v[p]), K)


@pytest.mark.parametrize("K", [0, 3, 98])
def test_selection_rejects_bad_k(orc, K):
    with pytest.raises(ValueError):
        orc.select_contrastive(np.zeros((1, 96), np.float32), K)


def test_transform_worked_example(orc):
    rows = golden_lines("nft_transform_example.txt")
    idx, r = orc.select_contrastive(np.array([[1, 2, 3, 4]], np.float32), 4)
    assert list(idx[0]) == [int(s) for _, s, _ in rows]
    want = np.array([float(x) for _, _, x in rows], np.float32)
    assert np.all(np.abs(r[0] - want) <= 2.0 ** -24)
    assert r[0][1] == np.float32(0.5 + 0.5 / math.sqrt(5))


def test_transform_invariants(orc):
    rng = np.random.default_rng(11)
    rw = rng.standard_normal((32, 96)).astype(np.float32)
    idx, r = orc.select_contrastive(rw, 24, global_std=True)
    assert np.all((r >= 0) & (r <= 1))
    # monotone in the raw reward within a prompt
    for p in range(32):
        x = rw[p, idx[p]]
        o = np.argsort(x, kind="stable")
        assert np.all(np.diff(r[p][o]) >= 0)
    # extremes of a prompt sit above / below its mean
    assert np.all(r[:, 0] >= 0.5) and np.all(r[:, 12] <= 0.5)


def test_transform_sample_at_mean_is_half(orc):
    """Symmetric rewards {-a, 0, a} around 0: the mean is exactly 0, so the
    sample at the mean maps to exactly 1/2."""
    v = np.array([[-3.0, 0.0, 3.0, -1.5, 1.5, 0.0]], np.float32)
    idx, r = orc.select_contrastive(v, 6)
    x = v[0, idx[0]]
    assert np.all(r[0][x == 0] == np.float32(0.5))


def test_transform_two_samples_per_prompt_std(orc):
    """K = 2 with the per-prompt std: (x - mean)/Z = +-1, so r is exactly 1 and 0."""
    rng = np.random.default_rng(12)
    v = rng.standard_normal((6, 20)).astype(np.float32)
    idx, r = orc.select_contrastive(v, 2, global_std=False)
    assert np.all(r[:, 0] == 1.0) and np.all(r[:, 1] == 0.0)


def test_transform_equal_rewards_give_half(orc):
    idx, r = orc.select_contrastive(np.full((3, 96), 0.7, np.float32), 24)
    assert np.all(r == np.float32(0.5))
    assert list(idx[0]) == list(range(12)) + list(range(12))


def test_transform_global_equals_per_prompt_for_one_prompt(orc):
    v = np.random.default_rng(13).standard_normal((1, 96)).astype(np.float32)
    _, r1 = orc.select_contrastive(v, 24, global_std=True)
    _, r2 = orc.select_contrastive(v, 24, global_std=False)
    assert np.array_equal(r1, r2)


def test_transform_global_std_uses_global_mean(orc):
    """Two prompts whose selected rewards are {0,0,...} + offset: per prompt the
    spread is the same but the global std also sees the offset between prompts."""
    v = np.zeros((2, 4), np.float32)
    v[0] = [1, 2, 3, 4]
    v[1] = [11, 12, 13, 14]
    _, r = orc.select_contrastive(v, 4, global_std=True)
    allx = np.array([4, 3, 1, 2, 14, 13, 11, 12], np.float64)
    Z = allx.std()
    mu = np.array([2.5, 12.5])
    want = 0.5 + 0.5 * np.clip((allx.reshape(2, 4) - mu[:, None]) / Z, -1, 1)
    assert np.all(np.abs(r - want) <= 2.0 ** -24)
