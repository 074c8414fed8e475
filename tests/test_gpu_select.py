"""Parity of select_contrastive (through the C ABI) with the oracle.

Selected seed indices must match bit for bit.  The shaped rewards are fp32
results of an fp64 computation whose summation order differs between the two
sides; the difference is at most one fp32 rounding step, so the tolerance is
2^-22 absolute on values in [0, 1].
"""

import numpy as np
import pytest
import torch

import nvfp4_quantized_dit_gb300 as nv
import workloads
from gpu_util import np_, require_gpu

pytestmark = pytest.mark.gpu

TOL = 2.0 ** -22


def _check(orc, rewards, K, global_std=True, with_transform=True):
    idx, r = nv.select_contrastive(rewards.cuda(), K, global_std, with_transform)
    torch.cuda.synchronize()
    oidx, orr = orc.select_contrastive(rewards.numpy(), K, global_std, with_transform)
    assert np.array_equal(np_(idx), oidx)
    if with_transform:
        assert np.all(np.abs(np_(r) - orr) <= TOL), np.max(np.abs(np_(r) - orr))


@pytest.mark.parametrize("name", ["tiny", "iter"])
def test_select_configs(orc, name):
    require_gpu()
    cfg = workloads.REWARDS[name]
    _check(orc, workloads.rewards(cfg, seed=0), cfg.K)


@pytest.mark.parametrize("P,N,K,global_std", [
    (1, 96, 24, False), (32, 96, 24, False), (33, 96, 24, True), (5, 10, 10, True),
    (3, 17, 2, False), (70, 1024, 64, True), (64, 96, 96, True),
    # more prompts than SMs: transform CTAs take several prompts each
    (400, 96, 24, True), (300, 128, 40, False),
])
def test_select_shapes(orc, P, N, K, global_std):
    require_gpu()
    g = torch.Generator().manual_seed(P * N + K)
    _check(orc, torch.randn(P, N, generator=g), K, global_std)


def test_select_ties_and_signed_zeros(orc):
    require_gpu()
    g = torch.Generator().manual_seed(3)
    v = torch.round(torch.randn(16, 96, generator=g) * 2) / 2
    v[v == 0] = torch.where(torch.rand(int((v == 0).sum()), generator=g) < 0.5,
                            torch.tensor(-0.0), torch.tensor(0.0))
    v[3] = 1.25  # all equal: Z = 0 for the per-prompt std
    _check(orc, v, 24, True)
    _check(orc, v, 24, False)


def test_select_without_transform(orc):
    require_gpu()
    v = workloads.rewards(workloads.REWARDS["iter"], seed=4)
    _check(orc, v, 24, True, with_transform=False)


def test_select_all_equal_gives_half(orc):
    require_gpu()
    _check(orc, torch.full((4, 96), 0.7), 24, True)
