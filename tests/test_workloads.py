"""The seeded synthetic inputs (workloads/): shapes, dtypes, the stated distributions and
determinism, for the linear-layer configurations and the DiT block.  The module holds no
method arithmetic; these checks keep both sides of every parity test on the same bytes."""

import math

import torch

import workloads


def test_linear_configs_shapes_and_determinism():
    cfg = workloads.LINEARS["tiny"]
    w = workloads.weight(cfg, seed=0)
    assert w.shape == (cfg.N, cfg.K) and w.dtype == torch.float32
    assert torch.equal(w, workloads.weight(cfg, seed=0))
    assert not torch.equal(w, workloads.weight(cfg, seed=1))
    x = workloads.activations(cfg, seed=0)
    assert x.shape == (cfg.M, cfg.K) and x.dtype == torch.bfloat16
    A, B = workloads.lora(cfg)
    assert A.shape == (workloads.LORA_RANK, cfg.K) and B.shape == (cfg.N, workloads.LORA_RANK)
    assert abs(A.std().item() - 1.0 / 32.0) < 0.1 / 32.0 and abs(B.std().item() - 0.01) < 0.001


def test_student_t_weights_have_the_stated_std():
    cfg = workloads.LINEARS["flux_up"]
    small = workloads.LinearConfig("t", M=8, K=1024, N=1024, w_dist="student_t4")
    w = workloads.weight(small, seed=0).float()
    assert abs(w.std().item() - 0.02) < 0.002           # t(4) scaled to std 0.02
    assert w.abs().max().item() > 6 * 0.02              # heavier tails than a normal of that std
    assert cfg.M == 8 * 4608 and (cfg.K, cfg.N) == (3072, 12288)


def test_block_inputs():
    cfg = workloads.BLOCKS["tiny"]
    x = workloads.block_input(cfg, seed=0)
    assert x.shape == (cfg.B * cfg.S, cfg.D) and x.dtype == torch.bfloat16
    assert torch.equal(x, workloads.block_input(cfg, seed=0))
    wts = workloads.block_weights(cfg, seed=0)
    assert tuple(wts) == workloads.BLOCK_LINEARS
    for name, (W, b) in wts.items():
        N, K = workloads.block_linear_shape(cfg, name)
        assert W.shape == (N, K) and b.shape == (N,) and W.dtype == b.dtype == torch.bfloat16
        assert abs(W.float().std().item() - 0.02) < 0.002
    # the four linears draw from different streams
    assert not torch.equal(wts["qkv"][0][: cfg.D], wts["o"][0])
    flux = workloads.BLOCKS["flux"]
    assert (flux.B, flux.S, flux.D, flux.H) == (8, 4608, 3072, 24) and flux.D % flux.H == 0
    assert math.isclose(flux.D / flux.H, 128)
