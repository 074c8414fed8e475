"""Seeded synthetic inputs for the NVFP4 FP4-explore hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no merging, no quantization, no GEMM, no selection).  It is
the one module that both the CPU oracle's tests and the CUDA library's tests and
benchmark use, so that both sides see identical bytes.

Shapes follow the linear layers named on the Sol-RL project page ("Efficiency
Comparison": FLUX.1, SD3.5-Large, SANA) and the rollout sizes of its
"Two-Stage Pipeline" section (N = 96 noises per prompt, K = 24 selected).
LoRA rank 32 follows the AI Trends summary of the paper (paragraph on training
stability: "LoRA(rank=32)").

Every generator is a pure function of (config, seed): it uses a private
``torch.Generator`` on the CPU, never the global RNG.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

LORA_RANK = 32
LORA_ALPHA = 32.0  # alpha / r = 1 in every configuration


@dataclass(frozen=True)
class LinearConfig:
    """One DiT linear layer: Y[M,N] = X[M,K] @ W[N,K]^T (+ bias)."""

    name: str
    M: int
    K: int
    N: int
    w_dtype: str = "bf16"          # "bf16" or "fp32"
    w_dist: str = "normal"         # "normal" (std 0.02) or "student_t4" (std 0.02)
    w_outlier_frac: float = 0.0    # fraction of input channels of W scaled up
    w_outlier_gain: float = 1.0
    x_outlier_frac: float = 0.0    # fraction of input channels of X scaled up
    x_outlier_gain: float = 1.0
    description: str = ""


@dataclass(frozen=True)
class RewardConfig:
    """Proxy rewards for P prompts x N seeds; K seeds are kept per prompt."""

    P: int
    N: int
    K: int
    global_std: bool = True


LINEARS = {
    "tiny": LinearConfig(
        "tiny", M=128, K=256, N=256, w_dtype="fp32",
        description="tiny NVFP4 linear: W fp32 [256,256], X bf16 [128,256]"),
    "sana": LinearConfig(
        "sana", M=16384, K=2240, N=2240,
        w_outlier_frac=0.01, w_outlier_gain=20.0,
        x_outlier_frac=0.01, x_outlier_gain=20.0,
        description="SANA-shaped rollout linear: 16 prompts x 1024 latent tokens"),
    "flux_up": LinearConfig(
        "flux_up", M=36864, K=3072, N=12288, w_dist="student_t4",
        x_outlier_frac=0.005, x_outlier_gain=30.0,
        description="FLUX.1-shaped MLP up-projection: 8 images x 4608 tokens"),
    "sd35_qkv": LinearConfig(
        "sd35_qkv", M=35432, K=2432, N=7296, w_dist="student_t4",
        x_outlier_frac=0.005, x_outlier_gain=30.0,
        description="SD3.5-Large-shaped attention QKV: 8 x 4429 tokens"),
    "sd35_mlp": LinearConfig(
        "sd35_mlp", M=35432, K=2432, N=9728, w_dist="student_t4",
        x_outlier_frac=0.005, x_outlier_gain=30.0,
        description="SD3.5-Large-shaped MLP up-projection"),
    "iter_up": LinearConfig(
        "iter_up", M=442368, K=3072, N=12288, w_dist="student_t4",
        x_outlier_frac=0.005, x_outlier_gain=30.0,
        description="iteration-shaped batch, up-projection: 96 rollouts x 4608 tokens"),
    "iter_down": LinearConfig(
        "iter_down", M=442368, K=12288, N=3072, w_dist="student_t4",
        x_outlier_frac=0.005, x_outlier_gain=30.0,
        description="iteration-shaped batch, down-projection"),
}

REWARDS = {
    "tiny": RewardConfig(P=1, N=96, K=24),
    "iter": RewardConfig(P=32, N=96, K=24),
}


def _gen(seed: int, stream: int) -> torch.Generator:
    """A private CPU generator; `stream` separates the tensors of one config."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + int(stream))
    return g


def _outlier_channels(n_channels: int, frac: float, g: torch.Generator) -> torch.Tensor:
    count = int(math.floor(n_channels * frac))
    return torch.randperm(n_channels, generator=g)[:count]


def weight(cfg: LinearConfig, seed: int = 0) -> torch.Tensor:
    """Base weight W [N, K] (fp32 or bf16 per the config), std 0.02."""
    g = _gen(seed, 1)
    if cfg.w_dist == "student_t4":
        # Student-t with 4 degrees of freedom, t = z / sqrt(chi2_4 / 4), built
        # from the private generator (torch.distributions has no generator
        # argument).  Its variance is 2, so scale by 0.02 / sqrt(2) for std 0.02.
        z = torch.randn(cfg.N, cfg.K, generator=g, dtype=torch.float32)
        chi2 = torch.zeros(cfg.N, cfg.K, dtype=torch.float32)
        for _ in range(4):
            e = torch.randn(cfg.N, cfg.K, generator=g, dtype=torch.float32)
            chi2.add_(e * e)
        t = z / torch.sqrt(chi2 / 4.0)
        w = t * (0.02 / math.sqrt(2.0))
    else:
        w = torch.randn(cfg.N, cfg.K, generator=g, dtype=torch.float32) * 0.02
    if cfg.w_outlier_frac > 0:
        ch = _outlier_channels(cfg.K, cfg.w_outlier_frac, _gen(seed, 2))
        w[:, ch] *= cfg.w_outlier_gain
    return w if cfg.w_dtype == "fp32" else w.to(torch.bfloat16)


def lora(cfg: LinearConfig, seed: int = 0, rank: int = LORA_RANK):
    """LoRA factors A [r, K] ~ N(0, (1/32)^2) and B [N, r] ~ N(0, 0.01^2), fp32."""
    A = torch.randn(rank, cfg.K, generator=_gen(seed, 3), dtype=torch.float32) * (1.0 / 32.0)
    B = torch.randn(cfg.N, rank, generator=_gen(seed, 4), dtype=torch.float32) * 0.01
    return A, B


def activations(cfg: LinearConfig, seed: int = 0, rows: int | None = None) -> torch.Tensor:
    """Activations X [M, K] bf16 ~ N(0, 1) with the config's outlier channels."""
    M = cfg.M if rows is None else rows
    x = torch.randn(M, cfg.K, generator=_gen(seed, 5), dtype=torch.float32)
    if cfg.x_outlier_frac > 0:
        ch = _outlier_channels(cfg.K, cfg.x_outlier_frac, _gen(seed, 6))
        x[:, ch] *= cfg.x_outlier_gain
    return x.to(torch.bfloat16)


def bias(cfg: LinearConfig, seed: int = 0) -> torch.Tensor:
    """Bias [N] bf16 ~ N(0, 0.02^2)."""
    return (torch.randn(cfg.N, generator=_gen(seed, 7), dtype=torch.float32) * 0.02).to(torch.bfloat16)


def rewards(cfg: RewardConfig, seed: int = 0) -> torch.Tensor:
    """Proxy rewards [P, N] fp32 ~ N(0, 1)."""
    return torch.randn(cfg.P, cfg.N, generator=_gen(seed, 8), dtype=torch.float32)


def random_nvfp4_operand(rows: int, K: int, seed: int, stream: int,
                         sf_lo: int = 0x20, sf_hi: int = 0x50):
    """Random NVFP4 operand bytes for GEMM-only tests.

    Returns (codes [rows, K/2] uint8, sf [rows, K/16] uint8 row-major logical,
    scale fp32 [rows]).  Codes are uniform over all 16 E2M1 bit patterns; scale
    bytes are uniform over [sf_lo, sf_hi] (finite, positive E4M3 patterns); the
    second-level scales are uniform in [0.5, 2).  Pure random bytes: no encoding
    arithmetic happens here.
    """
    g = _gen(seed, 100 + stream)
    codes = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    sf = torch.randint(sf_lo, sf_hi + 1, (rows, K // 16), generator=g, dtype=torch.int32).to(torch.uint8)
    scale = torch.rand(rows, generator=g, dtype=torch.float32) * 1.5 + 0.5
    return codes, sf, scale


def bf16_bits(t: torch.Tensor):
    """Raw uint16 bit patterns of a bf16 tensor as a numpy array (a view, no arithmetic)."""
    import numpy as np
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def activations_on_device(cfg: LinearConfig, device, seed: int = 0, rows: int | None = None) -> torch.Tensor:
    """Activations with the recipe of activations() (N(0, 1), the config's outlier
    channels scaled) drawn by a seeded generator on `device` instead of the CPU: for
    timing runs at sizes where drawing on the host would take long.  The values differ
    from activations(cfg, seed); nothing compares them with the oracle."""
    M = cfg.M if rows is None else rows
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 1_000_003 + 5)
    x = torch.randn(M, cfg.K, generator=g, dtype=torch.float32, device=device)
    if cfg.x_outlier_frac > 0:
        ch = _outlier_channels(cfg.K, cfg.x_outlier_frac, _gen(seed, 6)).to(device)
        x[:, ch] *= cfg.x_outlier_gain
    return x.to(torch.bfloat16)


@dataclass(frozen=True)
class BlockConfig:
    """A synthetic DiT block: B images of S tokens of width D, H attention heads of
    D/H channels; linears qkv [3D, D], o [D, D], up [4D, D] and dn [D, 4D], each
    with a bias."""

    name: str
    B: int
    S: int
    D: int
    H: int
    description: str = ""


BLOCKS = {
    "tiny": BlockConfig("tiny", B=2, S=128, D=256, H=2,
                        description="tiny DiT block: 2 x 128 tokens, D 256, 2 heads"),
    "flux": BlockConfig("flux", B=8, S=4608, D=3072, H=24,
                        description="FLUX.1-shaped DiT block: 8 images x 4608 tokens (4096 latent + "
                                    "512 text), D 3072, 24 heads of 128, MLP 4D"),
}

BLOCK_LINEARS = ("qkv", "o", "up", "dn")


def block_linear_shape(cfg: BlockConfig, name: str):
    """(N, K) of one of the block's linears."""
    D = cfg.D
    return {"qkv": (3 * D, D), "o": (D, D), "up": (4 * D, D), "dn": (D, 4 * D)}[name]


def block_weights(cfg: BlockConfig, seed: int = 0) -> dict:
    """{name: (W [N, K] bf16 ~ N(0, 0.02^2), bias [N] bf16 ~ N(0, 0.02^2))} for the
    block's four linears."""
    out = {}
    for i, name in enumerate(BLOCK_LINEARS):
        N, K = block_linear_shape(cfg, name)
        w = torch.randn(N, K, generator=_gen(seed, 200 + 2 * i), dtype=torch.float32) * 0.02
        b = torch.randn(N, generator=_gen(seed, 201 + 2 * i), dtype=torch.float32) * 0.02
        out[name] = (w.to(torch.bfloat16), b.to(torch.bfloat16))
    return out


def block_input(cfg: BlockConfig, seed: int = 0) -> torch.Tensor:
    """The block's input x [B*S, D] bf16 ~ N(0, 1)."""
    return torch.randn(cfg.B * cfg.S, cfg.D, generator=_gen(seed, 210), dtype=torch.float32).to(torch.bfloat16)
