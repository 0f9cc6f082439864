"""Seeded synthetic inputs for the five workloads of the FP8 linear layer.

This module only draws random numbers: it holds none of the layer's
arithmetic, and both the CUDA path and the CPU oracle take their inputs from
it. Every tensor is drawn in fp32 from a seeded torch CPU generator (numpy's
seeded generator for the expert-count Dirichlet) and rounded to BF16.

Workloads (shapes and distributions):
  tiny      X 128x512, W 512x256, both N(0,1).
  dense     X 4096x7168 N(0,1) with 0.1% of entries replaced by outliers of
            magnitude U(50,200) and random sign; W 7168x2048 N(0, 0.02^2).
  backward  dY 4096x2048 N(0, 1e-3^2); X and W as in ``dense``.
  moe       32 experts, 8192 routed token rows split by counts drawn from
            Dirichlet(0.5) then Multinomial(8192); W_up 32x7168x4096 and
            W_down 32x2048x7168 N(0, 0.02^2); X 8192x7168 N(0,1); the down
            projection input A 8192x2048 N(0,1); dY of the down projection
            8192x7168 N(0, 1e-3^2).
  longk     X 256xK and W Kx256, U(0.5, 1.5), K in {1024, 4096, 16384, 65536};
            a 16384x16384 N(0,1) tensor for the standalone 1x128 quantizer.

Sizes are parameters so that the tests can draw the same distributions at
sizes the oracle finishes in seconds.
"""
from __future__ import annotations

import numpy as np
import torch

OUTLIER_FRACTION = 1e-3
W_STD = 0.02
DY_STD = 1e-3
LONGK_VALUES = (1024, 4096, 16384, 65536)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float = 1.0, seed: int = 0) -> torch.Tensor:
    """BF16 tensor of i.i.d. N(0, std^2) values (drawn in fp32, then rounded)."""
    t = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def uniform(shape, lo: float, hi: float, seed: int = 0) -> torch.Tensor:
    t = torch.rand(*shape, generator=_gen(seed), dtype=torch.float32)
    return (t * (hi - lo) + lo).to(torch.bfloat16)


def with_outliers(shape, fraction: float = OUTLIER_FRACTION, lo: float = 50.0,
                  hi: float = 200.0, seed: int = 0) -> torch.Tensor:
    """N(0,1) BF16 tensor where round(fraction * numel) entries, at positions
    from a seeded permutation, are replaced by +-U(lo, hi)."""
    g = _gen(seed)
    t = torch.randn(*shape, generator=g, dtype=torch.float32)
    n = t.numel()
    count = int(round(fraction * n))
    if count:
        pos = torch.randperm(n, generator=g)[:count]
        mag = torch.rand(count, generator=g) * (hi - lo) + lo
        sign = torch.where(torch.rand(count, generator=g) < 0.5, -1.0, 1.0)
        t.view(-1)[pos] = mag * sign
    return t.to(torch.bfloat16)


def expert_counts(tokens: int = 8192, experts: int = 32, alpha: float = 0.5,
                  seed: int = 0) -> np.ndarray:
    """Per-expert token counts: p ~ Dirichlet(alpha), counts ~ Multinomial(tokens, p)."""
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(experts, alpha))
    return rng.multinomial(tokens, p).astype(np.int64)


def offsets_from_counts(counts) -> np.ndarray:
    off = np.zeros(len(counts) + 1, np.int32)
    off[1:] = np.cumsum(np.asarray(counts, np.int64))
    return off


def bits(t: torch.Tensor) -> np.ndarray:
    """numpy uint16 view of a CPU BF16 tensor's bit patterns."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny(M: int = 128, K: int = 512, N: int = 256, seed: int = 0):
    return {"X": normal((M, K), seed=seed), "W": normal((K, N), seed=seed + 1)}


def dense(M: int = 4096, K: int = 7168, N: int = 2048, seed: int = 0):
    return {"X": with_outliers((M, K), seed=seed),
            "W": normal((K, N), std=W_STD, seed=seed + 1)}


def backward(M: int = 4096, K: int = 7168, N: int = 2048, seed: int = 0):
    d = dense(M, K, N, seed)
    d["dY"] = normal((M, N), std=DY_STD, seed=seed + 2)
    return d


def moe(tokens: int = 8192, experts: int = 32, hidden: int = 7168, inter: int = 2048,
        up: int = 4096, seed: int = 0, with_weights: bool = True):
    """MoE expert GEMM inputs. W_up_e is [hidden x up], W_down_e [inter x hidden]."""
    counts = expert_counts(tokens, experts, seed=seed)
    d = {"counts": counts, "offsets": offsets_from_counts(counts),
         "X": normal((tokens, hidden), seed=seed + 10),
         "A": normal((tokens, inter), seed=seed + 11),
         "dY": normal((tokens, hidden), std=DY_STD, seed=seed + 12)}
    if with_weights:
        d["W_up"] = normal((experts, hidden, up), std=W_STD, seed=seed + 13)
        d["W_down"] = normal((experts, inter, hidden), std=W_STD, seed=seed + 14)
    return d


def longk(K: int, M: int = 256, N: int = 256, seed: int = 0):
    return {"X": uniform((M, K), 0.5, 1.5, seed=seed),
            "W": uniform((K, N), 0.5, 1.5, seed=seed + 1)}


def quant_stream(R: int = 16384, C: int = 16384, seed: int = 0):
    return {"X": normal((R, C), seed=seed)}
