"""Seeded synthetic inputs for the gate-aggregation path.

This module only draws random numbers and rounds them to the requested storage
type.  It contains none of the method's arithmetic, so it can feed both the CUDA
path and the CPU oracle without coupling them.

Recipe (fixed, so every caller sees the same values for the same seed):
  * generator: ``numpy.random.default_rng(seed)`` (PCG64), float32 standard normals
    drawn in a fixed order per helper;
  * rounding to bf16 is round-to-nearest-even (torch's float32 -> bfloat16 cast);
  * aggregation-only inputs: q, k, g, v ~ N(0, 1), each [B, T, width];
  * block inputs: h ~ N(0, 1) [B, T, d], then W_q, W_k [dqk, d], W_g, W_v [m, d],
    W_o [d, m] ~ N(0, 1/fan_in), RMSNorm gain = 1;
  * model inputs: token ids uniform over [0, vocab), tied embedding N(0, 0.02^2);
  * backward inputs: the upstream gradient dout ~ N(0, 1) [B, T, m], from its own
    generator default_rng(seed).
"""
from __future__ import annotations

import numpy as np
import torch

_TORCH_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f64": torch.float64}


def _normal(rng: np.random.Generator, shape, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return x


def cast(x: np.ndarray, dtype: str) -> torch.Tensor:
    """float32 numpy -> CPU torch tensor of the storage dtype ("f32", "bf16", "f64")."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(_TORCH_DT[dtype])


def oracle_view(t: torch.Tensor) -> np.ndarray:
    """CPU tensor -> numpy array the oracle accepts (bf16 as raw uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def agg_inputs(B: int, T: int, dqk: int, m: int, seed: int = 0, dtype: str = "bf16",
               g_scale: float = 1.0):
    """q, k [B, T, dqk] and g, v [B, T, m] ~ N(0, 1), drawn in the order q, k, g, v."""
    rng = np.random.default_rng(seed)
    q = cast(_normal(rng, (B, T, dqk)), dtype)
    k = cast(_normal(rng, (B, T, dqk)), dtype)
    g = cast(_normal(rng, (B, T, m), g_scale), dtype)
    v = cast(_normal(rng, (B, T, m)), dtype)
    return q, k, g, v


def upstream_grad(B: int, T: int, m: int, seed: int = 0, dtype: str = "bf16"):
    """dout ~ N(0, 1) [B, T, m]: the gradient of a loss with respect to an aggregation output."""
    rng = np.random.default_rng(seed)
    return cast(_normal(rng, (B, T, m)), dtype)


def block_inputs(B: int, T: int, d: int, dqk: int, m: int, seed: int = 0, dtype: str = "bf16"):
    """h and one block's weights, drawn in the order h, W_q, W_k, W_g, W_v, W_o."""
    rng = np.random.default_rng(seed)
    h = cast(_normal(rng, (B, T, d)), dtype)
    w = {
        "Wq": cast(_normal(rng, (dqk, d), d ** -0.5), dtype),
        "Wk": cast(_normal(rng, (dqk, d), d ** -0.5), dtype),
        "Wg": cast(_normal(rng, (m, d), d ** -0.5), dtype),
        "Wv": cast(_normal(rng, (m, d), d ** -0.5), dtype),
        "Wo": cast(_normal(rng, (d, m), m ** -0.5), dtype),
        "gamma": cast(np.ones(d, dtype=np.float32), dtype),
    }
    return h, w


def gated_set(d: int, m: int, rng_seed: int, dtype: str = "bf16"):
    """One extra gated-projection set (W_g, W_v, W_o) drawn in that order."""
    rng = np.random.default_rng(rng_seed)
    return {
        "Wg": cast(_normal(rng, (m, d), d ** -0.5), dtype),
        "Wv": cast(_normal(rng, (m, d), d ** -0.5), dtype),
        "Wo": cast(_normal(rng, (d, m), m ** -0.5), dtype),
    }


def model_inputs(B: int, T: int, d: int, vocab: int, seed: int = 0, dtype: str = "bf16"):
    """Token ids [B, T] (int64, uniform) and the tied embedding [vocab, d] ~ N(0, 0.02^2)."""
    rng = np.random.default_rng(seed)
    ids = torch.from_numpy(rng.integers(0, vocab, size=(B, T), dtype=np.int64))
    E = cast(_normal(rng, (vocab, d), 0.02), dtype)
    return ids, E


def random_rows(B: int, T: int, n: int, seed: int, extra=()) -> np.ndarray:
    """Sorted unique flat row indices b*T+i: the given extras plus n uniform draws."""
    rng = np.random.default_rng(seed)
    draws = rng.integers(0, B * T, size=n, dtype=np.int64)
    rows = np.unique(np.concatenate([np.asarray(list(extra), dtype=np.int64), draws]))
    return rows[(rows >= 0) & (rows < B * T)]
