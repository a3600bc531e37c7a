"""Seeded synthetic inputs for KDA prefill workloads.

This module is shared by the tests, the benchmark and the smoke check, on
both sides of the parity comparison. It holds none of the method's
arithmetic: it only draws random tensors with the shapes, value ranges and
length mix of the workloads the TPU report measures (T=8192 as 4x2048,
H=16, K=V=128, bf16 q/k/v; batches B in {1..64}; cached-prefix prefill with
a nonzero initial state).

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in this
order):
  1. sequence lengths, when random: ``rint(lognormal(ln 512, 1.0))`` clipped
     to [64, 8192] — a stand-in for the report's ShareGPT-derived length
     distribution, which is not available here;
  2. q, k ~ N(0,1), each (token, head) row L2-normalised, cast to bf16;
  3. v ~ N(0,1), cast to bf16;
  4. beta = sigmoid(N(0,1)), fp32;
  5. g = lower_bound * sigmoid(N(0, sigma_g)), fp32 per key channel, so
     lower_bound <= g <= 0;
  6. initial_state ~ N(0, state_std), fp32 [N,H,K,V], when requested.
Draws are float32 (``Generator.standard_normal(dtype=float32)``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

HEAD_DIM = 128


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seqlens: Optional[tuple]          # fixed lengths, or None to draw them
    num_seqs: int                     # used when seqlens is None
    num_heads: int
    seed: int
    sigma_g: float = 1.0
    state_std: Optional[float] = None  # None: no initial state (zeros)
    lower_bound: float = -5.0
    kind: str = "prefill"             # "decode": every sequence has the same few tokens

    def describe(self) -> dict:
        return dataclasses.asdict(self)


def _lognormal_lengths(rng, n: int) -> List[int]:
    x = rng.lognormal(math.log(512.0), 1.0, n)
    return [int(v) for v in np.clip(np.rint(x), 64, 8192)]


def workloads() -> dict:
    """The named workloads (tiny, headline, cached-prefix, batch sweep, wide, long;
    decode steps)."""
    w = {
        "tiny_T256_H2": Workload("tiny_T256_H2", (256,), 1, 2, seed=0),
        "headline_4x2048_H16": Workload("headline_4x2048_H16", (2048,) * 4, 4, 16, seed=1),
        "cached_prefix_B16_H16": Workload("cached_prefix_B16_H16", None, 16, 16, seed=2,
                                          state_std=0.02),
        "wide_1x16384_H96": Workload("wide_1x16384_H96", (16384,), 1, 96, seed=4,
                                     sigma_g=2.0, state_std=0.02),
        "wide_3x8192_H96": Workload("wide_3x8192_H96", (8192,) * 3, 3, 96, seed=4,
                                    sigma_g=2.0, state_std=0.02),
    }
    for b in (1, 2, 4, 8, 16, 32, 64):
        w[f"sweep_B{b}_H16"] = Workload(f"sweep_B{b}_H16", None, b, 16, seed=b)
    # one long sequence with the few heads one GPU holds under head-parallel
    # sharding: few, long chains (the split-sequence scan's case)
    w["long_1x65536_H4"] = Workload("long_1x65536_H4", (65536,), 1, 4, seed=5, state_std=0.02)
    # decode steps: one new token per sequence on a carried state
    w["decode_B256_H16"] = Workload("decode_B256_H16", (1,) * 256, 256, 16, seed=9, state_std=0.02, kind="decode")
    w["decode_B64x4_H16"] = Workload("decode_B64x4_H16", (4,) * 64, 64, 16, seed=10, state_std=0.02, kind="decode")
    return w


def seqlens_for(wl: Workload) -> List[int]:
    if wl.seqlens is not None:
        return list(wl.seqlens)
    return _lognormal_lengths(np.random.default_rng(wl.seed), wl.num_seqs)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / np.maximum(n, 1e-30)).astype(np.float32)


def make_inputs(seqlens, num_heads: int, seed: int, sigma_g: float = 1.0,
                state_std: Optional[float] = None, lower_bound: float = -5.0,
                rng: Optional[np.random.Generator] = None, head_dim: int = HEAD_DIM) -> dict:
    """Draw one batch. Returns CPU torch tensors: q, k, v bf16 [T,H,D]; g fp32
    [T,H,D]; beta fp32 [T,H]; cu_seqlens int32 [N+1]; initial_state fp32
    [N,H,D,D] or None; plus scale, lower_bound and seqlens."""
    if rng is None:
        rng = np.random.default_rng(seed)
    seqlens = [int(s) for s in seqlens]
    T, H, D, N = sum(seqlens), num_heads, head_dim, len(seqlens)
    f32 = np.float32
    q = _unit_rows(rng.standard_normal((T, H, D), dtype=f32))
    k = _unit_rows(rng.standard_normal((T, H, D), dtype=f32))
    v = rng.standard_normal((T, H, D), dtype=f32)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H), dtype=f32)))
    z = rng.standard_normal((T, H, D), dtype=f32) * f32(sigma_g)
    g = f32(lower_bound) * (1.0 / (1.0 + np.exp(-z)))
    s0 = None
    if state_std is not None:
        s0 = rng.standard_normal((N, H, D, D), dtype=f32) * f32(state_std)
    cu = np.zeros(N + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    return {
        "q": torch.from_numpy(q).to(torch.bfloat16),
        "k": torch.from_numpy(k).to(torch.bfloat16),
        "v": torch.from_numpy(v).to(torch.bfloat16),
        "g": torch.from_numpy(np.ascontiguousarray(g, dtype=f32)),
        "beta": torch.from_numpy(np.ascontiguousarray(beta, dtype=f32)),
        "cu_seqlens": torch.from_numpy(cu),
        "initial_state": None if s0 is None else torch.from_numpy(s0),
        "scale": float(D) ** -0.5,
        "lower_bound": float(lower_bound),
        "seqlens": seqlens,
    }


def make_norm_inputs(total_tokens: int, num_heads: int, seed: int, head_dim: int = HEAD_DIM) -> dict:
    """The extra inputs of the fused gated RMSNorm of o: the output-gate
    projection gate ~ N(0, 1.5^2) as bf16 [T,H,D], a per-channel weight
    1 + N(0, 0.2^2) as fp32 [D], and eps = 1e-5. CPU torch tensors."""
    rng = np.random.default_rng(seed)
    gate = rng.standard_normal((total_tokens, num_heads, head_dim), dtype=np.float32) * np.float32(1.5)
    weight = np.float32(1.0) + rng.standard_normal(head_dim, dtype=np.float32) * np.float32(0.2)
    return {"gate": torch.from_numpy(gate).to(torch.bfloat16), "weight": torch.from_numpy(weight), "eps": 1e-5}


def make_workload(wl: Workload) -> dict:
    rng = np.random.default_rng(wl.seed)
    if wl.seqlens is None:
        lens = _lognormal_lengths(rng, wl.num_seqs)
    else:
        lens = list(wl.seqlens)
    return make_inputs(lens, wl.num_heads, wl.seed, sigma_g=wl.sigma_g,
                       state_std=wl.state_std, lower_bound=wl.lower_bound, rng=rng)


def to_f64(x: Optional[torch.Tensor]):
    """Exact upcast to a float64 numpy array (bf16 and fp32 embed in fp64)."""
    if x is None:
        return None
    return x.detach().to("cpu", torch.float64).numpy()
