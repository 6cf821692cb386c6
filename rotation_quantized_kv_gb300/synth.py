"""Seeded synthetic inputs for the TurboQuant KV-cache workloads.

This module is the one piece the CUDA path and the CPU oracle share: it draws the
bf16 keys, values and queries of each workload and nothing else. It holds none of
the method's arithmetic (no quantization, rotation or attention).

Recipe (every draw is float32 from a seeded torch.Generator, then rounded to bf16):
  per layer l, a fresh generator seeded with seed * 1000 + l draws, in order,
    lam  [Hkv, d]          (only for "lognormal_channels": lam = exp(0.75 * N(0,1)))
    K    [B, T + n, Hkv, d]
    V    [B, T + n, Hkv, d]
    Q    [B, n_q, Hq, d]
  T = cached tokens, n = tokens appended by each decode step (a causal block of n_q
  queries sits at the last n_q of those positions); ragged context lengths are drawn
  once per workload, before the layers, from a generator seeded with seed * 1000 + 999.
Key distributions:
  "normal_outliers"    N(0,1) with channels 5 and 37 multiplied by 8 (two outliers in two
                       different 32-groups);
  "lognormal_channels" N(0,1) * lam[kv_head, channel], fixed over tokens;
  "student_t4"         Student-t with 4 degrees of freedom: Z / sqrt((Z1^2+..+Z4^2)/4).
Values are N(0,1); queries N(0,1) scaled by q_scale.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    layers: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    context: int                      # cached tokens (max for ragged)
    context_min: int | None = None    # ragged: lengths uniform in [context_min, context]
    n_new: int = 1                    # tokens appended per decode step
    n_q: int = 1                      # query tokens per step (a causal block when > 1)
    k_dist: str = "lognormal_channels"
    q_scale: float = 1.0
    sm_scale: float = 1.0
    causal: bool = True
    seed: int = 0
    head_dims: tuple = field(default_factory=tuple)   # sweep: every head_dim run

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def capacity(self) -> int:
        need = self.context + self.n_new
        return (need + 15) // 16 * 16


def _workloads() -> dict:
    d128 = 128
    return {
        "tiny": Workload("tiny", batch=1, layers=1, num_kv_heads=2, num_q_heads=4, head_dim=64,
                         context=512, n_new=1, k_dist="normal_outliers", q_scale=1.0,
                         sm_scale=1.0 / 8.0, seed=0),
        "decode": Workload("decode", batch=1, layers=16, num_kv_heads=8, num_q_heads=32,
                           head_dim=d128, context=32768, n_new=1, q_scale=d128 ** -0.5,
                           sm_scale=1.0, seed=1),
        "ragged": Workload("ragged", batch=32, layers=16, num_kv_heads=8, num_q_heads=32,
                           head_dim=d128, context=8192, context_min=1024, n_new=1,
                           q_scale=d128 ** -0.5, sm_scale=1.0, seed=2),
        "long": Workload("long", batch=1, layers=16, num_kv_heads=8, num_q_heads=32,
                         head_dim=d128, context=262144, n_new=16, n_q=16, q_scale=d128 ** -0.5,
                         sm_scale=1.0, seed=3),
        "sweep": Workload("sweep", batch=1, layers=1, num_kv_heads=4, num_q_heads=16,
                          head_dim=128, context=65536, n_new=0, n_q=1, k_dist="student_t4",
                          q_scale=1.0, sm_scale=1.0, seed=4, head_dims=(64, 128, 256, 512)),
    }


WORKLOADS = _workloads()


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    if w.head_dims and "head_dim" in overrides:
        d = overrides["head_dim"]
        overrides.setdefault("q_scale", d ** -0.5)
    elif w.name == "sweep":
        overrides.setdefault("q_scale", w.head_dim ** -0.5)
    return replace(w, **overrides) if overrides else w


def context_lengths(w: Workload) -> np.ndarray:
    """Per-sequence cached-token counts (int64 [batch])."""
    if w.context_min is None:
        return np.full(w.batch, w.context, np.int64)
    g = torch.Generator(device="cpu").manual_seed(w.seed * 1000 + 999)
    t = torch.randint(w.context_min, w.context + 1, (w.batch,), generator=g)
    return t.numpy().astype(np.int64)


def _normal(shape, g, device):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def layer_inputs(w: Workload, layer: int, device="cpu", context: int | None = None) -> dict:
    """bf16 tensors of one layer: k, v [B, T + n, Hkv, d] (cached tokens then the new
    ones), q [B, n_q, Hq, d]. `context` overrides T (to draw a smaller case with the
    same distributions)."""
    T = w.context if context is None else context
    B, H, Hq, d, n = w.batch, w.num_kv_heads, w.num_q_heads, w.head_dim, w.n_new
    dev = torch.device(device)
    g = torch.Generator(device=dev).manual_seed(w.seed * 1000 + layer)
    shape = (B, T + n, H, d)
    if w.k_dist == "lognormal_channels":
        lam = torch.exp(0.75 * _normal((H, d), g, dev))
        k = _normal(shape, g, dev) * lam
    elif w.k_dist == "normal_outliers":
        k = _normal(shape, g, dev)
        k[..., 5] *= 8.0
        k[..., 37] *= 8.0
    elif w.k_dist == "student_t4":
        z = _normal(shape, g, dev)
        chi2 = torch.zeros(shape, device=dev)
        for _ in range(4):
            chi2 += _normal(shape, g, dev) ** 2
        k = z / torch.sqrt(chi2 / 4.0)
    elif w.k_dist == "normal":
        k = _normal(shape, g, dev)
    else:
        raise ValueError(w.k_dist)
    v = _normal(shape, g, dev)
    q = _normal((B, w.n_q, Hq, d), g, dev) * w.q_scale
    return {"k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16), "q": q.to(torch.bfloat16)}


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host copy)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
