"""Seeded workload inputs materialised as torch tensors (on any device).

Same values as the numpy generators the oracle uses; shapes follow
``configs``.  No arithmetic of the decode method here.
"""
from __future__ import annotations

import torch

from .configs import Workload, weight_names
from .generate import normal_bf16_torch, kv_cache_torch, uniform_ints_torch


def kv_name(layer: int, which: str) -> str:
    return f"layer{layer}.{which}_cache"


def device_inputs(w: Workload, seed: int = 0, device="cuda", layers=None):
    """weights (name -> bf16 tensor), per-layer K/V caches [B, Hkv, cap, D],
    history int32 [B, cap] and the initial state int32 [B, 2] (token, pos)."""
    m = w.model
    cap = w.capacity
    weights = {}
    for (n, shape, mu, sig) in weight_names(m):
        weights[n] = normal_bf16_torch(n, shape, mu, sig, seed, device=device)
    L = m.L if layers is None else layers
    kc = [kv_cache_torch(kv_name(l, "k"), w.B, m.Hkv, cap, m.D, w.kv_len, seed, device=device) for l in range(L)]
    vc = [kv_cache_torch(kv_name(l, "v"), w.B, m.Hkv, cap, m.D, w.kv_len, seed, device=device) for l in range(L)]
    tok = uniform_ints_torch("prompt_token", w.B, 0, m.V, seed, device=device).to(torch.int32)
    pos = torch.tensor(w.kv_len, dtype=torch.int32, device=device)
    state = torch.stack([tok, pos], dim=1).contiguous()
    hist = torch.zeros(w.B, cap, dtype=torch.int32, device=device)
    hist[torch.arange(w.B, device=device), pos.long()] = tok
    return weights, kc, vc, hist, state
