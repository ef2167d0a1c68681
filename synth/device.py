"""Seeded workload inputs materialised as torch tensors (on any device).

Same values as the numpy generators the oracle uses; shapes follow
``configs``.  No arithmetic of the decode method here.
"""
from __future__ import annotations

import torch

from .configs import Workload, weight_names
from .generate import (normal_bf16_torch, kv_cache_torch, uniform_ints_torch, normal_bf16_np, kv_cache_np,
                       uniform_ints_np)


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


def host_inputs(w: Workload, seed: int = 0):
    """The inputs of ``device_inputs`` generated on the host with the numpy
    generators (same values): weights as uint16 bf16 codes by name, per-layer
    K/V caches [B, Hkv, cap, D] uint16, history int32 [B, cap], state int32
    [B, 2]."""
    import numpy as np
    m = w.model
    cap = w.capacity
    weights = {n: normal_bf16_np(n, shape, mu, sig, seed) for (n, shape, mu, sig) in weight_names(m)}
    kc = [kv_cache_np(kv_name(l, "k"), w.B, m.Hkv, cap, m.D, w.kv_len, seed) for l in range(m.L)]
    vc = [kv_cache_np(kv_name(l, "v"), w.B, m.Hkv, cap, m.D, w.kv_len, seed) for l in range(m.L)]
    tok = uniform_ints_np("prompt_token", w.B, 0, m.V, seed).astype(np.int32)
    pos = np.asarray(w.kv_len, dtype=np.int32)
    state = np.stack([tok, pos], axis=1).astype(np.int32)
    hist = np.zeros((w.B, cap), dtype=np.int32)
    hist[np.arange(w.B), pos] = tok
    return weights, kc, vc, hist, state


def to_device(host, device="cuda"):
    """Copy ``host_inputs``' arrays to ``device`` once: the same structure as
    ``device_inputs`` returns (bf16 weights and caches, int32 history and
    state)."""
    weights, kc, vc, hist, state = host

    def bf16(a):
        return torch.from_numpy(a.view("int16")).to(device).view(torch.bfloat16)

    return ({n: bf16(a) for n, a in weights.items()}, [bf16(a) for a in kc], [bf16(a) for a in vc],
            torch.from_numpy(hist).to(device), torch.from_numpy(state).to(device))
