"""Shared test helpers: seeded synthetic model inputs for the oracle."""
from __future__ import annotations

import numpy as np

import synth
from synth import weight_names, normal_bf16_np, kv_cache_np


class NpWeights:
    """Lazily generated bf16 weights (uint16 codes) of a model, cached."""

    def __init__(self, model, seed: int = 0):
        self.model = model
        self.seed = seed
        self.spec = {n: (shape, mu, sig) for (n, shape, mu, sig) in weight_names(model)}
        self.cache = {}

    def __call__(self, name):
        if name not in self.cache:
            shape, mu, sig = self.spec[name]
            self.cache[name] = normal_bf16_np(name, shape, mu, sig, self.seed)
        return self.cache[name]


def oracle_state(w, seed: int = 0):
    """Initial oracle DecodeState for workload ``w``."""
    from oracle.forward import initial_state
    m = w.model
    cap = w.capacity

    def kv(l, which):
        return kv_cache_np(synth.kv_name(l, which), w.B, m.Hkv, cap, m.D, w.kv_len, seed)
    return initial_state(m, w.B, cap, w.kv_len, synth.prompt_tokens_np(w, seed), kv)


def read_golden(name):
    import os
    p = os.path.join(os.path.dirname(__file__), "golden", name)
    rows = []
    for line in open(p):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        rows.append(line.split())
    return rows
