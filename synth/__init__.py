"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

Holds shapes and random-number generation only; none of the decode
method's arithmetic.
"""
from .configs import (ModelShape, Workload, TINY, LLAMA_1B, LLAMA_8B, WORKLOADS,
                      workload, custom, weight_names)
from .generate import (normal_bf16_np, normal_bf16_np_at, normal_bf16_torch,
                       kv_cache_np, kv_cache_torch, uniform_ints_np,
                       uniform_ints_torch, f32_to_bf16_bits_np, normal_table_f32)


def prompt_tokens_np(w: Workload, seed: int = 0):
    return uniform_ints_np("prompt_token", w.B, 0, w.model.V, seed)


def prompt_tokens_torch(w: Workload, seed: int = 0, device="cpu"):
    return uniform_ints_torch("prompt_token", w.B, 0, w.model.V, seed, device)


from .device import kv_name, device_inputs, host_inputs, to_device  # noqa: E402


__all__ = [n for n in dir() if not n.startswith("_")]
