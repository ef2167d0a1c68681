"""Model and workload shapes for the synthetic decode workloads.

Shapes only: no arithmetic of the decode method lives here.  Both the CUDA
path (through the Python binding and ``bench.py``) and the CPU oracle read
these tables, so the two sides always agree on what a workload is.

The five workloads are the Llama-style decoders that the decode-megakernel
pages measure or imply ("mega kernel initial", 1y33.com, results table:
Llama-3.2-1B-Instruct, batch 1) plus a tiny two-layer model for fast parity,
an 8B-shaped model, a ragged batch of 8 and a long-context batch of 4.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass(frozen=True)
class ModelShape:
    name: str
    L: int          # decoder layers
    H: int          # hidden size
    Hq: int         # query heads
    Hkv: int        # key/value heads
    D: int          # head dim
    F: int          # SwiGLU FFN size
    V: int          # vocabulary
    tied: bool      # lm_head shares the embedding table
    theta: float    # RoPE base
    eps: float = 1e-5

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_qkv(self) -> int:
        return (self.Hq + 2 * self.Hkv) * self.D

    def streamed_params(self) -> int:
        """bf16 parameters a decode step streams once (the embedding table
        is gathered by row, not streamed; a tied lm_head streams the table)."""
        per_layer = (self.n_qkv * self.H + self.H * self.Hq * self.D
                     + 2 * self.F * self.H + self.H * self.F + 2 * self.H)
        return self.L * per_layer + self.H + self.V * self.H


@dataclass(frozen=True)
class Workload:
    name: str
    model: ModelShape
    B: int
    kv_len: tuple          # per-sequence cached length before the first step
    steps: int
    chunk: int = 0         # split-KV chunk in keys; 0 = automatic
    ragged: bool = False   # kv_len drawn per sequence from the generator

    @property
    def capacity(self) -> int:
        return max(self.kv_len) + self.steps + 1


TINY = ModelShape("tiny", L=2, H=256, Hq=4, Hkv=2, D=64, F=512, V=1024,
                  tied=False, theta=1e4)
LLAMA_1B = ModelShape("llama-3.2-1b-shaped", L=16, H=2048, Hq=32, Hkv=8, D=64,
                      F=8192, V=128256, tied=True, theta=5e5)
LLAMA_8B = ModelShape("llama-3-8b-shaped", L=32, H=4096, Hq=32, Hkv=8, D=128,
                      F=14336, V=128256, tied=False, theta=5e5)

RAGGED_LO, RAGGED_HI = 512, 8192


def _ragged_lengths(B: int, seed: int) -> tuple:
    from .generate import uniform_ints_np
    v = uniform_ints_np("ragged_kv_len", B, RAGGED_LO, RAGGED_HI + 1, seed)
    return tuple(int(x) for x in v)


def workload(name: str, seed: int = 0) -> Workload:
    """The named workload.  ``seed`` only changes the ragged lengths."""
    if name == "tiny":
        return Workload("tiny", TINY, 1, (128,), 1)
    if name == "1b":
        return Workload("1b", LLAMA_1B, 1, (1024,), 128)
    if name == "8b":
        return Workload("8b", LLAMA_8B, 1, (4096,), 64)
    if name == "8b_b8":
        return Workload("8b_b8", LLAMA_8B, 8, _ragged_lengths(8, seed), 64,
                        ragged=True)
    if name == "8b_long":
        return Workload("8b_long", LLAMA_8B, 4, (32768,) * 4, 16, chunk=1024)
    raise KeyError(name)


WORKLOADS = ("tiny", "1b", "8b", "8b_b8", "8b_long")


def custom(model: ModelShape, B: int, kv_len, steps: int, chunk: int = 0,
           name: str = "custom") -> Workload:
    kv = tuple(int(x) for x in kv_len) if hasattr(kv_len, "__len__") else (int(kv_len),) * B
    assert len(kv) == B
    return Workload(name, model, B, kv, steps, chunk)


def weight_names(m: ModelShape) -> list:
    """(name, shape, mu, sigma) of every weight tensor, in registration order."""
    out = [("embed", (m.V, m.H), 0.0, 0.02)]
    for l in range(m.L):
        out += [
            (f"layer{l}.attn_norm", (m.H,), 1.0, 0.02),
            (f"layer{l}.wqkv", (m.n_qkv, m.H), 0.0, 0.02),
            (f"layer{l}.wo", (m.H, m.Hq * m.D), 0.0, 0.02),
            (f"layer{l}.mlp_norm", (m.H,), 1.0, 0.02),
            (f"layer{l}.wgu", (2 * m.F, m.H), 0.0, 0.02),
            (f"layer{l}.wd", (m.H, m.F), 0.0, 0.02),
        ]
    out.append(("final_norm", (m.H,), 1.0, 0.02))
    if not m.tied:
        out.append(("lm_head", (m.V, m.H), 0.0, 0.02))
    return out
