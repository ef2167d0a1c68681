"""A Llama-style dense decoder composed on the graph object, one decode step.

Per layer (the decoder-layer listing of "mega kernel initial", 1y33.com):
qkv GEMV with the attention RMSNorm fused on its input, attention
(RoPE-append, split-KV partials, combine), o_proj with the residual
epilogue, gate_up with the MLP RMSNorm fused and SiLU*mul, down with the
residual; then the lm_head GEMV with the final RMSNorm fused and per-tile
argmax, and SAMPLE.  Weights are registered first, then the KV caches and
the token history, then activations as the ops allocate them (the buffer
order the oracle's graph spec uses too).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from .graph import Graph, Buf


@dataclass
class LlamaDecode:
    graph: Graph
    names: dict = field(default_factory=dict)   # weight / cache name -> Buf
    hidden: list = field(default_factory=list)  # per-layer output Buf
    logits: Buf = None
    pairs: Buf = None
    history: Buf = None
    kcache: list = field(default_factory=list)
    vcache: list = field(default_factory=list)
    fused_norms: int = 0                        # norms folded by the fusion pass
    tokens: Buf = None                          # chunk steps: int32 [B, T] input tokens


def build_llama_decode(model, B: int, len0, capacity: int, weights: dict, kcache: list, vcache: list,
                       history: torch.Tensor, chunk: int = 0, device="cuda", num_ctas: int = 0,
                       tiles_target: int = 0, col_align: int = 4, wait_timeout_us: int = 0,
                       norms: str = "fused", T: int = 1) -> LlamaDecode:
    """weights: name -> bf16 tensor (names of synth.weight_names);
    kcache/vcache: per layer bf16 [B, Hkv, capacity, D]; history int32 [B, capacity].
    norms: "fused" (RMS_NORM_INPUT on the consuming GEMVs), "standalone"
    (RMSNORM tasks), or "fuse_pass" (standalone norms folded by the fusion pass).
    T > 1: every step is a chunk step of T tokens per sequence (their
    activations are rows s * T + t); the caller writes tokens 1..T-1 into
    ``tokens`` before each step."""
    assert norms in ("fused", "standalone", "fuse_pass")
    m = model
    g = Graph(B, device=device, num_ctas=num_ctas, tiles_target=tiles_target, col_align=col_align,
              wait_timeout_us=wait_timeout_us)
    out = LlamaDecode(graph=g)
    W = out.names

    def reg(name, t, rows=None, cols=None):
        W[name] = g.register(t, rows, cols)
        return W[name]

    reg("embed", weights["embed"])
    for l in range(m.L):
        for nm in ("attn_norm", "wqkv", "wo", "mlp_norm", "wgu", "wd"):
            t = weights[f"layer{l}.{nm}"]
            reg(f"layer{l}.{nm}", t, *((1, t.numel()) if t.dim() == 1 else (None, None)))
    t = weights["final_norm"]
    reg("final_norm", t, 1, t.numel())
    lm = W["embed"] if m.tied else reg("lm_head", weights["lm_head"])
    for l in range(m.L):
        out.kcache.append(reg(f"layer{l}.k_cache", kcache[l], B * m.Hkv, capacity * m.D))
        out.vcache.append(reg(f"layer{l}.v_cache", vcache[l], B * m.Hkv, capacity * m.D))
    out.history = reg("history", history)
    if T > 1:
        out.tokens = g.set_chunk(T)

    def normed(x, gamma):
        """(input, gamma kwarg) of a GEMV that reads RMSNorm(x) * gamma."""
        if norms == "fused":
            return x, gamma
        return g.rmsnorm(x, gamma, eps=m.eps), None

    h = g.embed(W["embed"])
    for l in range(m.L):
        x, gm = normed(h, W[f"layer{l}.attn_norm"])
        qkv = g.matmul(x, W[f"layer{l}.wqkv"], gamma=gm, eps=m.eps)
        att = g.attention(qkv, out.kcache[l], out.vcache[l], m.Hq, m.Hkv, m.D, capacity, len0, chunk,
                          m.theta)
        h1 = g.matmul(att, W[f"layer{l}.wo"], residual=h)
        x, gm = normed(h1, W[f"layer{l}.mlp_norm"])
        gu = g.matmul(x, W[f"layer{l}.wgu"], gamma=gm, silu_mul=True, eps=m.eps)
        h = g.matmul(gu, W[f"layer{l}.wd"], residual=h1)
        out.hidden.append(h)
    x, gm = normed(h, W["final_norm"])
    out.logits, out.pairs = g.matmul(x, lm, gamma=gm, eps=m.eps, argmax=True)
    g.sample(out.pairs, out.history, m.V, capacity)
    if norms == "fuse_pass":
        out.fused_norms = g.fuse_rmsnorm()
    return out
