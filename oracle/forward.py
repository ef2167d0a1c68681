"""CPU oracle: one greedy decode step of a Llama-style dense decoder, in float64.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import this module.  It shares no code
with the CUDA path and never calls it.

What is computed.  The decode megakernel ("mega kernel initial", 1y33.com,
its graph-building part) writes a decoder layer as five graph ops: a qkv
projection of the RMS-normalised residual stream, attention over the KV
cache (RoPE, append, split-KV), an output projection added to the residual,
a gate/up projection of the normalised stream with SiLU(gate) * up, and a
down projection added to the residual; the final
RMSNorm fused into the lm_head GEMV and a SAMPLE task taking the argmax over
the vocabulary (its OpId table).  Split-KV flash decoding, the fused
epilogues and the column tiling reach exactly (up to floating-point
re-association) the plain result of a standard Llama decoder layer.  So the
forward below is that plain definition, one operation after another, with
no tiling, chunking or fusion: attention is a single softmax over every
cached key.  The split-KV partial/combine pair is given separately
(``attention_partial`` / ``attention_combine``) so tests can pin the
identity that the megakernel relies on.

Number formats.  Weights, norm gains and the KV cache are bf16 data
(carried as uint16 codes and widened exactly).  Everything else is float64.
The one place where the method itself quantises is the append of the new
key/value row into the bf16 cache; that rounding is taken on the float32
value (float64 -> float32 -> bf16, round to nearest even), the precision the
kernel rounds in, and the rounded row is what attention then reads.

Readings where the pages are silent (listed with reasons in the design
notes): RoPE is the rotate-half form with inv_freq_i = theta**(-2i/D) built
in float64; the new token sits at position pos and attends to pos+1 keys;
the softmax scale is 1/sqrt(D); gate/up are stacked as [gate; up] rows;
argmax ties go to the lowest index; the embedding is a row gather of the
bf16 table widened to float.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


# ------------------------------------------------------------------ formats
def bf16_to_f64(u16) -> np.ndarray:
    """Exact widening of bf16 codes (uint16) to float64."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def round_to_bf16_via_f32(x) -> np.ndarray:
    """float64 -> float32 (nearest) -> bf16 code (nearest even)."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return r.astype(np.uint16)


# ------------------------------------------------------------------ operations
def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """x * (1 / sqrt(mean(x^2) + eps)) * gamma over the last axis."""
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x * (1.0 / np.sqrt(ms + eps)) * gamma


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def rope_inv_freq(D: int, theta: float) -> np.ndarray:
    i = np.arange(D // 2, dtype=np.float64)
    return theta ** (-2.0 * i / D)


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE of the last axis (length D) at integer position pos:
    pairs (i, i + D/2) are rotated by the angle pos * theta**(-2i/D)."""
    D = v.shape[-1]
    ang = float(pos) * rope_inv_freq(D, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., : D // 2], v[..., D // 2:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def attention_single(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """softmax(q K^T / sqrt(D)) V for q [Hg, D], K/V [n, D] (float64)."""
    D = q.shape[-1]
    s = q @ K.T / np.sqrt(D)
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return (p @ V) / p.sum(axis=-1, keepdims=True)


def attention_partial(q: np.ndarray, K: np.ndarray, V: np.ndarray):
    """One split-KV partial ("ATTENTION_PARTIAL": online softmax over one KV
    chunk giving (m, l, o) scratch).  Returns per head: m = max score,
    l = sum exp(s - m), o = sum exp(s - m) v (unnormalised).  An empty chunk
    gives m = -inf, l = 0, o = 0."""
    Hg, D = q.shape
    if K.shape[0] == 0:
        return (np.full(Hg, -np.inf), np.zeros(Hg), np.zeros((Hg, D)))
    s = q @ K.T / np.sqrt(D)
    m = s.max(axis=-1)
    p = np.exp(s - m[:, None])
    return m, p.sum(axis=-1), p @ V


def attention_combine(parts):
    """Log-sum-exp merge of split-KV partials ("ATTENTION_COMBINE")."""
    ms = np.stack([p[0] for p in parts])          # [P, Hg]
    M = ms.max(axis=0)
    w = np.where(np.isfinite(ms), np.exp(ms - M[None, :]), 0.0)
    L = sum(w[i] * parts[i][1] for i in range(len(parts)))
    O = sum(w[i][:, None] * parts[i][2] for i in range(len(parts)))
    return O / L[:, None]


def chunk_bounds(L_cur: int, P: int):
    """Key ranges of the P split-KV chunks over L_cur keys: chunk c covers
    [c*e, min((c+1)*e, L_cur)) with e = ceil(L_cur / P); trailing chunks may
    be empty."""
    e = -(-L_cur // P)
    return [(min(c * e, L_cur), min((c + 1) * e, L_cur)) for c in range(P)]


def argmax_first(x: np.ndarray) -> int:
    return int(np.argmax(x))


def top2_margin(x: np.ndarray) -> float:
    if x.size < 2:
        return float("inf")
    part = np.partition(x, -2)
    return float(part[-1] - part[-2])


# ------------------------------------------------------------------ model
@dataclass
class DecodeState:
    """Caller-visible decode state: next input token and its position per
    sequence, bf16 KV caches per layer ([B, Hkv, cap, D] uint16 codes), and
    the history of sampled tokens."""
    token: np.ndarray
    pos: np.ndarray
    kcache: list
    vcache: list
    history: np.ndarray


@dataclass
class StepResult:
    logits: np.ndarray                      # [B, V] float64
    hidden: list = field(default_factory=list)   # per layer [B, H] float64
    tokens: np.ndarray = None               # [B] int64
    margin: np.ndarray = None               # [B] top-2 logit margin


def _gemv(W_u16: np.ndarray, x: np.ndarray) -> np.ndarray:
    """y = W x with bf16 W [out, in] widened to float64; x [B, in]."""
    return x @ bf16_to_f64(W_u16).T


def decode_step(model, weights, st: DecodeState, keep_hidden: bool = True) -> StepResult:
    """One greedy decode step for every sequence; updates ``st`` in place.

    ``model`` has L, H, Hq, Hkv, D, F, V, theta, eps, tied; ``weights`` maps
    the names of ``synth.weight_names`` to uint16 bf16 codes (a mapping or a
    callable name -> array)."""
    W = weights if callable(weights) else weights.__getitem__
    B = st.token.shape[0]
    H, Hq, Hkv, D, F = model.H, model.Hq, model.Hkv, model.D, model.F
    G = Hq // Hkv
    E = W("embed")
    h = bf16_to_f64(E[st.token])                                  # [B, H]
    res = StepResult(logits=None)
    for l in range(model.L):
        xn = rmsnorm(h, bf16_to_f64(W(f"layer{l}.attn_norm")), model.eps)
        qkv = _gemv(W(f"layer{l}.wqkv"), xn)                     # [B, (Hq+2Hkv)D]
        att = np.zeros((B, Hq * D))
        Kc, Vc = st.kcache[l], st.vcache[l]
        for s in range(B):
            p = int(st.pos[s])
            q = qkv[s, : Hq * D].reshape(Hq, D)
            k = qkv[s, Hq * D: (Hq + Hkv) * D].reshape(Hkv, D)
            v = qkv[s, (Hq + Hkv) * D:].reshape(Hkv, D)
            Kc[s, :, p, :] = round_to_bf16_via_f32(rope(k, p, model.theta))
            Vc[s, :, p, :] = round_to_bf16_via_f32(v)
            qr = rope(q, p, model.theta)
            for g in range(Hkv):
                Kf = bf16_to_f64(Kc[s, g, : p + 1])
                Vf = bf16_to_f64(Vc[s, g, : p + 1])
                o = attention_single(qr[g * G:(g + 1) * G], Kf, Vf)
                att[s, g * G * D:(g + 1) * G * D] = o.reshape(-1)
        h = h + _gemv(W(f"layer{l}.wo"), att)
        xn = rmsnorm(h, bf16_to_f64(W(f"layer{l}.mlp_norm")), model.eps)
        gu = _gemv(W(f"layer{l}.wgu"), xn)
        act = silu(gu[:, :F]) * gu[:, F:]
        h = h + _gemv(W(f"layer{l}.wd"), act)
        if keep_hidden:
            res.hidden.append(h.copy())
    xn = rmsnorm(h, bf16_to_f64(W("final_norm")), model.eps)
    lm = W("embed") if model.tied else W("lm_head")
    logits = _gemv(lm, xn)
    res.logits = logits
    res.tokens = np.array([argmax_first(logits[s]) for s in range(B)], dtype=np.int64)
    res.margin = np.array([top2_margin(logits[s]) for s in range(B)])
    for s in range(B):
        p = int(st.pos[s])
        st.history[s, p + 1] = res.tokens[s]
        st.token[s] = res.tokens[s]
        st.pos[s] = p + 1
    return res


def chunk_step(model, weights, st: DecodeState, tokens: np.ndarray) -> StepResult:
    """Several tokens per sequence in one step (a prefill chunk, or a batch
    of draft tokens to verify): ``tokens`` [B, T] are the inputs at
    positions pos .. pos + T - 1, the first of them the pending token
    ``st.token``.  Each layer runs on all B * T rows; token t appends its
    key/value row at pos + t and attends, causally, to rows 0 .. pos + t
    (the cache plus the chunk's earlier tokens).  Returns the logits of
    every row ([B, T, V]) and hidden states [B, T, H]; the next token is the
    argmax of each sequence's last row; history gets the given tokens and
    the sampled one, pos advances by T.  This is T decode steps with the
    inputs fixed in advance, written as the plain definition."""
    W = weights if callable(weights) else weights.__getitem__
    tokens = np.asarray(tokens, dtype=np.int64)
    B, T = tokens.shape
    assert np.array_equal(tokens[:, 0], st.token), "the chunk starts with the pending token"
    H, Hq, Hkv, D, F = model.H, model.Hq, model.Hkv, model.D, model.F
    G = Hq // Hkv
    h = bf16_to_f64(W("embed")[tokens.reshape(-1)])               # [B*T, H], row s*T + t
    res = StepResult(logits=None)
    for l in range(model.L):
        xn = rmsnorm(h, bf16_to_f64(W(f"layer{l}.attn_norm")), model.eps)
        qkv = _gemv(W(f"layer{l}.wqkv"), xn)
        att = np.zeros((B * T, Hq * D))
        Kc, Vc = st.kcache[l], st.vcache[l]
        for s in range(B):
            for t in range(T):
                r, p = s * T + t, int(st.pos[s]) + t
                q = qkv[r, : Hq * D].reshape(Hq, D)
                k = qkv[r, Hq * D: (Hq + Hkv) * D].reshape(Hkv, D)
                v = qkv[r, (Hq + Hkv) * D:].reshape(Hkv, D)
                Kc[s, :, p, :] = round_to_bf16_via_f32(rope(k, p, model.theta))
                Vc[s, :, p, :] = round_to_bf16_via_f32(v)
                qr = rope(q, p, model.theta)
                for g in range(Hkv):
                    o = attention_single(qr[g * G:(g + 1) * G], bf16_to_f64(Kc[s, g, : p + 1]),
                                         bf16_to_f64(Vc[s, g, : p + 1]))
                    att[r, g * G * D:(g + 1) * G * D] = o.reshape(-1)
        h = h + _gemv(W(f"layer{l}.wo"), att)
        xn = rmsnorm(h, bf16_to_f64(W(f"layer{l}.mlp_norm")), model.eps)
        gu = _gemv(W(f"layer{l}.wgu"), xn)
        h = h + _gemv(W(f"layer{l}.wd"), silu(gu[:, :F]) * gu[:, F:])
        res.hidden.append(h.reshape(B, T, H).copy())
    xn = rmsnorm(h, bf16_to_f64(W("final_norm")), model.eps)
    logits = _gemv(W("embed") if model.tied else W("lm_head"), xn).reshape(B, T, -1)
    res.logits = logits
    res.tokens = np.array([argmax_first(logits[s, -1]) for s in range(B)], dtype=np.int64)
    res.margin = np.array([top2_margin(logits[s, -1]) for s in range(B)])
    for s in range(B):
        p = int(st.pos[s])
        st.history[s, p + 1: p + T] = tokens[s, 1:]
        st.history[s, p + T] = res.tokens[s]
        st.token[s] = res.tokens[s]
        st.pos[s] = p + T
    return res


def initial_state(model, B: int, cap: int, kv_len, tokens, kv_provider) -> DecodeState:
    """State before the first step: ``kv_provider(layer, 'k'|'v')`` returns a
    [B, Hkv, cap, D] uint16 cache holding kv_len[s] valid rows."""
    kc = [kv_provider(l, "k") for l in range(model.L)]
    vc = [kv_provider(l, "v") for l in range(model.L)]
    hist = np.zeros((B, cap), dtype=np.int64)
    pos = np.array(kv_len, dtype=np.int64)
    tok = np.array(tokens, dtype=np.int64)
    for s in range(B):
        hist[s, pos[s]] = tok[s]
    return DecodeState(token=tok, pos=pos, kcache=kc, vcache=vc, history=hist)
