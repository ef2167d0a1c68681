"""Brute-force, element-by-element Llama decode step in plain Python floats.

An independent second statement of the decode step, used to pin the NumPy
oracle on tiny inputs.  Written without NumPy linear algebra: explicit loops
over weight rows, RoPE as multiplication of (x_i + i*x_{i+D/2}) by
exp(i * angle), softmax as explicit exponentials, and bf16 conversion through
the IEEE-754 bit patterns via ``struct``.
"""
from __future__ import annotations

import cmath
import math
import struct


def bf16(code: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(code) & 0xFFFF) << 16))[0]


def to_bf16_code(x: float) -> int:
    """Round x to float32 (nearest), then to bf16 (nearest, ties to even)."""
    bits = struct.unpack("<I", struct.pack("<f", x))[0]
    upper, lower = bits >> 16, bits & 0xFFFF
    if lower > 0x8000 or (lower == 0x8000 and (upper & 1)):
        upper += 1
    return upper & 0xFFFF


def row(mat, r):
    return [bf16(c) for c in mat[r].tolist()]


def matvec(mat, x):
    out = []
    for r in range(mat.shape[0]):
        w = mat[r].tolist()
        acc = 0.0
        for j in range(len(x)):
            acc += bf16(w[j]) * x[j]
        out.append(acc)
    return out


def rms_normalise(x, gamma_codes, eps):
    ss = 0.0
    for v in x:
        ss += v * v
    inv = 1.0 / math.sqrt(ss / len(x) + eps)
    g = gamma_codes.tolist()
    return [x[i] * inv * bf16(g[i]) for i in range(len(x))]


def rotate(vec, pos, theta):
    D = len(vec)
    half = D // 2
    out = [0.0] * D
    for i in range(half):
        z = complex(vec[i], vec[i + half]) * cmath.exp(1j * pos * theta ** (-2.0 * i / D))
        out[i], out[i + half] = z.real, z.imag
    return out


def decode_step(model, W, token, pos, kc, vc):
    """One step for a single sequence.  W(name) -> uint16 array; kc/vc are
    per-layer [Hkv, cap, D] uint16 arrays that receive the new row.
    Returns (logits, per-layer hidden, next token)."""
    H, Hq, Hkv, D, F = model.H, model.Hq, model.Hkv, model.D, model.F
    G = Hq // Hkv
    h = row(W("embed"), token)
    hidden = []
    for l in range(model.L):
        xn = rms_normalise(h, W(f"layer{l}.attn_norm"), model.eps)
        qkv = matvec(W(f"layer{l}.wqkv"), xn)
        att = [0.0] * (Hq * D)
        for g in range(Hkv):
            k = rotate(qkv[Hq * D + g * D: Hq * D + (g + 1) * D], pos, model.theta)
            v = qkv[(Hq + Hkv) * D + g * D: (Hq + Hkv) * D + (g + 1) * D]
            for d in range(D):
                kc[l][g, pos, d] = to_bf16_code(k[d])
                vc[l][g, pos, d] = to_bf16_code(v[d])
        for hh in range(Hq):
            g = hh // G
            q = rotate(qkv[hh * D:(hh + 1) * D], pos, model.theta)
            scores = []
            for j in range(pos + 1):
                kr = kc[l][g, j].tolist()
                scores.append(sum(q[d] * bf16(kr[d]) for d in range(D)) / math.sqrt(D))
            mx = max(scores)
            ex = [math.exp(s - mx) for s in scores]
            tot = sum(ex)
            for j in range(pos + 1):
                vr = vc[l][g, j].tolist()
                for d in range(D):
                    att[hh * D + d] += ex[j] / tot * bf16(vr[d])
        o = matvec(W(f"layer{l}.wo"), att)
        h1 = [h[i] + o[i] for i in range(H)]
        xn = rms_normalise(h1, W(f"layer{l}.mlp_norm"), model.eps)
        gu = matvec(W(f"layer{l}.wgu"), xn)
        act = []
        for j in range(F):
            gate, up = gu[j], gu[F + j]
            act.append(gate / (1.0 + math.exp(-gate)) * up)
        dn = matvec(W(f"layer{l}.wd"), act)
        h = [h1[i] + dn[i] for i in range(H)]
        hidden.append(list(h))
    xn = rms_normalise(h, W("final_norm"), model.eps)
    logits = matvec(W("embed") if model.tied else W("lm_head"), xn)
    best = 0
    for i in range(1, len(logits)):
        if logits[i] > logits[best]:
            best = i
    return logits, hidden, best
