"""Oracle-side graph spec of a Llama-style decode step.

TEST INFRASTRUCTURE ONLY (see ``oracle/forward.py``).

Writes the decoder-layer listing of "mega kernel initial" (1y33.com, the
"building the graph" part) as plain op records for ``oracle.lowering.lower``:
embed -> per layer [qkv matmul with RMSNorm input, attention, o_proj with
residual, gate_up with RMSNorm input and SiLU*mul, down with residual] ->
lm_head matmul with the final RMSNorm fused and the per-tile argmax
epilogue -> SAMPLE.

Buffers are registered append-only, in this order (the library's Python
builder follows the same convention, so indices agree):
  0 state [B, 2] int32 (token, pos)     1, 2 RoPE cos / sin tables
  weights in ``synth.weight_names`` order
  per layer: K cache, V cache ([B*Hkv, cap*D] bf16)
  history [B, cap] int32
  (chunk steps, T > 1: tokens [B, T] int32, the step's input tokens)
  then activations and scratch as each op allocates its output.
Activations have B*T rows (row s*T + t); T = 1 is the decode step.
"""
from __future__ import annotations

from .lowering import (F_SILU_MUL, F_ADD_RESIDUAL, F_RMS_NORM_INPUT, F_ARGMAX_EPI,
                       NO_BUF, tiles, partials_per_sequence)

BF16, F32, I32, PAIR = 1, 2, 3, 4


def llama_decode_spec(model, B: int, len0, cap: int, chunk: int, num_ctas: int,
                      tiles_target: int = 0, col_align: int = 16, norms: str = "fused",
                      T: int = 1) -> dict:
    """norms: "fused" sets RMS_NORM_INPUT on the GEMVs that consume a norm;
    "standalone" emits each norm as its own op (a fresh output buffer) read
    by a plain GEMV."""
    assert norms in ("fused", "standalone")
    m = model
    tt = tiles_target or num_ctas
    bufs = [(I32, B, 2), (F32, cap, m.D // 2), (F32, cap, m.D // 2)]
    idx = {}

    def reg(name, dtype, rows, cols):
        bufs.append((dtype, rows, cols))
        idx[name] = len(bufs) - 1
        return idx[name]

    reg("embed", BF16, m.V, m.H)
    for l in range(m.L):
        reg(f"layer{l}.attn_norm", BF16, 1, m.H)
        reg(f"layer{l}.wqkv", BF16, m.n_qkv, m.H)
        reg(f"layer{l}.wo", BF16, m.H, m.Hq * m.D)
        reg(f"layer{l}.mlp_norm", BF16, 1, m.H)
        reg(f"layer{l}.wgu", BF16, 2 * m.F, m.H)
        reg(f"layer{l}.wd", BF16, m.H, m.F)
    reg("final_norm", BF16, 1, m.H)
    lm = idx["embed"] if m.tied else reg("lm_head", BF16, m.V, m.H)
    for l in range(m.L):
        reg(f"layer{l}.k_cache", BF16, B * m.Hkv, cap * m.D)
        reg(f"layer{l}.v_cache", BF16, B * m.Hkv, cap * m.D)
    hist = reg("history", I32, B, cap)
    tok = reg("tokens", I32, B, T) if T > 1 else NO_BUF
    M = B * T

    ops = []
    act = [0]

    def fresh(dtype, rows, cols):
        act[0] += 1
        return reg(f"act{act[0]}", dtype, rows, cols)

    def matmul(x, w, n, k, aux=NO_BUF, flags=0, eps=0.0, pairs=NO_BUF, out=None):
        out = fresh(F32, M, n) if out is None else out
        ops.append(dict(kind="matmul", x=x, w=w, out=out, aux=aux, pairs=pairs,
                        flags=flags, m=M, n=n, k=k, eps=eps))
        return out

    def normed(x, gamma, flags):
        """(input, aux, flags) of a GEMV that reads RMSNorm(x) * gamma."""
        if norms == "fused":
            return x, gamma, flags | F_RMS_NORM_INPUT
        xn = fresh(F32, M, m.H)
        ops.append(dict(kind="rmsnorm", x=x, gamma=gamma, residual=NO_BUF, out=xn, B=B, H=m.H, eps=m.eps))
        return xn, NO_BUF, flags

    h = fresh(F32, M, m.H)
    ops.append(dict(kind="embed", table=idx["embed"], out=h, B=B, H=m.H))
    G = m.Hq // m.Hkv
    P = partials_per_sequence(len0, m.Hkv, chunk, num_ctas)
    for l in range(m.L):
        x, a, f = normed(h, idx[f"layer{l}.attn_norm"], 0)
        qkv = matmul(x, idx[f"layer{l}.wqkv"], m.n_qkv, m.H, aux=a, flags=f, eps=m.eps)
        scr = fresh(F32, sum(P) * m.Hkv, T * G * (m.D + 2))
        att = fresh(F32, M, m.Hq * m.D)
        ops.append(dict(kind="attention", qkv=qkv, k=idx[f"layer{l}.k_cache"],
                        v=idx[f"layer{l}.v_cache"], out=att, scratch=scr, B=B, Hq=m.Hq,
                        Hkv=m.Hkv, D=m.D, capacity=cap, len0=list(len0), chunk=chunk))
        h1 = matmul(att, idx[f"layer{l}.wo"], m.H, m.Hq * m.D, aux=h, flags=F_ADD_RESIDUAL)
        x, a, f = normed(h1, idx[f"layer{l}.mlp_norm"], F_SILU_MUL)
        gu = matmul(x, idx[f"layer{l}.wgu"], m.F, m.H, aux=a, flags=f, eps=m.eps)
        h = matmul(gu, idx[f"layer{l}.wd"], m.H, m.F, aux=h1, flags=F_ADD_RESIDUAL)
    x, a, f = normed(h, idx["final_norm"], F_ARGMAX_EPI)
    NT = len(tiles(m.V, tt, col_align))
    logits = fresh(F32, M, m.V)
    pairs = fresh(PAIR, NT, M)
    matmul(x, lm, m.V, m.H, aux=a, flags=f, eps=m.eps, pairs=pairs, out=logits)
    ops.append(dict(kind="sample", pairs=pairs, history=hist, B=B, V=m.V, capacity=cap))
    return dict(num_ctas=num_ctas, tiles_target=tiles_target, col_align=col_align,
                buffers=bufs, ops=ops, names=idx, T=T, tokens=tok)


def fuse_rmsnorm(spec: dict):
    """Epilogue fusion on an op list: a norm without a residual whose output
    is read only as the x of GEMVs without an aux operand is folded into
    them (x = the norm's input, aux = its gain, RMS_NORM_INPUT, its eps) and
    dropped.  Returns (new spec, number of norms folded)."""
    import copy
    ops = copy.deepcopy(spec["ops"])

    def reads(op, b):
        k = op["kind"]
        if k == "embed":
            return op["table"] == b
        if k == "matmul":
            return b in (op["x"], op["w"], op.get("aux", NO_BUF))
        if k == "attention":
            return b in (op["qkv"], op["k"], op["v"])
        if k == "sample":
            return op["pairs"] == b
        if k == "rmsnorm":
            return b in (op["x"], op["gamma"], op.get("residual", NO_BUF))
        raise ValueError(k)

    out, folded = [], 0
    for i, op in enumerate(ops):
        if op["kind"] == "rmsnorm" and op.get("residual", NO_BUF) == NO_BUF:
            users = [j for j, r in enumerate(ops) if j != i and reads(r, op["out"])]
            ok = bool(users) and all(
                j > i and ops[j]["kind"] == "matmul" and ops[j]["x"] == op["out"] and ops[j]["w"] != op["out"]
                and ops[j].get("aux", NO_BUF) == NO_BUF and not ops[j]["flags"] & (F_RMS_NORM_INPUT | F_ADD_RESIDUAL)
                for j in users)
            if ok:
                for j in users:
                    ops[j].update(x=op["x"], aux=op["gamma"], eps=op["eps"],
                                  flags=ops[j]["flags"] | F_RMS_NORM_INPUT)
                folded += 1
                continue
        out.append(op)
    new = dict(spec)
    new["ops"] = out
    return new, folded
