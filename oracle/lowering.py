"""Oracle lowering: graph ops -> 64-byte task descriptors + dependents edges.

TEST INFRASTRUCTURE ONLY (see ``oracle/forward.py``).  Written independently
of the C++ lowering in the library; the two must emit identical bytes.

Source: "mega kernel initial" (1y33.com).
* Each op becomes one or more 64-byte task descriptors (the lowering part
  and its TaskDescriptor listing: op_id@0, config_id@2, step@4, flags@6,
  remaining_deps@8, num_dependents@12, dependents_offset@16, in_buf[3]@20,
  out_buf@26, m@28, n@32, k@36, kv_len@40, reserved[5]@44).
* A matmul fans out into one GEMV task per output-column tile, roughly one
  per SM; 3072 columns over 8 tiles gives 8 tasks of 384 columns.
* Attention becomes ATTENTION_PARTIAL tasks per (sequence, KV-head group,
  KV chunk) followed by a combine (plain flash decoding); the current k/v
  are RoPE-appended by ATTENTION_APPEND (the OpId table).
* RMSNorm-on-input, residual add and SiLU*mul are flags on the GEMV
  (bit0 SILU_MUL, bit1 ADD_RESIDUAL, bit2 RMS_NORM_INPUT).
* Every op output remembers which task wrote which column range; a reader
  depends on the writers of what it reads.  Parents are then flipped into
  per-task dependents lists flattened into one edge array, and tasks are
  emitted in topological order.

Readings taken where the page is silent (the same frozen spec the library
implements): the tile rule col_tile = round_up(ceil(n / tiles_target),
col_align); one COMBINE per (sequence, KV head); the split-KV chunk rule in
``partials_per_sequence``; bit3 ARGMAX_EPI on the lm_head GEMV, whose tiles
carry their tile index in reserved[4] (the pair column they write); the embedding
row gather as a MEMCPY task carrying the table's row count in reserved[1];
the per-tile (max, index) pairs stored tile-major ([T, B]); field maps per
op as in ``lower`` below.
Access ranges are tracked as row x column rectangles of each buffer's 2-D
view, so per-sequence writes (embedding, combine) do not alias.  In a KV
cache block, columns [0, cap*D) stand for the rows of earlier steps and
[cap*D, cap*D + D) for the row this step appends: APPEND writes only the
latter, PARTIAL reads only the former (it takes the appended key and value
from qkv, rotated and rounded as APPEND stores them), so the partials do not
wait for the append.  COMBINE takes the appended row as an input (its
in_buf[1..2] are the caches), so the append is complete before the
attention output is and every reader of the decode state stays an
ancestor of SAMPLE, which advances it.

Chunk steps (T tokens per sequence per step, a prefill chunk or a batch of
speculative draft tokens; the TaskDescriptor listing names ``step`` as the
draft-step tag).  Our reading, byte-identical to the above when T = 1:
activations have B*T rows (row s*T + t); the embedding gather and the cache
append become one task per token with ``step`` = t; token t's appended row
stands as columns [cap*D + t*D, cap*D + (t+1)*D) of its cache block; each
partial serves the T tokens of its sequence and its scratch slot holds
T*G*(D+2) floats; attention tasks carry T-1 in the high half of
reserved[2], the embedding gather in reserved[2], SAMPLE in reserved[1];
tokens 1..T-1 come from an int32 [B, T] input buffer (in_buf[1] of the
embedding gathers and of SAMPLE), which no task writes.
"""
from __future__ import annotations

import struct

import numpy as np

ABI_VERSION = 1

OP_NOP, OP_MEMCPY, OP_GEMV, OP_RMSNORM, OP_ATTENTION, OP_MLP, OP_SAMPLE = 0, 1, 2, 3, 4, 5, 6
OP_ATT_APPEND, OP_ATT_PARTIAL, OP_ATT_COMBINE = 7, 8, 9

F_SILU_MUL, F_ADD_RESIDUAL, F_RMS_NORM_INPUT, F_ARGMAX_EPI = 1, 2, 4, 8

TC_MIN_ROWS = 3   # activation rows from which GEMV tiles are config 1 (tensor cores)

NO_BUF = 0xFFFF
BUF_STATE, BUF_ROPE_COS, BUF_ROPE_SIN = 0, 1, 2

TASK_DTYPE = np.dtype([
    ("op_id", "<u2"), ("config_id", "<u2"), ("step", "<u2"), ("flags", "<u2"),
    ("remaining_deps", "<i4"), ("num_dependents", "<i4"), ("dependents_offset", "<u4"),
    ("in_buf", "<u2", (3,)), ("out_buf", "<u2"),
    ("m", "<i4"), ("n", "<i4"), ("k", "<i4"), ("kv_len", "<i4"),
    ("reserved", "<u4", (5,)),
])
assert TASK_DTYPE.itemsize == 64


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def tile_width(n: int, tiles_target: int, col_align: int) -> int:
    return ceil_div(ceil_div(n, tiles_target), col_align) * col_align


def tiles(n: int, tiles_target: int, col_align: int):
    """[(col_begin, col_count)] of the GEMV column tiles of an n-column op."""
    w = tile_width(n, tiles_target, col_align)
    return [(c, min(w, n - c)) for c in range(0, n, w)]


KSPLIT_BUF = 0xFFFE           # pseudo buffer: the library's K-split scratch records
KSPLIT_REC = 256 * 8 + 8      # floats per record


def ksplit_plan(n: int, k: int, flags: int, m: int, tiles_target: int, col_align: int):
    """(W, nb, S) of a GEMV op: rows per tile or block, blocks, K splits.

    Our reading for batch >= 8 (tensor-core GEMV tiles, whose every MMA costs
    the same for up to 256 weight rows): when the usual per-SM tiles are
    narrow (seg * width < 128 rows; seg = 2 with SILU_MUL, gate and up rows
    sharing the MMA), the op is cut into blocks of up to 256 / seg rows
    (ceil(seg * n / 256) blocks, width rounded up to 8) and each block into
    S = min(k / 64, tiles_target // blocks) consecutive K ranges of whole
    64-column blocks; S < 2, an argmax epilogue, or m < TC_MIN_ROWS keep the tiling."""
    W = tile_width(n, tiles_target, col_align)
    seg = 2 if flags & F_SILU_MUL else 1
    plain = (W, ceil_div(n, W), 1)
    if m < TC_MIN_ROWS or flags & F_ARGMAX_EPI or seg * W >= 128 or k % 64:
        return plain
    nb = ceil_div(seg * n, 256)
    Wb = ceil_div(ceil_div(n, nb), 8) * 8
    S = max(1, min(k // 64, tiles_target // ceil_div(n, Wb)))
    if S < 2:
        return plain
    return Wb, ceil_div(n, Wb), S


def partials_per_sequence(len0, Hkv: int, chunk: int, num_ctas: int):
    """Split-KV chunk count P_s per sequence (fixed at lowering time).
    chunk > 0: ceil(len0_s / chunk).  chunk == 0: chunks of E keys, E the
    smallest length of at least max(128, ceil(Hkv * sum(len0) / num_ctas))
    for which Hkv * sum_s max(1, ceil(len0_s / E)) <= num_ctas (or the
    longest sequence, when even one chunk per sequence is more than that):
    the partial tasks of a ragged batch carry about the same bytes and fit
    one wave of the CTAs."""
    lens = [int(l) for l in len0]
    if chunk > 0:
        return [max(1, ceil_div(l, chunk)) for l in lens]

    def count(E):
        return Hkv * sum(max(1, ceil_div(l, E)) for l in lens)

    lo = max(128, ceil_div(Hkv * sum(lens), num_ctas))
    hi = max(lo, max(lens) if lens else lo)
    if count(lo) > num_ctas:  # smallest E in (lo, hi] that fits, else hi
        a, b = lo, hi
        while b - a > 1:
            m = (a + b) // 2
            if count(m) <= num_ctas:
                b = m
            else:
                a = m
        lo = b
    return [max(1, ceil_div(l, lo)) for l in lens]


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


class _Writes:
    """Per-buffer record of which task wrote which row x column rectangle."""

    def __init__(self):
        self.by_buf = {}

    def add(self, buf, task, r0, r1, c0, c1):
        self.by_buf.setdefault(buf, []).append((task, r0, r1, c0, c1))

    def writers(self, buf, r0, r1, c0, c1):
        out = set()
        for (t, a0, a1, b0, b1) in self.by_buf.get(buf, ()):
            if a0 < r1 and r0 < a1 and b0 < c1 and c0 < b1:
                out.add(t)
        return out


def lower(spec: dict):
    """Lower a graph spec to (tasks [N] TASK_DTYPE, edges [E] uint32).

    spec = {"num_ctas", "tiles_target" (0 = num_ctas), "col_align",
            "buffers": [(dtype, rows, cols)] indexed by buffer id,
            "ops": [dict(kind=..., ...)] in call order}."""
    num_ctas = spec["num_ctas"]
    tt = spec.get("tiles_target", 0) or num_ctas
    align = spec.get("col_align", 16)
    bufs = spec["buffers"]
    T = spec.get("T", 1)                 # tokens per sequence per step
    tok = spec.get("tokens", NO_BUF)     # int32 [B, T] input tokens (T > 1)
    descs = []       # list of dict fields
    parents = []     # list of sets
    W = _Writes()
    records = 0      # K-split scratch records assigned so far

    def emit(fields, reads, writes):
        t = len(descs)
        ps = set()
        for (b, r0, r1, c0, c1) in reads:
            ps |= W.writers(b, r0, r1, c0, c1)
        for (b, r0, r1, c0, c1) in writes:
            W.add(b, t, r0, r1, c0, c1)
        descs.append(fields)
        parents.append(ps)

    for op in spec["ops"]:
        kind = op["kind"]
        if kind == "embed":
            B, H = op["B"], op["H"]
            for s in range(B):
                for t in range(T):
                    # token 0: the pending token in the state; 1..: the input buffer
                    src = (BUF_STATE, s, s + 1, 0, 2) if t == 0 else (tok, s, s + 1, t, t + 1)
                    emit(dict(op_id=OP_MEMCPY, step=t,
                              in_buf=(op["table"], tok if T > 1 else NO_BUF, NO_BUF),
                              out_buf=op["out"], m=B, n=H,
                              reserved=(s, bufs[op["table"]][1], T - 1, 0, 0)),
                         reads=[src],
                         writes=[(op["out"], s * T + t, s * T + t + 1, 0, H)])
        elif kind == "matmul":
            B, n, K, fl = op["m"], op["n"], op["k"], op["flags"]
            aux = op.get("aux", NO_BUF)
            pairs = op.get("pairs", NO_BUF)
            eps_bits = f32_bits(op["eps"]) if fl & F_RMS_NORM_INPUT else 0
            Wb, nb, S = ksplit_plan(n, K, fl, B, tt, align)
            if S > 1:
                # split j of a row block multiplies K columns [k0, k1); the
                # last split adds the others' partial sums (read from their
                # scratch records, in order) and runs the epilogue
                KB = K // 64
                for c0 in range(0, n, Wb):
                    cn = min(Wb, n - c0)
                    for j in range(S):
                        k0, k1 = (j * KB // S) * 64, ((j + 1) * KB // S) * 64
                        reads = [(op["x"], 0, B, k0, k1)]
                        if j + 1 < S:
                            writes = [(KSPLIT_BUF, records + j, records + j + 1, 0, KSPLIT_REC)]
                        else:
                            reads.append((KSPLIT_BUF, records, records + j, 0, KSPLIT_REC))
                            if fl & F_ADD_RESIDUAL:
                                reads.append((aux, 0, B, c0, c0 + cn))
                            writes = [(op["out"], 0, B, c0, c0 + cn)]
                        emit(dict(op_id=OP_GEMV, config_id=1, flags=fl,
                                  in_buf=(op["x"], op["w"], aux), out_buf=op["out"],
                                  m=B, n=n, k=K, kv_len=j | (S << 16),
                                  reserved=(c0, cn, eps_bits, k0 | ((k1 - k0) << 16), records + j)),
                             reads, writes)
                    records += S
                continue
            for t, (c0, cn) in enumerate(tiles(n, tt, align)):
                reads = [(op["x"], 0, B, 0, K)]
                if fl & F_ADD_RESIDUAL:
                    reads.append((aux, 0, B, c0, c0 + cn))
                writes = [(op["out"], 0, B, c0, c0 + cn)]
                if fl & F_ARGMAX_EPI:
                    writes.append((pairs, t, t + 1, 0, B))
                emit(dict(op_id=OP_GEMV, config_id=0 if B < TC_MIN_ROWS else 1, flags=fl,
                          in_buf=(op["x"], op["w"], aux), out_buf=op["out"],
                          m=B, n=n, k=K,
                          reserved=(c0, cn, eps_bits,
                                    pairs if fl & F_ARGMAX_EPI else 0,
                                    t if fl & F_ARGMAX_EPI else 0)),
                     reads, writes)
        elif kind == "attention":
            B, Hq, Hkv, D, cap = op["B"], op["Hq"], op["Hkv"], op["D"], op["capacity"]
            G = Hq // Hkv
            cfg = 0 if D == 64 else 1
            qkv, kc, vc, out, scr = op["qkv"], op["k"], op["v"], op["out"], op["scratch"]
            P = partials_per_sequence(op["len0"], Hkv, op["chunk"], num_ctas)
            base = []
            acc = 0
            for s in range(B):
                base.append([acc + g * P[s] for g in range(Hkv)])
                acc += Hkv * P[s]
            common = dict(m=B, n=D, k=Hq, kv_len=cap)
            hkv_t = Hkv | ((T - 1) << 16)
            rec = T * G * (D + 2)            # floats of one scratch slot
            new0, new1 = cap * D, cap * D + T * D   # the columns standing for this step's rows
            for s in range(B):
                for g in range(Hkv):
                    kcol = Hq * D + g * D
                    vcol = (Hq + Hkv) * D + g * D
                    row = s * Hkv + g
                    for t in range(T):
                        r = s * T + t
                        emit(dict(op_id=OP_ATT_APPEND, config_id=cfg, step=t, in_buf=(qkv, kc, vc),
                                  out_buf=kc, reserved=(s, g, hkv_t, 0, 0), **common),
                             reads=[(qkv, r, r + 1, kcol, kcol + D),
                                    (qkv, r, r + 1, vcol, vcol + D),
                                    (BUF_STATE, s, s + 1, 0, 2)],
                             writes=[(kc, row, row + 1, new0 + t * D, new0 + (t + 1) * D),
                                     (vc, row, row + 1, new0 + t * D, new0 + (t + 1) * D)])
            for s in range(B):
                for g in range(Hkv):
                    row = s * Hkv + g
                    r0, r1 = s * T, s * T + T
                    for c in range(P[s]):
                        slot = base[s][g] + c
                        emit(dict(op_id=OP_ATT_PARTIAL, config_id=cfg, in_buf=(qkv, kc, vc),
                                  out_buf=scr,
                                  reserved=(s, g, hkv_t, c | (P[s] << 16), base[s][g]),
                                  **common),
                             reads=[(qkv, r0, r1, g * G * D, (g + 1) * G * D),
                                    (qkv, r0, r1, Hq * D + g * D, Hq * D + (g + 1) * D),
                                    (qkv, r0, r1, (Hq + Hkv) * D + g * D, (Hq + Hkv) * D + (g + 1) * D),
                                    (kc, row, row + 1, 0, cap * D),
                                    (vc, row, row + 1, 0, cap * D),
                                    (BUF_STATE, s, s + 1, 0, 2)],
                             writes=[(scr, slot, slot + 1, 0, rec)])
            for s in range(B):
                for g in range(Hkv):
                    row = s * Hkv + g
                    emit(dict(op_id=OP_ATT_COMBINE, config_id=cfg,
                              in_buf=(scr, kc, vc), out_buf=out,
                              reserved=(s, g, hkv_t, P[s], base[s][g]), **common),
                         reads=[(scr, base[s][g], base[s][g] + P[s], 0, rec),
                                (kc, row, row + 1, new0, new1),
                                (vc, row, row + 1, new0, new1)],
                         writes=[(out, s * T, s * T + T, g * G * D, (g + 1) * G * D)])
        elif kind == "rmsnorm":
            # standalone RMS norm per sequence (OpId table: usually fused,
            # rarely standalone); a residual makes it FUSED_RESIDUAL (bit 1)
            B, H = op["B"], op["H"]
            res = op.get("residual", NO_BUF)
            for s in range(B * T):          # one task per activation row
                reads = [(op["x"], s, s + 1, 0, H)]
                if res != NO_BUF:
                    reads.append((res, s, s + 1, 0, H))
                emit(dict(op_id=OP_RMSNORM, flags=F_ADD_RESIDUAL if res != NO_BUF else 0,
                          in_buf=(op["x"], op["gamma"], res), out_buf=op["out"], m=B, n=H,
                          reserved=(s, f32_bits(op["eps"]), 0, 0, 0)),
                     reads, writes=[(op["out"], s, s + 1, 0, H)])
        elif kind == "sample":
            B, V, cap = op["B"], op["V"], op["capacity"]
            NT = len(tiles(V, tt, align))
            for s in range(B):
                last = s * T + T - 1        # the sequence's last row decides the next token
                reads = [(op["pairs"], 0, NT, last, last + 1), (BUF_STATE, s, s + 1, 0, 2)]
                if T > 1:
                    reads.append((tok, s, s + 1, 0, T))
                emit(dict(op_id=OP_SAMPLE, in_buf=(op["pairs"], tok if T > 1 else NO_BUF, NO_BUF),
                          out_buf=op["history"], m=B, n=V, k=NT, kv_len=cap,
                          reserved=(s, T - 1, 0, 0, 0)),
                     reads=reads,
                     writes=[(op["history"], s, s + 1, 0, cap),
                             (BUF_STATE, s, s + 1, 0, 2)])
        else:
            raise ValueError(kind)

    N = len(descs)
    children = [[] for _ in range(N)]
    for t in range(N):
        for p in sorted(parents[t]):
            assert p < t
            children[p].append(t)
    tasks = np.zeros(N, dtype=TASK_DTYPE)
    off = 0
    edges = []
    for t, f in enumerate(descs):
        d = tasks[t]
        d["op_id"] = f["op_id"]
        d["config_id"] = f.get("config_id", 0)
        d["step"] = f.get("step", 0)
        d["flags"] = f.get("flags", 0)
        d["remaining_deps"] = len(parents[t])
        d["num_dependents"] = len(children[t])
        d["dependents_offset"] = off
        d["in_buf"] = f["in_buf"]
        d["out_buf"] = f["out_buf"]
        d["m"] = f.get("m", 0)
        d["n"] = f.get("n", 0)
        d["k"] = f.get("k", 0)
        d["kv_len"] = f.get("kv_len", 0)
        d["reserved"] = f["reserved"]
        edges.extend(children[t])
        off += len(children[t])
    return tasks, np.array(edges, dtype=np.uint32)
