"""DAG validator for a lowered task graph (descriptors + dependents edges).

TEST INFRASTRUCTURE ONLY (see ``oracle/forward.py``).

Checks the properties that "mega kernel initial" (1y33.com) states for its
lowered graph and that the interpreter's correctness rests on:

* tasks are in topological order: every edge points to a later task
  (the edge-array part: no task depends on a later one);
* each task's dependency count equals its number of parents, and the edge
  array is the flattened, offset-indexed dependents lists;
* a task's level is 1 + the max level of its parents, and two tasks of the
  same level are independent (the levels part);
* every pair of tasks touching overlapping data, at least one writing, is
  ordered by a path in the DAG (no read/write or write/write race);
* every read of a buffer that the graph writes is covered by earlier writes,
  except reads of data carried in from the previous step (the decode state,
  the KV rows of earlier steps) and reads of buffers whose writers all come
  later.

Access rectangles are decoded from the descriptor fields alone, by code
separate from the lowering that produced them.  A chunk step of T tokens per
sequence is read from the fields that carry T - 1 (reserved[2] of the
embedding gathers, the high half of reserved[2] of attention tasks,
reserved[1] of SAMPLE); ``step`` must be the token index of the per-token
tasks (embedding gathers and cache appends) and 0 everywhere else.
"""
from __future__ import annotations

from collections import defaultdict

import numpy as np

from .lowering import (OP_MEMCPY, OP_GEMV, OP_RMSNORM, OP_SAMPLE, OP_ATT_APPEND, OP_ATT_PARTIAL,
                       OP_ATT_COMBINE, F_ADD_RESIDUAL, F_ARGMAX_EPI, NO_BUF, BUF_STATE, KSPLIT_BUF,
                       KSPLIT_REC)


class ValidationError(AssertionError):
    pass


def task_accesses(d) -> tuple:
    """(reads, writes) as lists of (buf, r0, r1, c0, c1) for one descriptor."""
    op = int(d["op_id"])
    ib = [int(x) for x in d["in_buf"]]
    ob = int(d["out_buf"])
    rs = [int(x) for x in d["reserved"]]
    m, n, k, kv = int(d["m"]), int(d["n"]), int(d["k"]), int(d["kv_len"])
    R, Wr = [], []
    step = int(d["step"])
    if op == OP_MEMCPY:
        s, T = rs[0], rs[2] + 1
        if step >= T:
            raise ValidationError(f"embedding gather with step {step} >= T {T}")
        R.append((BUF_STATE, s, s + 1, 0, 2) if step == 0 else (ib[1], s, s + 1, step, step + 1))
        Wr.append((ob, s * T + step, s * T + step + 1, 0, n))
    elif op == OP_RMSNORM:
        s = rs[0]
        R.append((ib[0], s, s + 1, 0, n))
        if int(d["flags"]) & F_ADD_RESIDUAL:
            R.append((ib[2], s, s + 1, 0, n))
        Wr.append((ob, s, s + 1, 0, n))
    elif op == OP_GEMV and int(d["config_id"]) == 1 and (kv >> 16) >= 2:
        # split j of a K-split row block: its K range of x; the last split
        # reads the others' scratch records and writes the block's outputs
        c0, cn = rs[0], rs[1]
        S, j = kv >> 16, kv & 0xFFFF
        k0, kn = rs[3] & 0xFFFF, rs[3] >> 16
        if j >= S or kn <= 0 or k0 + kn > k:
            raise ValidationError(f"bad K split {j}/{S} [{k0}, {k0 + kn}) of K {k}")
        R.append((ib[0], 0, m, k0, k0 + kn))
        if j + 1 < S:
            Wr.append((KSPLIT_BUF, rs[4], rs[4] + 1, 0, KSPLIT_REC))
        else:
            R.append((KSPLIT_BUF, rs[4] - j, rs[4], 0, KSPLIT_REC))
            if int(d["flags"]) & F_ADD_RESIDUAL:
                R.append((ib[2], 0, m, c0, c0 + cn))
            Wr.append((ob, 0, m, c0, c0 + cn))
    elif op == OP_GEMV:
        c0, cn = rs[0], rs[1]
        R.append((ib[0], 0, m, 0, k))
        if int(d["flags"]) & F_ADD_RESIDUAL:
            R.append((ib[2], 0, m, c0, c0 + cn))
        Wr.append((ob, 0, m, c0, c0 + cn))
        if int(d["flags"]) & F_ARGMAX_EPI:
            # the tile writes its (max, index) pairs into column reserved[4]
            Wr.append((rs[3], rs[4], rs[4] + 1, 0, m))
    elif op in (OP_ATT_APPEND, OP_ATT_PARTIAL, OP_ATT_COMBINE):
        s, g, Hkv, T = rs[0], rs[1], rs[2] & 0xFFFF, (rs[2] >> 16) + 1
        D, Hq, cap = n, k, kv
        G = Hq // Hkv
        row = s * Hkv + g
        q0, q1 = s * T, s * T + T           # the sequence's activation rows
        if op == OP_ATT_APPEND:
            if step >= T:
                raise ValidationError(f"append with step {step} >= T {T}")
            r = s * T + step
            R += [(ib[0], r, r + 1, Hq * D + g * D, Hq * D + (g + 1) * D),
                  (ib[0], r, r + 1, (Hq + Hkv) * D + g * D, (Hq + Hkv) * D + (g + 1) * D),
                  (BUF_STATE, s, s + 1, 0, 2)]
            # token t's row: columns [cap*D + t*D, cap*D + (t+1)*D) of the (s, g) block
            a0 = cap * D + step * D
            Wr += [(ib[1], row, row + 1, a0, a0 + D), (ib[2], row, row + 1, a0, a0 + D)]
        elif op == OP_ATT_PARTIAL:
            c, P = rs[3] & 0xFFFF, rs[3] >> 16
            assert c < P
            slot = rs[4] + c
            # q, k and v of the group from qkv; the cache rows of earlier
            # steps (columns [0, cap*D)), carried in from the previous step
            R += [(ib[0], q0, q1, g * G * D, (g + 1) * G * D),
                  (ib[0], q0, q1, Hq * D + g * D, Hq * D + (g + 1) * D),
                  (ib[0], q0, q1, (Hq + Hkv) * D + g * D, (Hq + Hkv) * D + (g + 1) * D),
                  (ib[1], row, row + 1, 0, cap * D, True), (ib[2], row, row + 1, 0, cap * D, True),
                  (BUF_STATE, s, s + 1, 0, 2)]
            Wr.append((ob, slot, slot + 1, 0, T * G * (D + 2)))
        else:
            P, base = rs[3], rs[4]
            R.append((ib[0], base, base + P, 0, T * G * (D + 2)))
            R += [(ib[1], row, row + 1, cap * D, cap * D + T * D),
                  (ib[2], row, row + 1, cap * D, cap * D + T * D)]
            Wr.append((ob, q0, q1, g * G * D, (g + 1) * G * D))
    elif op == OP_SAMPLE:
        s, T = rs[0], rs[1] + 1
        last = s * T + T - 1
        R += [(ib[0], 0, k, last, last + 1), (BUF_STATE, s, s + 1, 0, 2)]
        if T > 1:
            R.append((ib[1], s, s + 1, 0, T))
        Wr += [(ob, s, s + 1, 0, kv), (BUF_STATE, s, s + 1, 0, 2)]
    else:
        raise ValidationError(f"unknown op_id {op}")
    if op not in (OP_MEMCPY, OP_ATT_APPEND) and step != 0:
        raise ValidationError(f"op {op} with step {step}: only per-token tasks carry a step")
    return R, Wr


def _covered(intervals, c0, c1) -> bool:
    cur = c0
    for a, b in sorted(intervals):
        if a > cur:
            return False
        cur = max(cur, b)
        if cur >= c1:
            return True
    return cur >= c1


def validate(tasks: np.ndarray, edges: np.ndarray, check_hazards: bool = True) -> dict:
    """Raise ValidationError on the first violated property; return stats."""
    N = len(tasks)
    deps = tasks["remaining_deps"].astype(np.int64)
    cnt = tasks["num_dependents"].astype(np.int64)
    off = tasks["dependents_offset"].astype(np.int64)
    if int(cnt.sum()) != len(edges):
        raise ValidationError("edge array length != sum of num_dependents")
    expect_off = np.concatenate([[0], np.cumsum(cnt)[:-1]]) if N else cnt
    if not np.array_equal(off, expect_off):
        raise ValidationError("dependents_offset is not the exclusive prefix sum")
    parents = [[] for _ in range(N)]
    for t in range(N):
        ch = edges[off[t]: off[t] + cnt[t]].astype(np.int64)
        if len(ch) and (ch.min() <= t):
            raise ValidationError(f"task {t} has an edge to an earlier task")
        if len(ch) > 1 and not np.all(np.diff(ch) > 0):
            raise ValidationError(f"task {t} children not strictly ascending")
        for c in ch:
            parents[int(c)].append(t)
    for t in range(N):
        if len(parents[t]) != deps[t]:
            raise ValidationError(f"task {t}: remaining_deps {deps[t]} != {len(parents[t])} parents")
    level = np.zeros(N, dtype=np.int64)
    for t in range(N):
        if parents[t]:
            level[t] = 1 + max(level[p] for p in parents[t])
    acc = [task_accesses(tasks[t]) for t in range(N)]

    # read coverage
    writes_by_buf = defaultdict(list)
    for t in range(N):
        for (b, r0, r1, c0, c1) in acc[t][1]:
            writes_by_buf[b].append((t, r0, r1, c0, c1))
    for t in range(N):
        for rd in acc[t][0]:
            b, r0, r1, c0, c1 = rd[:5]
            carried = len(rd) > 5 and rd[5]
            ws = writes_by_buf.get(b)
            if carried or b == BUF_STATE or not ws or min(w[0] for w in ws) >= t:
                continue      # carried in from the previous step (state, old KV rows) or external
            for r in range(r0, r1):
                iv = [(a0, a1) for (wt, q0, q1, a0, a1) in ws if wt < t and q0 <= r < q1]
                if not _covered(iv, c0, c1):
                    raise ValidationError(f"task {t} reads buf {b} row {r} [{c0},{c1}) "
                                          f"not covered by earlier writes")
    stats = dict(tasks=N, edges=len(edges), levels=int(level.max()) + 1 if N else 0)
    if not check_hazards:
        return stats

    # ancestry bitsets (python ints) in topological order
    anc = [0] * N
    for t in range(N):
        a = 0
        for p in parents[t]:
            a |= anc[p] | (1 << p)
        anc[t] = a

    def ordered(a, b):
        lo, hi = (a, b) if a < b else (b, a)
        return (anc[hi] >> lo) & 1 == 1

    by_buf = defaultdict(list)
    for t in range(N):
        for rd in acc[t][0]:
            b, r0, r1, c0, c1 = rd[:5]
            by_buf[b].append((t, r0, r1, c0, c1, False))
        for (b, r0, r1, c0, c1) in acc[t][1]:
            by_buf[b].append((t, r0, r1, c0, c1, True))
    for b, lst in by_buf.items():
        ws = [x for x in lst if x[5]]
        for (wt, a0, a1, b0, b1, _) in ws:
            for (t, r0, r1, c0, c1, isw) in lst:
                if t == wt or not (a0 < r1 and r0 < a1 and b0 < c1 and c0 < b1):
                    continue
                if not ordered(wt, t):
                    kind = "write/write" if isw else "read/write"
                    raise ValidationError(f"{kind} race on buf {b}: tasks {wt} and {t}")
                if level[wt] == level[t]:
                    raise ValidationError(f"same-level tasks {wt},{t} touch buf {b}")
    return stats


def levels(tasks: np.ndarray, edges: np.ndarray) -> np.ndarray:
    """Level of every task: 0 without parents, else 1 + max parent level."""
    N = len(tasks)
    level = np.zeros(N, dtype=np.int64)
    cnt = tasks["num_dependents"].astype(np.int64)
    off = tasks["dependents_offset"].astype(np.int64)
    for t in range(N):
        for c in edges[off[t]: off[t] + cnt[t]]:
            level[c] = max(level[c], level[t] + 1)
    return level
