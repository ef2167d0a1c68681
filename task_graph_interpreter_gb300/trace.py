"""Chrome trace-event export of a traced decode step.

`mk_decode_step_ex(..., trace=1)` records per task the CTA, the SM and
%globaltimer stamps (dependency wait begun, body started, outputs complete)
plus marks inside the GEMV and PARTIAL bodies.  This module turns those
records into the trace-event JSON that chrome://tracing and Perfetto read:
one track per CTA, a "wait" slice for each dependency wait and a slice per
task body named by its op, so scheduling overhead (waits) and body time
can be told apart at a glance.
"""
from __future__ import annotations

import json

import numpy as np

from . import _lib as L

_OP_NAMES = {
    L.MK_OP_NOP: "nop", L.MK_OP_MEMCPY: "embed", L.MK_OP_GEMV: "gemv", L.MK_OP_RMSNORM: "rmsnorm",
    L.MK_OP_SAMPLE: "sample", L.MK_OP_ATTENTION_APPEND: "append", L.MK_OP_ATTENTION_PARTIAL: "partial",
    L.MK_OP_ATTENTION_COMBINE: "combine",
}
# the descriptor fields the names use (offsets of the 64-byte descriptor)
_DESC = np.dtype({"names": ["op_id", "flags", "n", "k"], "formats": ["<u2", "<u2", "<i4", "<i4"],
                  "offsets": [0, 6, 32, 36], "itemsize": 64})


def chrome_trace(records: np.ndarray, tasks_bytes: bytes, path: str | None = None) -> dict:
    """Trace-event dict for `records` (uint64 [N, 8] from mk_get_trace) of
    the tasks in `tasks_bytes` (mk_get_tasks); written to `path` as JSON if
    given.  Times are microseconds from the earliest wait stamp; tasks with
    no end stamp (not run) are left out."""
    rec = np.asarray(records, dtype=np.uint64).reshape(-1, 8)
    tasks = np.frombuffer(tasks_bytes, dtype=_DESC)
    if len(tasks) != len(rec):
        raise ValueError(f"{len(rec)} trace records for {len(tasks)} tasks")
    ran = rec[:, 3] != 0
    t0 = int(rec[ran, 1].min()) if ran.any() else 0
    us = lambda t: (int(t) - t0) / 1000.0
    events = []
    for i in np.nonzero(ran)[0]:
        r = rec[i]
        cta, smid = int(r[0]) >> 32, int(r[0]) & 0xFFFFFFFF
        op = int(tasks["op_id"][i])
        name = _OP_NAMES.get(op, f"op{op}")
        if op == L.MK_OP_GEMV:
            name += f" n={int(tasks['n'][i])} k={int(tasks['k'][i])}"
        if r[2] > r[1]:
            events.append({"name": "wait", "cat": "wait", "ph": "X", "ts": us(r[1]), "dur": (int(r[2]) - int(r[1])) / 1000.0,
                           "pid": 0, "tid": cta, "args": {"task": int(i)}})
        events.append({"name": name, "cat": "task", "ph": "X", "ts": us(r[2]),
                       "dur": max(int(r[3]) - int(r[2]), 0) / 1000.0, "pid": 0, "tid": cta,
                       "args": {"task": int(i), "sm": smid, "ring_waits": int(r[7])}})
        for j, mark in enumerate(("first slot ready", "slots consumed", "epilogue done")):
            if r[4 + j]:
                events.append({"name": mark, "cat": "mark", "ph": "i", "s": "t", "ts": us(r[4 + j]), "pid": 0,
                               "tid": cta, "args": {"task": int(i)}})
    out = {"traceEvents": events, "displayTimeUnit": "ns"}
    if path:
        with open(path, "w") as f:
            json.dump(out, f)
    return out
