"""Failure detection on the GPU without a GPU fault.

Each failure is made on the host: a descriptor patched before upload (one
dependency too many, an unknown op), or a state holding a token outside the
vocabulary.  Every device wait is bounded (20 ms here), so the kernel
returns, reports the failing task through mk_status, and the context stays
usable: the tests then run good steps on the same device.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import lowering as ol
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import compare_step

pytestmark = pytest.mark.gpu


def _graph(timeout_us=20000):
    from task_graph_interpreter_gb300.llama import build_llama_decode
    w = synth.custom(synth.TINY, 1, [128], 4, name="tiny4")
    weights, kc, vc, hist, state = synth.device_inputs(w, 0, "cuda")
    dec = build_llama_decode(w.model, w.B, w.kv_len, w.capacity, weights, kc, vc, hist, device="cuda",
                             wait_timeout_us=timeout_us)
    dec.graph.state.copy_(state)
    dec.graph.lower()
    return w, dec, state


def _patch(dec, task, **fields):
    from task_graph_interpreter_gb300 import _lib as L
    t = np.frombuffer(dec.graph.tasks_bytes(), dtype=ol.TASK_DTYPE).copy()
    for k, v in fields.items():
        t[task][k] = v
    L.mk_debug_patch_task(dec.graph.h, task, t[task].tobytes())


def _good_step_still_works():
    w, dec, _ = _graph()
    dec.graph.upload()
    dec.graph.step()
    code, _ = dec.graph.status()
    assert code == 0
    dec.graph.close()


def test_dependency_count_too_high_times_out_and_reports_task():
    from task_graph_interpreter_gb300 import _lib as L
    w, dec, _ = _graph()
    t = np.frombuffer(dec.graph.tasks_bytes(), dtype=ol.TASK_DTYPE)
    victim = int(np.nonzero(t["op_id"] == ol.OP_GEMV)[0][40])
    _patch(dec, victim, remaining_deps=int(t[victim]["remaining_deps"]) + 1)
    dec.graph.upload()
    dec.graph.step()
    code, task = dec.graph.status()
    # the first wait to expire is the victim's or that of a task downstream
    # of it that began waiting earlier
    assert code == L.MK_DEV_DEP_TIMEOUT
    assert task == victim or task in _descendants(t, dec.graph.edges(), victim)
    dec.graph.close()
    torch.cuda.synchronize()
    _good_step_still_works()


def _descendants(t, edges, root):
    seen, stack = set(), [root]
    while stack:
        p = stack.pop()
        o, n = int(t["dependents_offset"][p]), int(t["num_dependents"][p])
        for c in edges[o:o + n]:
            if int(c) not in seen:
                seen.add(int(c))
                stack.append(int(c))
    return seen


def test_unknown_op_is_reported():
    from task_graph_interpreter_gb300 import _lib as L
    w, dec, _ = _graph()
    _patch(dec, 5, op_id=42)
    dec.graph.upload()
    dec.graph.step()
    code, task = dec.graph.status()
    assert code == L.MK_DEV_BAD_OP and task == 5
    dec.graph.close()
    _good_step_still_works()


def test_token_outside_vocabulary_is_rejected_then_graph_recovers():
    from task_graph_interpreter_gb300 import _lib as L
    w, dec, state = _graph()
    dec.graph.upload()
    dec.graph.state[0, 0] = w.model.V + 5
    dec.graph.step()
    code, task = dec.graph.status()
    assert code == L.MK_DEV_BAD_INDEX and task == 0
    # the status read reset the counters: the same graph runs a good step
    dec.graph.state.copy_(state)
    dec.graph.step()
    assert dec.graph.status()[0] == 0
    W = NpWeights(w.model)
    st = oracle_state(w)
    res = of.decode_step(w.model, W, st)
    compare_step(dec, res, st)
    dec.graph.close()


def test_trace_respects_every_dependency():
    w, dec, _ = _graph()
    dec.graph.upload()
    dec.graph.step(trace=True)
    assert dec.graph.status()[0] == 0
    tr = dec.graph.trace()
    t = np.frombuffer(dec.graph.tasks_bytes(), dtype=ol.TASK_DTYPE)
    edges = dec.graph.edges()
    off, q = dec.graph.queues()
    N = len(t)
    assert np.all(tr[:, 2] >= tr[:, 1]) and np.all(tr[:, 3] >= tr[:, 2])
    cta = (tr[:, 0] >> 32).astype(np.int64)
    for c in range(len(off) - 1):
        assert np.all(cta[q[off[c]:off[c + 1]]] == c)
    from task_graph_interpreter_gb300 import _lib as L
    task_ll, buf_ll = L.mk_get_ll_plan(dec.graph.h, N, len(dec.graph.bufs) + 3)
    assert task_ll.any()
    # a decode combine polls its partials' tagged records
    polled = np.zeros(N, dtype=bool)
    polled[(t["op_id"] == ol.OP_ATT_COMBINE) & (buf_ll[t["in_buf"][:, 0]] == 1)] = True
    assert polled.any()
    for p in range(N):
        ch = edges[t["dependents_offset"][p]: t["dependents_offset"][p] + t["num_dependents"][p]]
        # a child waiting on counters starts after its parents end; one that
        # polls tagged pairs starts at once and ends only after its parents
        # began (their output is written before their end stamp)
        tagged = (task_ll[ch] == 1) | (polled[ch] & (t["op_id"][p] == ol.OP_ATT_PARTIAL))
        ctr = ch[~tagged]
        ll = ch[tagged]
        assert np.all(tr[ctr, 2] >= tr[p, 3]), f"a child of task {p} started before it ended"
        assert np.all(tr[ll, 3] >= tr[p, 2]), f"a tagged child of task {p} ended before it began"
    ev = dec.graph.chrome_trace()["traceEvents"]
    assert sum(e["cat"] == "task" for e in ev) == N
    dec.graph.close()


@pytest.mark.parametrize("B", [1, 8])
def test_steps_across_the_counter_and_tag_wrap(B):
    # Dependency counters and their targets (epoch x adds per step) are
    # uint32 and wrap after 2^32 / adds steps, and so does the step tag of
    # the tagged pairs.  Put the graph a step before the counter that gains
    # the most per step wraps (and the tag just before 2^32), then run steps
    # across both wraps: every step must still match the oracle (an unsigned
    # comparison would let waits pass early once a target wraps).
    from task_graph_interpreter_gb300 import _lib as L
    lens = [128, 5, 64, 128, 100, 17, 128, 90][:B]
    w = synth.custom(synth.TINY, B, lens, 5, name=f"tiny_wrap{B}")
    dec = build_gpu_wrap(w)
    n = len(dec.graph.tasks_bytes()) // 64
    _, _, _, sig, _ = L.mk_get_sync_plan(dec.graph.h, n)
    adds = int(np.bincount(sig.astype(np.int64)).max())
    epoch = (2 ** 32 - 1) // adds - 1          # (epoch + 2) * adds passes 2^32
    s = torch.cuda.current_stream().cuda_stream
    L.mk_debug_set_epoch(dec.graph.h, s, epoch, 2 ** 32 - 3)
    W = NpWeights(w.model, 0)
    st = oracle_state(w, 0)
    try:
        for _ in range(4):
            dec.graph.step()
            code, task = dec.graph.status()
            assert code == 0, f"device status {code} at task {task}"
            res = of.decode_step(w.model, W, st)
            _, clear = compare_step(dec, res, st)
            if not clear:
                break
    finally:
        dec.graph.close()


def build_gpu_wrap(w):
    from tests.gpu_common import build_gpu
    return build_gpu(w, 0, wait_timeout_us=200000)
