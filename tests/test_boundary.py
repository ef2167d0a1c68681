"""Host-side tests of the C ABI (no GPU): symbols, lowering parity, errors.

The C++ lowering must emit exactly the bytes of the oracle's independent
lowering for every workload; nothing here dereferences a registered pointer,
so fake 256-byte-aligned addresses stand in for device memory.
"""
import re
import os

import numpy as np
import pytest

import synth
from oracle import lowering as ol
from oracle.graph import llama_decode_spec
from oracle.validate import validate

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from task_graph_interpreter_gb300 import build as _b
    _b()
    from task_graph_interpreter_gb300 import _lib
    _lib.lib()
    return _lib


def test_library_exports_every_declared_symbol(L):
    hdr = open(os.path.join(ROOT, "include", "mk.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    declared = set(re.findall(r"\b(mk_[a-z_]+)\s*\(", hdr))
    assert declared == set(L.EXPORTS)
    lib = L.lib()
    for name in declared:
        assert hasattr(lib, name), name


def _replay(L, spec, B, fuse=False, g_fused=[0]):
    """Feed an oracle graph spec to libmk through the C ABI (fake pointers);
    with fuse, run the library's RMS-norm fusion pass before lowering."""
    g = L.mk_graph_create(num_ctas=spec["num_ctas"], tiles_target=spec["tiles_target"],
                          col_align=spec["col_align"])
    base = 1 << 40
    L.mk_set_state(g, base, B)
    for i, (dt, rows, cols) in enumerate(spec["buffers"][3:], start=3):
        idx = L.mk_add_buffer(g, base + i * (1 << 24), dt, rows, cols)
        assert idx == i
    if spec.get("T", 1) > 1:
        L.mk_set_chunk(g, spec["T"], spec["tokens"])
    for op in spec["ops"]:
        k = op["kind"]
        if k == "embed":
            L.mk_add_embed(g, op["table"], op["out"], op["B"], op["H"])
        elif k == "matmul":
            L.mk_add_matmul(g, op["x"], op["w"], op["out"], op["aux"], op["pairs"], op["flags"],
                            op["m"], op["n"], op["k"], op["eps"])
        elif k == "attention":
            L.mk_add_attention(g, op["qkv"], op["k"], op["v"], op["out"], op["scratch"], op["B"],
                               op["Hq"], op["Hkv"], op["D"], op["capacity"], op["len0"], op["chunk"], 5e5)
        elif k == "sample":
            L.mk_add_sample(g, op["pairs"], op["history"], op["B"], op["V"], op["capacity"])
        elif k == "rmsnorm":
            L.mk_add_rmsnorm(g, op["x"], op["gamma"], op["residual"], op["out"], op["B"], op["H"], op["eps"])
    if fuse:
        g_fused[0] = L.mk_fuse_rmsnorm(g)
    L.mk_lower(g)
    return g


@pytest.mark.parametrize("name", synth.WORKLOADS)
@pytest.mark.parametrize("num_ctas,col_align", [(152, 16), (37, 16), (152, 4), (148, 1)])
def test_cpp_lowering_is_byte_identical_to_oracle(L, name, num_ctas, col_align):
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, num_ctas, col_align=col_align)
    tasks, edges = ol.lower(spec)
    g = _replay(L, spec, w.B)
    try:
        got = L.mk_get_tasks(g)
        assert len(got) == tasks.nbytes
        if got != tasks.tobytes():
            gt = np.frombuffer(got, dtype=ol.TASK_DTYPE)
            bad = int(np.nonzero(gt != tasks)[0][0])
            pytest.fail(f"descriptor {bad} differs:\n lib    {gt[bad]}\n oracle {tasks[bad]}")
        assert np.array_equal(L.mk_get_edges(g), edges)
        off, q = L.mk_get_queues(g)
        assert len(off) == num_ctas + 1 and off[0] == 0 and off[-1] == len(tasks)
        assert np.array_equal(np.sort(q), np.arange(len(tasks)))
        for c in range(num_ctas):
            qq = q[off[c]:off[c + 1]]
            assert np.all(np.diff(qq) > 0), "each CTA queue must be in topological order"
        _check_queues_deadlock_free(tasks, edges, off, q)
    finally:
        L.mk_destroy(g)


def _check_queues_deadlock_free(tasks, edges, off, q):
    """The dependency edges plus 'runs after' within each CTA queue form an
    acyclic graph: some task is always at the head of its queue with every
    parent done, so all co-resident CTAs finish."""
    N = len(tasks)
    succ = [[] for _ in range(N)]
    indeg = np.zeros(N, np.int64)
    for p in range(N):
        o, n = int(tasks["dependents_offset"][p]), int(tasks["num_dependents"][p])
        for c in edges[o:o + n]:
            succ[p].append(int(c))
            indeg[int(c)] += 1
    for c in range(len(off) - 1):
        qq = q[off[c]:off[c + 1]]
        for a, b in zip(qq[:-1], qq[1:]):
            succ[int(a)].append(int(b))
            indeg[int(b)] += 1
    ready = [t for t in range(N) if indeg[t] == 0]
    seen = 0
    while ready:
        t = ready.pop()
        seen += 1
        for c in succ[t]:
            indeg[c] -= 1
            if indeg[c] == 0:
                ready.append(c)
    assert seen == N, "CTA queues and dependencies form a cycle"


@pytest.mark.parametrize("name", ["tiny", "8b_b8", "8b_long"])
def test_scratch_size_matches_the_allocation(L, name):
    # the attention scratch and argmax pairs the spec allocates are exactly
    # the bytes the library asks for
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4)
    g = _replay(L, spec, w.B)
    try:
        for op in spec["ops"]:
            buf = op.get("scratch") if op["kind"] == "attention" else op.get("pairs") if op["kind"] == "matmul" else None
            if buf is None or buf == ol.NO_BUF:
                continue
            dt, rows, cols = spec["buffers"][buf]
            assert L.mk_scratch_size(g, buf) == rows * cols * (8 if dt == 4 else 4)   # MK_PAIR is 8 bytes
        with pytest.raises(L.MkError):
            L.mk_scratch_size(g, 3)   # the embedding table is neither
    finally:
        L.mk_destroy(g)


def test_cpp_lowering_validates(L):
    w = synth.workload("1b")
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152)
    g = _replay(L, spec, w.B)
    try:
        tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
        validate(tasks, L.mk_get_edges(g))
    finally:
        L.mk_destroy(g)


def test_worked_example_through_the_library(L):
    # the page's worked example: 3072 qkv columns over 8 tiles, 384 columns each
    g = L.mk_graph_create(num_ctas=8, tiles_target=8, col_align=16)
    try:
        assert L.mk_gemv_tiles(g, 3072) == 8
        L.mk_set_state(g, 1 << 40, 1)
        x = L.mk_add_buffer(g, (1 << 40) + (1 << 24), L.MK_F32, 1, 2048)
        wq = L.mk_add_buffer(g, (1 << 40) + (2 << 24), L.MK_BF16, 3072, 2048)
        y = L.mk_add_buffer(g, (1 << 40) + (3 << 24), L.MK_F32, 1, 3072)
        L.mk_add_matmul(g, x, wq, y, L.MK_NO_BUF, L.MK_NO_BUF, 0, 1, 3072, 2048, 0.0)
        L.mk_lower(g)
        t = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
        assert len(t) == 8
        assert list(t["reserved"][:, 0]) == [384 * i for i in range(8)]
        assert set(t["reserved"][:, 1]) == {384}
    finally:
        L.mk_destroy(g)


def test_errors_are_reported(L):
    with pytest.raises(L.MkError) as e:
        L.mk_graph_create(num_ctas=4, abi_version=99)
    assert e.value.code == L.MK_ERR_ABI
    g = L.mk_graph_create(num_ctas=4)
    try:
        with pytest.raises(L.MkError) as e:
            L.mk_add_buffer(g, 1 << 40, L.MK_F32, 1, 1)     # before the state
        assert e.value.code == L.MK_ERR_STATE
        L.mk_set_state(g, 1 << 40, 1)
        with pytest.raises(L.MkError) as e:
            L.mk_add_buffer(g, (1 << 40) + 8, L.MK_F32, 1, 1)  # misaligned
        assert e.value.code == L.MK_ERR_ARG
        x = L.mk_add_buffer(g, (1 << 40) + (1 << 24), L.MK_F32, 1, 256)
        w = L.mk_add_buffer(g, (1 << 40) + (2 << 24), L.MK_BF16, 64, 256)
        y = L.mk_add_buffer(g, (1 << 40) + (3 << 24), L.MK_F32, 1, 64)
        gm = L.mk_add_buffer(g, (1 << 40) + (4 << 24), L.MK_BF16, 1, 256)
        with pytest.raises(L.MkError) as e:   # both norm and residual: one aux slot
            L.mk_add_matmul(g, x, w, y, gm, L.MK_NO_BUF, L.MK_F_RMS_NORM_INPUT | L.MK_F_ADD_RESIDUAL,
                            1, 64, 256, 1e-5)
        assert e.value.code == L.MK_ERR_ARG
        with pytest.raises(L.MkError) as e:   # K mismatch with x
            L.mk_add_matmul(g, x, w, y, L.MK_NO_BUF, L.MK_NO_BUF, 0, 1, 64, 512, 0.0)
        assert e.value.code == L.MK_ERR_ARG
        with pytest.raises(L.MkError) as e:   # bad buffer index
            L.mk_add_matmul(g, 77, w, y, L.MK_NO_BUF, L.MK_NO_BUF, 0, 1, 64, 256, 0.0)
        assert e.value.code == L.MK_ERR_ARG
        with pytest.raises(L.MkError) as e:   # nothing to lower yet
            L.mk_lower(g)
        assert e.value.code == L.MK_ERR_STATE
        L.mk_add_matmul(g, x, w, y, gm, L.MK_NO_BUF, L.MK_F_RMS_NORM_INPUT, 1, 64, 256, 1e-5)
        with pytest.raises(L.MkError) as e:   # step before upload
            L.mk_decode_step(g, 0)
        assert e.value.code == L.MK_ERR_STATE
        L.mk_lower(g)
        with pytest.raises(L.MkError) as e:   # add after lower
            L.mk_add_matmul(g, x, w, y, gm, L.MK_NO_BUF, L.MK_F_RMS_NORM_INPUT, 1, 64, 256, 1e-5)
        assert e.value.code == L.MK_ERR_STATE
    finally:
        L.mk_destroy(g)


class _FakeTensor:
    """Stands in for a large device tensor when only its address and shape matter."""
    _next = 1 << 44

    def __init__(self, *shape, dtype=None):
        import torch
        self.shape = tuple(shape)
        self.dtype = dtype or torch.bfloat16
        n = int(np.prod(shape))
        self._ptr = _FakeTensor._next
        _FakeTensor._next += ((n * 4 + 4095) // 4096) * 4096 + 4096

    def numel(self):
        return int(np.prod(self.shape))

    def dim(self):
        return len(self.shape)

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return self._ptr


@pytest.mark.parametrize("name", ["tiny", "8b", "8b_b8"])
def test_product_builder_matches_oracle_graph(L, name):
    """The package's Llama builder registers buffers and ops in the same order
    as the oracle's graph spec, so its lowered bytes equal the oracle's."""
    import torch
    from task_graph_interpreter_gb300.llama import build_llama_decode
    w = synth.workload(name)
    m = w.model
    weights = {n: _FakeTensor(*shape) for (n, shape, _, _) in synth.weight_names(m)}
    kc = [_FakeTensor(w.B, m.Hkv, w.capacity, m.D) for _ in range(m.L)]
    vc = [_FakeTensor(w.B, m.Hkv, w.capacity, m.D) for _ in range(m.L)]
    hist = torch.zeros(w.B, w.capacity, dtype=torch.int32)
    dec = build_llama_decode(m, w.B, w.kv_len, w.capacity, weights, kc, vc, hist, chunk=w.chunk,
                             device="cpu", num_ctas=152)
    dec.graph.lower()
    spec = llama_decode_spec(m, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4)
    tasks, edges = ol.lower(spec)
    assert dec.graph.tasks_bytes() == tasks.tobytes()
    assert np.array_equal(dec.graph.edges(), edges)
    dec.graph.close()


def _check_sync_plan(tasks, edges, plan, ll=None):
    """When every wait of a task is satisfied, every parent of the task has
    signalled, and no wait can be satisfied without all its signallers.
    A task that reads tagged pairs (ll = (task_ll, buf_ll)) waits on no
    counter; each of its parents then writes its x or its residual, and
    that buffer carries pairs."""
    wait_off, wait, sig_off, sig, words = plan
    task_ll, buf_ll = ll if ll is not None else (np.zeros(len(tasks), np.uint8), None)
    N = len(tasks)
    parents = [set() for _ in range(N)]
    for p in range(N):
        o, n = int(tasks["dependents_offset"][p]), int(tasks["num_dependents"][p])
        for c in edges[o:o + n]:
            parents[int(c)].add(p)
    signallers = {}
    for p in range(N):
        got = [int(x) for x in sig[sig_off[p]:sig_off[p + 1]]]
        assert len(got) == len(set(got)), f"task {p} signals a counter twice"
        for c in got:
            assert c < words
            signallers.setdefault(c, set()).add(p)
    for t in range(N):
        covered = set()
        entries = wait[wait_off[t]:wait_off[t + 1]]
        if task_ll[t]:
            op = int(tasks["op_id"][t])
            assert op in (ol.OP_GEMV, ol.OP_ATT_PARTIAL, ol.OP_ATT_APPEND) and len(entries) == 0
            res = op == ol.OP_GEMV and int(tasks["flags"][t]) & ol.F_ADD_RESIDUAL
            x, aux = int(tasks["in_buf"][t][0]), int(tasks["in_buf"][t][2])
            assert buf_ll[x] and (not res or buf_ll[aux])
            for p in parents[t]:
                assert int(tasks["out_buf"][p]) in ((x, aux) if res else (x,)), f"task {t}: parent {p}"
            assert int(tasks["remaining_deps"][t]) == len(parents[t])
            continue
        # the last split of a K-split row block waits for its sibling splits
        # inside its body (the block's arrival counter), not through the plan;
        # a combine whose partials' records carry pairs polls those partials
        S, j = int(tasks["kv_len"][t]) >> 16, int(tasks["kv_len"][t]) & 0xFFFF
        deferred = set()
        scr = int(tasks["in_buf"][t][0])
        if int(tasks["op_id"][t]) == ol.OP_ATT_COMBINE and buf_ll is not None and buf_ll[scr]:
            deferred = {p for p in parents[t] if int(tasks["out_buf"][p]) == scr}
            assert all(int(tasks["op_id"][p]) == ol.OP_ATT_PARTIAL for p in deferred)
            assert len(deferred) == int(tasks["reserved"][t][3]), f"combine {t}: polls {len(deferred)} partials"
            assert int(tasks["reserved"][t][2]) >> 16 == 0 and int(tasks["reserved"][t][3]) <= 32
            covered = set(deferred)
        elif int(tasks["op_id"][t]) == ol.OP_GEMV and int(tasks["config_id"][t]) == 1 and S >= 2 and j == S - 1:
            deferred = set(range(t - (S - 1), t))
            assert deferred <= parents[t], f"task {t}: sibling splits are not its parents"
            for q in deferred:
                assert int(tasks["kv_len"][q]) == (q - (t - (S - 1))) | (S << 16)
                assert tuple(tasks["reserved"][q][:2]) == tuple(tasks["reserved"][t][:2])
            covered = set(deferred)
        assert len({int(c) for c, _ in entries}) == len(entries)
        for c, n in entries:
            c, n = int(c), int(n)
            assert c < words
            if c < N:
                assert c <= t, f"task {t} waits on the set counter of a later task {c}"
            who = signallers.get(c, set())
            assert len(who) == n, f"task {t}: counter {c} expects {n}, has {len(who)} signallers"
            assert who <= parents[t], f"task {t}: counter {c} is signalled by a non-parent"
            assert not (who & covered)
            covered |= who
        assert covered == parents[t], f"task {t}: waits cover {len(covered)} of {len(parents[t])} parents"
        assert sum(int(n) for _, n in entries) + len(deferred) == int(tasks["remaining_deps"][t])


@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_sync_plan_is_equivalent_to_the_edges(L, name):
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4)
    g = _replay(L, spec, w.B)
    try:
        tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
        plan = L.mk_get_sync_plan(g, len(tasks))
        ll = L.mk_get_ll_plan(g, len(tasks), len(spec["buffers"]))
        _check_sync_plan(tasks, L.mk_get_edges(g), plan, ll)
        polls = np.isin(tasks["op_id"], [ol.OP_GEMV, ol.OP_ATT_PARTIAL, ol.OP_ATT_APPEND])
        if w.B <= 2:
            # every GEMV, split-KV partial and cache append reads tagged pairs
            # (their inputs come from GEMV, COMBINE, embedding or norm tasks),
            # no other task does; every attention scratch carries pairs too
            # (decode combines poll their partials' records).  From three
            # activation rows the GEMVs run on tensor cores, without pairs
            assert np.all(ll[0][polls] == 1) and np.all(ll[0][~polls] == 0)
            comb = tasks[tasks["op_id"] == ol.OP_ATT_COMBINE]
            assert all(ll[1][int(b)] for b in comb["in_buf"][:, 0])
        else:
            assert not ll[0].any() and not ll[1].any()
        # a B = 1 hand-off between GEMVs costs one atomic per tile, not one per edge
        if w.B == 1 and name != "tiny":
            assert len(plan[3]) < len(L.mk_get_edges(g)) / 20
    finally:
        L.mk_destroy(g)


def _tagged_plan(L, spec, B):
    g = _replay(L, spec, B)
    try:
        tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE).copy()
        plan = L.mk_get_sync_plan(g, len(tasks))
        ll = L.mk_get_ll_plan(g, len(tasks), len(spec["buffers"]))
        _check_sync_plan(tasks, L.mk_get_edges(g), plan, ll)
        return tasks, ll
    finally:
        L.mk_destroy(g)


def test_tagged_plan_takes_standalone_norm_outputs(L):
    # RMSNORM bodies write pairs too: with standalone norms every GEMV and
    # attention reader still polls, and the norm outputs carry pairs
    w = synth.workload("1b")
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4, norms="standalone")
    tasks, (task_ll, buf_ll) = _tagged_plan(L, spec, w.B)
    norms = tasks["op_id"] == ol.OP_RMSNORM
    assert norms.any() and not task_ll[norms].any()
    assert all(buf_ll[int(o)] for o in tasks["out_buf"][norms])
    polls = np.isin(tasks["op_id"], [ol.OP_GEMV, ol.OP_ATT_PARTIAL, ol.OP_ATT_APPEND])
    assert np.all(task_ll[polls] == 1)


def test_tagged_plan_refuses_a_buffer_written_twice(L):
    # two matmuls writing one buffer: its readers could not tell the two
    # writes apart by the step tag, so the buffer carries no pairs and its
    # reader waits on counters
    g = L.mk_graph_create(num_ctas=16, tiles_target=16, col_align=4)
    base = 1 << 40
    try:
        L.mk_set_state(g, base, 1)
        H = 256
        x = L.mk_add_buffer(g, base + 1 * (1 << 24), L.MK_F32, 1, H)
        w1 = L.mk_add_buffer(g, base + 2 * (1 << 24), L.MK_BF16, H, H)
        w2 = L.mk_add_buffer(g, base + 3 * (1 << 24), L.MK_BF16, H, H)
        y = L.mk_add_buffer(g, base + 4 * (1 << 24), L.MK_F32, 1, H)
        z = L.mk_add_buffer(g, base + 5 * (1 << 24), L.MK_F32, 1, H)
        u = L.mk_add_buffer(g, base + 6 * (1 << 24), L.MK_F32, 1, H)
        L.mk_add_matmul(g, x, w1, y, ol.NO_BUF, ol.NO_BUF, 0, 1, H, H, 0.0)
        L.mk_add_matmul(g, y, w2, z, ol.NO_BUF, ol.NO_BUF, 0, 1, H, H, 0.0)   # reads y once written
        L.mk_add_matmul(g, z, w1, y, ol.NO_BUF, ol.NO_BUF, 0, 1, H, H, 0.0)   # writes y again
        L.mk_add_matmul(g, y, w2, u, ol.NO_BUF, ol.NO_BUF, 0, 1, H, H, 0.0)
        L.mk_lower(g)
        tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
        task_ll, buf_ll = L.mk_get_ll_plan(g, len(tasks), u + 1)
        assert buf_ll[z] == 1 and buf_ll[y] == 0
        reads_y = tasks["in_buf"][:, 0] == y
        reads_z = tasks["in_buf"][:, 0] == z
        assert not task_ll[reads_y].any() and task_ll[reads_z].all()
    finally:
        L.mk_destroy(g)


def test_sync_plan_follows_a_patched_dependency_count(L):
    w = synth.workload("tiny")
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 16, col_align=4)
    g = _replay(L, spec, w.B)
    try:
        tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE).copy()
        victim = int(np.nonzero(tasks["op_id"] == ol.OP_GEMV)[0][10])
        t = tasks[victim].copy()
        t["remaining_deps"] += 1
        L.mk_debug_patch_task(g, victim, t.tobytes())
        wait_off, wait, _, sig, _ = L.mk_get_sync_plan(g, len(tasks))
        entries = wait[wait_off[victim]:wait_off[victim + 1]]
        task_ll, _ = L.mk_get_ll_plan(g, len(tasks), len(spec["buffers"]))
        # a task reading tagged pairs counts only the surplus on a counter
        want = 1 if task_ll[victim] else int(t["remaining_deps"])
        assert sum(int(n) for _, n in entries) == want
        own = [(int(c), int(n)) for c, n in entries if int(c) < len(tasks)]
        assert own and own[0][1] > np.count_nonzero(sig == own[0][0]), "the extra dependency can never be met"
    finally:
        L.mk_destroy(g)



@pytest.mark.parametrize("name", ["tiny", "1b", "8b_b8"])
def test_standalone_rmsnorm_lowering_is_byte_identical(L, name):
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4, norms="standalone")
    tasks, edges = ol.lower(spec)
    validate(tasks, edges)
    assert np.count_nonzero(tasks["op_id"] == ol.OP_RMSNORM) == w.B * (2 * w.model.L + 1)
    g = _replay(L, spec, w.B)
    try:
        assert L.mk_get_tasks(g) == tasks.tobytes()
        assert np.array_equal(L.mk_get_edges(g), edges)
    finally:
        L.mk_destroy(g)


@pytest.mark.parametrize("name", ["tiny", "8b"])
def test_fusion_pass_matches_oracle_fusion_and_hand_flags(L, name):
    from oracle.graph import fuse_rmsnorm
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4, norms="standalone")
    fused, n = fuse_rmsnorm(spec)
    assert n == 2 * w.model.L + 1
    tasks, edges = ol.lower(fused)
    count = [0]
    g = _replay(L, spec, w.B, fuse=True, g_fused=count)
    try:
        assert count[0] == n
        assert L.mk_get_tasks(g) == tasks.tobytes()
        assert np.array_equal(L.mk_get_edges(g), edges)
    finally:
        L.mk_destroy(g)
    # the folded graph is the hand-flagged one up to buffer numbering
    hand, hedges = ol.lower(llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4))
    assert len(hand) == len(tasks) and np.array_equal(hedges, edges)
    for f in ("op_id", "config_id", "flags", "remaining_deps", "num_dependents", "dependents_offset", "m", "n",
              "k", "kv_len"):
        assert np.array_equal(hand[f], tasks[f]), f
    gemv = hand["op_id"] == ol.OP_GEMV
    assert np.array_equal(hand["reserved"][gemv][:, [0, 1, 2, 4]], tasks["reserved"][gemv][:, [0, 1, 2, 4]])


def test_fusion_pass_leaves_norms_with_other_readers(L):
    """A norm whose output is also a residual (or that carries a residual)
    stays standalone."""
    g = L.mk_graph_create(num_ctas=8, tiles_target=8, col_align=16)
    try:
        base = 1 << 40
        L.mk_set_state(g, base, 1)
        nb = iter(range(1, 100))
        add = lambda dt, r, c: L.mk_add_buffer(g, base + next(nb) * (1 << 24), dt, r, c)
        x, gm = add(L.MK_F32, 1, 256), add(L.MK_BF16, 1, 256)
        xn, w = add(L.MK_F32, 1, 256), add(L.MK_BF16, 256, 256)
        y, z = add(L.MK_F32, 1, 256), add(L.MK_F32, 1, 256)
        L.mk_add_rmsnorm(g, x, gm, L.MK_NO_BUF, xn, 1, 256, 1e-5)
        L.mk_add_matmul(g, xn, w, y, L.MK_NO_BUF, L.MK_NO_BUF, 0, 1, 256, 256, 0.0)
        L.mk_add_matmul(g, y, w, z, xn, L.MK_NO_BUF, L.MK_F_ADD_RESIDUAL, 1, 256, 256, 0.0)
        assert L.mk_fuse_rmsnorm(g) == 0
        L.mk_lower(g)
        t = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
        assert (t["op_id"] == ol.OP_RMSNORM).sum() == 1
    finally:
        L.mk_destroy(g)


def test_chrome_trace_export_from_records(L, tmp_path):
    # synthetic records for the tiny graph: one task after another on two CTAs
    import json
    from task_graph_interpreter_gb300.trace import chrome_trace
    w = synth.workload("tiny")
    tasks, _ = ol.lower(llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 2, col_align=4))
    N = len(tasks)
    rec = np.zeros((N, 8), np.uint64)
    t = 1_000_000
    for i in range(N):
        rec[i, 0] = ((i % 2) << 32) | (10 + i % 2)
        rec[i, 1], rec[i, 2], rec[i, 3] = t, t + 500, t + 2500   # 0.5 us wait, 2 us body
        if tasks["op_id"][i] == ol.OP_GEMV:
            rec[i, 4] = t + 700
        t += 3000
    rec[N - 1, 3] = 0                                            # a task that did not run
    out = chrome_trace(rec, tasks.tobytes(), str(tmp_path / "step.json"))
    ev = json.load(open(tmp_path / "step.json"))["traceEvents"]
    assert ev == out["traceEvents"]
    bodies = [e for e in ev if e["cat"] == "task"]
    waits = [e for e in ev if e["cat"] == "wait"]
    assert len(bodies) == N - 1 and len(waits) == N - 1
    assert bodies[0]["ts"] == 0.5 and bodies[0]["dur"] == 2.0 and waits[0]["ts"] == 0.0
    assert {e["tid"] for e in bodies} == {0, 1}
    assert any(e["name"].startswith("gemv n=") for e in bodies)
    assert sum(e["cat"] == "mark" for e in ev) == int(np.count_nonzero(tasks["op_id"][:N - 1] == ol.OP_GEMV))
    with pytest.raises(ValueError):
        chrome_trace(rec[:-1], tasks.tobytes())


@pytest.mark.parametrize("name,B,T", [("tiny", 1, 4), ("tiny", 2, 4), ("tiny", 3, 2), ("1b", 2, 4), ("tiny", 8, 1),
                                      ("8b", 2, 4), ("8b_long", 2, 2)])
@pytest.mark.parametrize("norms", ["fused", "standalone"])
def test_chunk_step_lowering_is_byte_identical_and_valid(L, name, B, T, norms):
    # chunk steps (T tokens per sequence): the C++ lowering and the oracle's
    # independent lowering agree byte for byte, and the DAG validates
    w = synth.workload(name)
    lens = list(w.kv_len[:B]) + [w.kv_len[0]] * max(0, B - len(w.kv_len))
    cap = max(lens) + 2 * T + 1
    spec = llama_decode_spec(w.model, B, lens, cap, w.chunk, 152, col_align=4, norms=norms, T=T)
    tasks, edges = ol.lower(spec)
    g = _replay(L, spec, B)
    try:
        assert L.mk_get_tasks(g) == tasks.tobytes()
        assert np.array_equal(L.mk_get_edges(g), edges)
    finally:
        L.mk_destroy(g)
    if name == "tiny":
        validate(tasks, edges)
    else:
        validate(tasks, edges, check_hazards=False)
    # per-token tasks carry their token index; T - 1 rides in the fields the spec names
    emb = tasks[tasks["op_id"] == ol.OP_MEMCPY]
    app = tasks[tasks["op_id"] == ol.OP_ATT_APPEND]
    assert sorted(emb["step"].tolist()) == sorted(list(range(T)) * B)
    assert set(app["step"].tolist()) == set(range(T))
    assert np.all(app["reserved"][:, 2] >> 16 == T - 1)
    assert np.all(tasks[tasks["op_id"] == ol.OP_SAMPLE]["reserved"][:, 1] == T - 1)


def test_chunk_step_validator_catches_a_missing_causal_edge(L):
    # the combine of a chunk step must wait for every token's append: drop
    # one append -> combine edge and the validator reports the race
    w = synth.workload("tiny")
    spec = llama_decode_spec(w.model, 1, [128], 140, 0, 16, col_align=4, T=4)
    tasks, edges = ol.lower(spec)
    validate(tasks, edges)
    app = [int(i) for i in np.nonzero(tasks["op_id"] == ol.OP_ATT_APPEND)[0] if tasks["step"][i] == 3]
    t = app[0]
    off, cnt = int(tasks["dependents_offset"][t]), int(tasks["num_dependents"][t])
    kids = [int(c) for c in edges[off:off + cnt]]
    comb = [c for c in kids if tasks["op_id"][c] == ol.OP_ATT_COMBINE][0]
    bad_t = tasks.copy()
    keep = [c for c in kids if c != comb]
    new_edges = np.concatenate([edges[:off], np.array(keep, dtype=np.uint32), edges[off + cnt:]])
    bad_t["num_dependents"][t] = cnt - 1
    bad_t["dependents_offset"][t + 1:] -= 1
    bad_t["remaining_deps"][comb] -= 1
    with pytest.raises(AssertionError):
        validate(bad_t, new_edges)


def test_chunk_step_errors(L):
    g = L.mk_graph_create(num_ctas=8)
    try:
        base = 1 << 40
        L.mk_set_state(g, base, 2)
        tok = L.mk_add_buffer(g, base + (1 << 24), L.MK_I32, 2, 4)
        bad = L.mk_add_buffer(g, base + (2 << 24), L.MK_I32, 2, 5)
        with pytest.raises(L.MkError):
            L.mk_set_chunk(g, 4, bad)          # not [B, T]
        with pytest.raises(L.MkError):
            L.mk_set_chunk(g, 1, tok)          # T < 2
        bigtok = L.mk_add_buffer(g, base + (3 << 24), L.MK_I32, 2, 8)
        with pytest.raises(L.MkError):
            L.mk_set_chunk(g, 8, bigtok)       # B * T > 8
        L.mk_set_chunk(g, 4, tok)
        with pytest.raises(L.MkError) as e:
            L.mk_set_chunk(g, 4, tok)          # once
        assert e.value.code == L.MK_ERR_STATE
    finally:
        L.mk_destroy(g)


@pytest.mark.parametrize("name,num_ctas", [("tiny", 152), ("tiny", 16), ("8b_b8", 152)])
def test_ksplit_lowering_validates(L, name, num_ctas):
    # batch-8 GEMVs with narrow per-SM tiles become K-split row blocks: the
    # DAG (splits -> the block's last split -> readers) validates, each
    # block's splits cover K exactly once in order, and its last split is
    # the only writer of the block's outputs
    w = synth.workload(name) if name != "tiny" else synth.custom(synth.TINY, 8, [128] * 8, 2, name="tiny8")
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, num_ctas, col_align=4)
    tasks, edges = ol.lower(spec)
    validate(tasks, edges, check_hazards=(name == "tiny"))
    g = _replay(L, spec, w.B)
    try:
        assert L.mk_get_tasks(g) == tasks.tobytes()
    finally:
        L.mk_destroy(g)
    gemv = tasks[tasks["op_id"] == ol.OP_GEMV]
    split = gemv[(gemv["kv_len"] >> 16) >= 2]
    assert len(split) > 0
    K = {}
    for d in split:
        key = (int(d["in_buf"][1]), int(d["reserved"][0]), int(d["in_buf"][0]))
        K.setdefault(key, []).append((int(d["kv_len"]) & 0xFFFF, int(d["reserved"][3]) & 0xFFFF,
                                      int(d["reserved"][3]) >> 16, int(d["k"]), int(d["kv_len"]) >> 16))
    for key, parts in K.items():
        parts.sort()
        S = parts[0][4]
        assert [p[0] for p in parts] == list(range(S))
        col = 0
        for (_, k0, kn, k, _) in parts:
            assert k0 == col and kn % 64 == 0 and kn > 0
            col += kn
        assert col == parts[0][3]
    # every split tile of an op fits the tile target; rows per block <= 256 / seg
    assert np.all(split["reserved"][:, 1] * np.where(split["flags"] & ol.F_SILU_MUL, 2, 1) <= 256)


def test_tagged_scratch_only_for_polling_combines(L):
    # a decode combine polls its partials' tagged records only up to 32
    # partials: 128 keys in chunks of 4 (32 partials) tag the scratch, in
    # chunks of 3 (43) they do not, and neither does a chunk step
    w = synth.workload("tiny")
    for chunk, T, tagged in ((4, 1, True), (3, 1, False), (4, 2, False)):
        spec = llama_decode_spec(w.model, 1, [128], 140, chunk, 16, col_align=4, T=T)
        g = _replay(L, spec, 1)
        try:
            tasks = np.frombuffer(L.mk_get_tasks(g), dtype=ol.TASK_DTYPE)
            task_ll, buf_ll = L.mk_get_ll_plan(g, len(tasks), len(spec["buffers"]))
            comb = tasks[tasks["op_id"] == ol.OP_ATT_COMBINE]
            assert all(bool(buf_ll[int(b)]) == tagged for b in comb["in_buf"][:, 0]), (chunk, T)
            _check_sync_plan(tasks, L.mk_get_edges(g), L.mk_get_sync_plan(g, len(tasks)), (task_ll, buf_ll))
        finally:
            L.mk_destroy(g)


# The largest dynamic shared memory a CTA may opt in to on sm_100-class
# GPUs (227 KB); a kilobyte is left for the kernel's static shared words.
_SMEM_OPT_IN = 227 * 1024


@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_kernel_shared_memory_fits_one_cta_per_sm(L, name):
    """The interpreter's shared memory at its full ring (one or two rows:
    ring, control block, task records, scratch; three to eight: also the
    tensor-core activation tiles) fits the opt-in limit, so the ring is
    never shortened at launch on these workloads."""
    w = synth.workload(name)
    spec = llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152)
    g = _replay(L, spec, w.B)
    try:
        smem, threads, stages = L.mk_kernel_info(g)
    finally:
        L.mk_destroy(g)
    assert threads == 384  # two consumer warpgroups and the producer warpgroup
    assert stages == 5  # ring slots of 32 KB
    assert stages * 32768 < smem <= _SMEM_OPT_IN - 1024
