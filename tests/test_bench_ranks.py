"""bench.py's multi-rank aggregation on CPU: two gloo ranks (replicas, no
data-path collective) agree on the slowest rank's time and report the
whole-job throughput from it."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        assert bench.dist_env()[:2] == (rank, ws)
        local = 2.0 + rank          # rank 1 is the slow replica
        t = bench.reduce_max(local, ws)
        out[rank] = (t, bench.job_throughput(4, 10, t, ws))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_replicas():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == (3.0, 4 * 10 / 3.0 * 2)


def test_single_rank_is_the_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25, 1) == 1.25
    assert bench.job_throughput(8, 64, 2.0, 1) == pytest.approx(256.0)


def test_bench_checks_the_timed_graph_is_a_whole_step():
    # the harness refuses a graph without every layer, the lm_head or SAMPLE
    import importlib.util
    import numpy as np
    import pytest
    import synth
    from oracle import lowering as ol
    from oracle.graph import llama_decode_spec
    from task_graph_interpreter_gb300 import _lib as L
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    w = synth.workload("1b")
    tasks, _ = ol.lower(llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, 152, col_align=4))
    bench.check_whole_step(tasks.tobytes(), w, L)
    no_sample = tasks[tasks["op_id"] != ol.OP_SAMPLE]
    with pytest.raises(RuntimeError):
        bench.check_whole_step(no_sample.tobytes(), w, L)
    one_layer_less = tasks[np.nonzero(tasks["op_id"] == ol.OP_ATT_COMBINE)[0][w.B * w.model.Hkv]:]
    with pytest.raises(RuntimeError):
        bench.check_whole_step(one_layer_less.tobytes(), w, L)

