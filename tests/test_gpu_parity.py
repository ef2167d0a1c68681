"""CUDA path vs the float64 oracle, element by element, through the C ABI.

Sizes: the tiny model (several tiles per op and a short last tile), a
ragged batch with empty and one-key chunks (the batch-3 kernel class), and
the 1B-shaped model at full size in the launch configuration the benchmark
uses (one CTA per SM).
"""
import numpy as np
import pytest
import torch

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import build_gpu, compare_step, compare_cache_rows

pytestmark = pytest.mark.gpu

MODES = {"mega": 0, "per_op": 1, "per_op_graph": 2, "levels": 3, "per_op_pdl": 4}


def _run_and_compare(w, steps, mode="mega", num_ctas=0, seed=0, check_cache=True, norms="fused"):
    from task_graph_interpreter_gb300 import _lib as L
    dec = build_gpu(w, seed, num_ctas, norms=norms)
    if norms == "fuse_pass":
        assert dec.fused_norms == 2 * w.model.L + 1
    W = NpWeights(w.model, seed)
    st = oracle_state(w, seed)
    clear_steps = 0
    try:
        for i in range(steps):
            pos_before = [int(p) for p in st.pos]
            dec.graph.step(MODES[mode])
            code, task = dec.graph.status()
            assert code == 0, f"device status {code} at task {task}"
            res = of.decode_step(w.model, W, st)
            dmax, clear = compare_step(dec, res, st)
            if check_cache:
                compare_cache_rows(dec, st, pos_before)
            hist = dec.history.tensor.cpu().numpy()
            for s in range(w.B):
                assert hist[s, pos_before[s] + 1] == dec.graph.state[s, 0].item()
            if not clear:
                break                   # a near-tie: later inputs may differ legitimately
            clear_steps += 1
    finally:
        dec.graph.close()
    return clear_steps


def test_tiny_one_step_megakernel():
    assert _run_and_compare(synth.workload("tiny"), 1) == 1


def test_capacity_is_reported_not_overrun():
    # the tiny workload has room for exactly one generated token
    dec = build_gpu(synth.workload("tiny"))
    try:
        dec.graph.step()
        assert dec.graph.status()[0] == 0
        dec.graph.step()
        from task_graph_interpreter_gb300 import _lib as L
        code, task = dec.graph.status()
        assert code == L.MK_DEV_CAPACITY
    finally:
        dec.graph.close()


@pytest.mark.parametrize("mode", ["per_op", "per_op_graph", "levels", "per_op_pdl"])
def test_tiny_other_modes(mode):
    w = synth.custom(synth.TINY, 1, [128], 2, name="tiny2")
    assert _run_and_compare(w, 2, mode) >= 1


def test_tiny_multi_step_greedy_tokens():
    w = synth.custom(synth.TINY, 1, [128], 8, name="tiny8")
    assert _run_and_compare(w, 8) >= 6


def test_ragged_batch_with_empty_and_single_key_chunks():
    # B = 3 uses the batch-3..8 kernel; kv lengths 0, 4 and 70 with one-key
    # chunks give P = 1, 4, 70 partials, some of them empty as keys grow
    w = synth.custom(synth.TINY, 3, [0, 4, 70], 3, chunk=1, name="tiny_ragged")
    assert _run_and_compare(w, 3) >= 2


def test_batch_two_and_few_ctas():
    w = synth.custom(synth.TINY, 2, [33, 128], 2, name="tiny_b2")
    assert _run_and_compare(w, 2, num_ctas=7) >= 1


def test_modes_are_bitwise_identical_and_deterministic():
    w = synth.workload("tiny")
    outs = []
    for mode in ("mega", "mega", "per_op", "levels", "per_op_pdl"):
        dec = build_gpu(w)
        dec.graph.step(MODES[mode])
        assert dec.graph.status()[0] == 0
        outs.append((dec.logits.tensor.cpu().clone(), [h.tensor.cpu().clone() for h in dec.hidden]))
        dec.graph.close()
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0])
        for a, b in zip(o[1], outs[0][1]):
            assert torch.equal(a, b)


def test_modes_interleaved_on_one_graph():
    # megakernel steps write and poll tagged pairs, the other modes do not:
    # pairs left by an earlier megakernel step (or by none) must never pass
    # for the current one, so every step still matches the oracle
    w = synth.custom(synth.TINY, 2, [40, 128], 6, name="tiny_mix")
    dec = build_gpu(w)
    W = NpWeights(w.model, 0)
    st = oracle_state(w, 0)
    try:
        for mode in ("mega", "per_op", "mega", "levels", "per_op_pdl", "mega"):
            dec.graph.step(MODES[mode])
            code, task = dec.graph.status()
            assert code == 0, f"{mode}: device status {code} at task {task}"
            res = of.decode_step(w.model, W, st)
            _, clear = compare_step(dec, res, st)
            if not clear:
                break
    finally:
        dec.graph.close()


@pytest.mark.slow
def test_1b_full_size_two_steps():
    w = synth.custom(synth.LLAMA_1B, 1, [1024], 2, name="1b2")
    assert _run_and_compare(w, 2, check_cache=False) >= 1


@pytest.mark.parametrize("norms", ["standalone", "fuse_pass"])
def test_standalone_and_pass_fused_rmsnorm(norms):
    # standalone RMSNORM tasks (one per sequence, batch 2) and the same graph
    # after the fusion pass both match the oracle
    w = synth.custom(synth.TINY, 2, [40, 128], 3, name="tiny_norms")
    assert _run_and_compare(w, 3, norms=norms) >= 2


def test_tiny_long_chunks_take_tensor_core_partials():
    # chunks of 1024 keys (eight blocks of 128): the split-KV partials run on
    # tensor cores (score MMAs on K blocks brought by TMA, P V on CUDA
    # cores), at head dim 64; a short sequence keeps single-block chunks
    w = synth.custom(synth.TINY, 3, [2000, 1100, 90], 3, chunk=1024, name="tiny_long_chunks")
    assert _run_and_compare(w, 3) >= 2


@pytest.mark.parametrize("F,B", [(1792, 1), (1792, 2), (768, 1), (5376, 1)])
def test_ffn_widths_of_every_gemv_slot_geometry(F, B):
    # the down projection's K = F picks the GEMV's k-segment and warp layout:
    # 1792 = 7 x 256 (seven 16-byte pieces per lane, one warp column: 8 rows
    # per slot are covered, not the 9 that would fit), 768 (three 256-column
    # k-segments), 5376 (three 1792-column k-segments); B = 2 takes the
    # single-piece layout
    import dataclasses
    m = dataclasses.replace(synth.TINY, F=F, name=f"tiny_f{F}")
    w = synth.custom(m, B, [100, 37][:B], 3, name=f"tiny_f{F}_b{B}")
    assert _run_and_compare(w, 2) >= 1


@pytest.mark.parametrize("chunk", [5, 4, 3])
def test_combines_polling_one_and_two_groups_of_partials(chunk):
    # 128 cached keys in chunks of 5, 4 and 3: 26, 32 and 43 partials per
    # (sequence, KV head).  Up to 32 the decode combine polls its partials'
    # tagged records (two load groups past 16); past 32 the scratch carries
    # no pairs and the combine waits for its partials through counters
    w = synth.custom(synth.TINY, 1, [128], 3, chunk=chunk, name=f"tiny_c{chunk}")
    assert _run_and_compare(w, 2) >= 1
