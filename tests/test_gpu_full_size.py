"""Parity at the benchmark's full widths: the 8B-shaped model (hidden 4096,
FFN 14336, 32/8 heads of 128, the full 128256-entry LM head) truncated to
one or two decoder layers, so that the float64 oracle finishes in seconds,
in the launch configuration the benchmark uses (one CTA per SM).

  - B = 1, KV 4096: the headline workload's tiles, partial chunking (19
    chunks per KV head) and LM head;
  - B = 8 with the ragged KV lengths of the batch-8 workload: tensor-core
    GEMV tiles at full width, one-wave chunking of a ragged batch;
  - B = 4, KV 32768, chunk 1024: the long-context workload's 32 partials per
    KV head and its combine.
"""
import dataclasses

import pytest

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import build_gpu, compare_step, compare_cache_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _compared_steps(w, steps, seed=0):
    dec = build_gpu(w, seed)
    W = NpWeights(w.model, seed)
    st = oracle_state(w, seed)
    compared = 0
    try:
        if w.B == 8:
            assert dec.graph.tensor_core_tiles() > 0, "batch 8 should take the tensor-core path"
        for _ in range(steps):
            pos_before = [int(p) for p in st.pos]
            dec.graph.step()
            code, task = dec.graph.status()
            assert code == 0, f"device status {code} at task {task}"
            res = of.decode_step(w.model, W, st)
            _, clear = compare_step(dec, res, st)
            compare_cache_rows(dec, st, pos_before)
            compared += 1
            if not clear:
                break
        return compared
    finally:
        dec.graph.close()


def _truncated(name, layers):
    base = synth.workload(name)
    m = dataclasses.replace(base.model, L=layers)
    return base, m


def test_8b_width_b1_two_layers():
    base, m = _truncated("8b", 2)
    w = synth.custom(m, base.B, base.kv_len, 2, chunk=base.chunk, name="8b_l2")
    n = _compared_steps(w, 2)
    assert n >= 1


def test_8b_width_ragged_b8_tensor_tiles():
    base, m = _truncated("8b_b8", 1)
    w = synth.custom(m, base.B, base.kv_len, 1, chunk=base.chunk, name="8b_b8_l1")
    n = _compared_steps(w, 1)
    assert n == 1


def test_8b_width_long_context_b4():
    base, m = _truncated("8b_long", 1)
    w = synth.custom(m, base.B, base.kv_len, 1, chunk=base.chunk, name="8b_long_l1")
    n = _compared_steps(w, 1)
    assert n == 1
