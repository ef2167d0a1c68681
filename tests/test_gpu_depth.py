"""Parity at the workloads' real depth and over many greedy steps.

The float64 oracle and the CUDA path run the same seeded model, and every
step is compared: logits (max |delta| and cosine), every layer's hidden
state (relative L2), the sampled token (exact unless the oracle's top-2
margin is inside the error bound), the history, the positions and the KV
rows appended to every layer's caches.

  - the Llama-3.2-1B-shaped model at all 16 layers for 32 greedy steps
    (error build-up over depth and over a long greedy run);
  - the Llama-3-8B-shaped model at all 32 layers for 2 steps;
  - batches of 5 and 7 (tensor-core tiles with rows past the batch zero)
    on the tiny model and at 1B width;
  - the ragged batch of 8 (tensor-core GEMV tiles) at 8B width, 2 layers,
    over 4 steps.
"""
import dataclasses

import pytest

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import build_gpu, compare_step, compare_cache_rows

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _run(w, steps, seed=0, check_cache=True):
    """Steps compared before the first near-tie (or all of them)."""
    dec = build_gpu(w, seed)
    W = NpWeights(w.model, seed)
    st = oracle_state(w, seed)
    compared = 0
    try:
        for _ in range(steps):
            pos_before = [int(p) for p in st.pos]
            dec.graph.step()
            code, task = dec.graph.status()
            assert code == 0, f"device status {code} at task {task}"
            res = of.decode_step(w.model, W, st)
            _, clear = compare_step(dec, res, st)
            if check_cache:
                compare_cache_rows(dec, st, pos_before)
            hist = dec.history.tensor.cpu().numpy()
            for s in range(w.B):
                assert hist[s, pos_before[s] + 1] == int(st.token[s]) or not clear
            compared += 1
            if not clear:
                break
        return compared
    finally:
        dec.graph.close()


def _layers(model, L):
    return dataclasses.replace(model, L=L)


def test_1b_all_layers_32_greedy_steps():
    w = synth.custom(synth.LLAMA_1B, 1, [1024], 32, name="1b_32")
    assert _run(w, 32) >= 24


def test_8b_all_layers_two_steps():
    w = synth.custom(synth.LLAMA_8B, 1, [4096], 2, name="8b_2")
    assert _run(w, 2) >= 1


@pytest.mark.parametrize("B", [5, 7])
def test_tiny_batch_5_and_7(B):
    lens = [128, 3, 77, 40, 128, 9, 100][:B]
    w = synth.custom(synth.TINY, B, lens, 3, name=f"tiny_b{B}")
    assert _run(w, 3) >= 2


def test_1b_width_batch_5_two_layers():
    lens = [1024, 700, 513, 1000, 64]
    w = synth.custom(_layers(synth.LLAMA_1B, 2), 5, lens, 2, name="1b_b5_l2")
    assert _run(w, 2) >= 1


def test_1b_all_layers_batch_7():
    lens = [1024, 900, 128, 1024, 333, 777, 1]
    w = synth.custom(synth.LLAMA_1B, 7, lens, 2, name="1b_b7")
    assert _run(w, 2) >= 1


def test_8b_width_ragged_b8_two_layers_four_steps():
    base = synth.workload("8b_b8")
    w = synth.custom(_layers(base.model, 2), base.B, base.kv_len, 4, chunk=base.chunk, name="8b_b8_l2")
    assert _run(w, 4) >= 3
