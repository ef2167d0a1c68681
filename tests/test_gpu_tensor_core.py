"""Decode with three to eight activation rows: GEMV tiles on the tcgen05
tensor-core path (rows past the batch enter as zeros; TMA-loaded,
128-byte-swizzled weight tiles, activations as three bf16 parts, f32 accumulators
in tensor memory) against the float64 oracle, through the C ABI.

The tiny model spans several tiles per op with a short last tile, K of 256
and 512 (a single K range) and ragged KV lengths including an empty cache;
the 1B-shaped model has K = 2048 and 8192 (several K ranges per tile) and
the tied 128256-row LM head.
"""
import pytest

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import build_gpu, compare_step, compare_cache_rows

pytestmark = pytest.mark.gpu


def _run(w, steps, seed=0):
    """Steps compared with the oracle; after a near-tie token (checked to be
    within the error bound of the best) later inputs may differ, so the
    comparison stops there."""
    dec = build_gpu(w, seed)
    W = NpWeights(w.model, seed)
    st = oracle_state(w, seed)
    compared = 0
    try:
        tiles = dec.graph.tensor_core_tiles()
        assert tiles > 0, "no GEMV tile took the tensor-core path"
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
    finally:
        dec.graph.close()
    return compared


def test_tiny_batch8_tensor_core_tiles_match_oracle():
    w = synth.custom(synth.TINY, 8, [0, 1, 5, 17, 64, 100, 128, 33], 4, name="tiny_b8")
    assert _run(w, 4) >= 2


@pytest.mark.slow
def test_1b_batch8_tensor_core_tiles_match_oracle():
    w = synth.custom(synth.LLAMA_1B, 8, [700, 64, 1024, 9, 300, 512, 1000, 128], 1, name="1b_b8")
    assert _run(w, 1) == 1


@pytest.mark.parametrize("B", [3, 4])
def test_tiny_batch3_and_4_tensor_core_tiles_match_oracle(B):
    # the smallest batches on the tensor cores: 3 or 4 of the 8 activation
    # rows live, the accumulators read back at batch width 8
    w = synth.custom(synth.TINY, B, [128, 5, 77, 40][:B], 4, name=f"tiny_tc_b{B}")
    assert _run(w, 4) >= 2


def test_1b_width_batch4_tensor_core_tiles_match_oracle():
    import dataclasses
    m = dataclasses.replace(synth.LLAMA_1B, L=2)
    w = synth.custom(m, 4, [1024, 300, 777, 64], 2, name="1b_b4_l2")
    assert _run(w, 2) >= 1
