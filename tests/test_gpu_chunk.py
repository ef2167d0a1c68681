"""Chunk steps (several tokens per sequence per step) against the oracle.

A chunk step feeds T tokens of each sequence through one launch: token 0 is
the pending token in the state, tokens 1..T-1 come from the step's tokens
buffer (a prefill chunk, or draft tokens to verify).  Token t sits at
position pos + t and attends causally to the cache and the chunk's earlier
tokens; every GEMV runs on the B * T activation rows (the tensor-core tiles
when B * T = 8); the per-token tasks carry t in the descriptor's step field.
The float64 oracle's ``chunk_step`` is the plain definition (T decode steps
with the inputs fixed in advance).  Compared per step: the logits of every
row, every layer's hidden state of every row, the T cache rows appended per
sequence and layer, the sampled token, the history and the position.
"""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state
from tests.gpu_common import LOGIT_ATOL, LOGIT_COS, HIDDEN_RTOL, cosine, compare_cache_rows

pytestmark = pytest.mark.gpu


def _run_chunks(w, T, steps, seed=0):
    from task_graph_interpreter_gb300.llama import build_llama_decode
    import torch
    m = w.model
    weights, kc, vc, hist, state = synth.device_inputs(w, seed, "cuda")
    dec = build_llama_decode(m, w.B, w.kv_len, w.capacity, weights, kc, vc, hist, chunk=w.chunk, device="cuda",
                             T=T)
    g = dec.graph
    g.state.copy_(state)
    g.lower()
    g.upload()
    if w.B * T == 8:
        assert g.tensor_core_tiles() > 0, "B * T = 8 rows should take the tensor-core path"
    W = NpWeights(m, seed)
    st = oracle_state(w, seed)
    B = w.B
    done = 0
    try:
        for step in range(steps):
            drafts = synth.uniform_ints_np(f"draft{step}", B * T, 0, m.V, seed).reshape(B, T)
            drafts[:, 0] = st.token
            dec.tokens.tensor.copy_(torch.from_numpy(drafts.astype(np.int32)))
            pos_before = [int(p) for p in st.pos]
            g.step()
            code, task = g.status()
            assert code == 0, f"device status {code} at task {task}"
            res = of.chunk_step(m, W, st, drafts)
            got = dec.logits.tensor.double().cpu().numpy().reshape(B, T, -1)
            d = float(np.abs(got - res.logits).max())
            assert d <= LOGIT_ATOL, f"step {step}: logits max |delta| {d}"
            for s in range(B):
                for t in range(T):
                    c = cosine(got[s, t], res.logits[s, t])
                    assert c >= LOGIT_COS, f"step {step}: cosine {c} at ({s}, {t})"
            for l, hb in enumerate(dec.hidden):
                h = hb.tensor.double().cpu().numpy().reshape(B, T, -1)
                rel = np.linalg.norm(h - res.hidden[l]) / np.linalg.norm(res.hidden[l])
                assert rel <= HIDDEN_RTOL, f"step {step}: layer {l} hidden rel L2 {rel}"
            for t in range(T):
                compare_cache_rows(dec, st, [p + t for p in pos_before])
            sg = g.state.cpu().numpy()
            hs = dec.history.tensor.cpu().numpy()
            clear = True
            for s in range(B):
                p = pos_before[s]
                assert int(sg[s, 1]) == p + T
                assert list(hs[s, p + 1: p + T]) == list(drafts[s, 1:])
                tok = int(sg[s, 0])
                assert int(hs[s, p + T]) == tok
                if res.margin[s] > 2 * d + 1e-6:
                    assert tok == int(res.tokens[s]), f"step {step}: token {tok} != oracle {res.tokens[s]}"
                else:
                    clear = False
                    assert res.logits[s, -1, tok] >= res.logits[s, -1].max() - 2 * d - 1e-6
            done += 1
            if not clear:
                break
    finally:
        g.close()
    return done


@pytest.mark.parametrize("B,T", [(1, 4), (2, 4), (3, 2), (1, 8)])
def test_tiny_chunk_steps(B, T):
    lens = [128, 40, 3][:B]
    w = synth.custom(synth.TINY, B, lens, 3 * T + 1, name=f"tiny_chunk{B}x{T}")
    assert _run_chunks(w, T, 3) >= 2


@pytest.mark.parametrize("B,T", [(1, 4), (2, 4)])
def test_1b_width_chunk_steps(B, T):
    m = dataclasses.replace(synth.LLAMA_1B, L=2)
    lens = [1024, 517][:B]
    w = synth.custom(m, B, lens, 3 * T + 1, name=f"1b_chunk{B}x{T}")
    assert _run_chunks(w, T, 3) >= 2


def test_chunk_step_with_one_key_chunks():
    # one-key split-KV chunks: some chunks hold only this step's keys, some
    # only keys a row may not see yet (empty for those rows)
    w = synth.custom(synth.TINY, 1, [5], 3 * 4 + 1, chunk=1, name="tiny_chunk_c1")
    assert _run_chunks(w, 4, 3) >= 2


def test_chunk_step_with_tensor_core_partials():
    # T = 2 tokens x 2 heads = 4 query rows and chunks of 600 keys (five
    # blocks of 128): the partials run on tensor cores, this step's keys
    # through the same hand-off as the cached blocks
    w = synth.custom(synth.TINY, 2, [1200, 700], 3 * 2 + 1, chunk=600, name="tiny_chunk_tc")
    assert _run_chunks(w, 2, 3) >= 2
