"""Helpers for GPU parity tests: run the CUDA path and the oracle on the same
seeded inputs and compare them."""
from __future__ import annotations

import math

import numpy as np
import torch

import synth
from oracle import forward as of
from tests.common import NpWeights, oracle_state

# Acceptance tolerances for floating-point results (fp32 kernels vs the
# float64 oracle): logits max |delta| <= 3e-2 with cosine >= 0.9999, every
# layer's hidden state within 1e-2 relative L2.
LOGIT_ATOL = 3e-2
LOGIT_COS = 0.9999
HIDDEN_RTOL = 1e-2


def build_gpu(w, seed=0, mode_ctas=0, layers_keep_hidden=True, wait_timeout_us=0, norms="fused"):
    from task_graph_interpreter_gb300.llama import build_llama_decode
    weights, kc, vc, hist, state = synth.device_inputs(w, seed, "cuda")
    dec = build_llama_decode(w.model, w.B, w.kv_len, w.capacity, weights, kc, vc, hist, chunk=w.chunk,
                             device="cuda", num_ctas=mode_ctas, wait_timeout_us=wait_timeout_us, norms=norms)
    dec.graph.state.copy_(state)
    dec.graph.lower()
    dec.graph.upload()
    dec.inputs = (weights, kc, vc, hist, state)
    return dec


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


def compare_step(dec, res, st_oracle, check_hidden=True):
    """Compare one step's GPU outputs with the oracle step result.  Returns the
    max |logit delta| and whether every token decision was unambiguous."""
    m_logits = dec.logits.tensor.double().cpu().numpy()
    B = m_logits.shape[0]
    dmax = float(np.abs(m_logits - res.logits).max())
    assert dmax <= LOGIT_ATOL, f"logits max |delta| {dmax}"
    for s in range(B):
        c = cosine(m_logits[s], res.logits[s])
        assert c >= LOGIT_COS, f"logits cosine {c} for sequence {s}"
    if check_hidden:
        for l, hb in enumerate(dec.hidden):
            h = hb.tensor.double().cpu().numpy()
            rel = np.linalg.norm(h - res.hidden[l]) / np.linalg.norm(res.hidden[l])
            assert rel <= HIDDEN_RTOL, f"layer {l} hidden rel L2 {rel}"
    state = dec.graph.state.cpu().numpy()
    clear = True
    for s in range(B):
        tok = int(state[s, 0])
        if res.margin[s] > 2 * dmax + 1e-6:
            assert tok == int(res.tokens[s]), f"token {tok} != oracle {res.tokens[s]} (margin {res.margin[s]})"
        else:
            # near-tie: any token within the error bound of the max is correct
            clear = False
            assert res.logits[s, tok] >= res.logits[s].max() - 2 * dmax - 1e-6
        assert int(state[s, 1]) == int(st_oracle.pos[s])
    return dmax, clear


def compare_cache_rows(dec, st_oracle, pos_before):
    """The rows appended this step match the oracle's within one bf16 ulp of
    each element plus 2^-8 of the row's RMS.  The rows are bf16 roundings of
    f32 values whose inputs carry the error accumulated over the layers
    before (bounded for the hidden states by 1e-2 relative L2); elements far
    below the row's magnitude can then round a few bf16 steps away, most of
    all under the tensor cores' truncating f32 accumulation.  2^-8 of the
    RMS stays well inside the hidden-state bound and far below the O(RMS)
    errors of a wrong head, position or rotation."""
    for l in range(len(dec.kcache)):
        for which, bufs, ref in (("k", dec.kcache, st_oracle.kcache), ("v", dec.vcache, st_oracle.vcache)):
            t = bufs[l].tensor
            for s, p in enumerate(pos_before):
                got = t[s, :, p, :].float().cpu().numpy().astype(np.float64)
                want = of.bf16_to_f64(ref[l][s, :, p, :])
                tol = np.abs(want) * 2.0 ** -7 + 2.0 ** -8 * np.sqrt(np.mean(want ** 2)) + 1e-30
                err = np.abs(got - want)
                i = np.unravel_index(np.argmax(err - tol), err.shape)
                assert np.all(err <= tol), (f"layer {l} {which} row {p} seq {s}: |err| {err[i]:.3g} at {i}, "
                                            f"want {want[i]:.6g} got {got[i]:.6g}, row rms "
                                            f"{np.sqrt(np.mean(want ** 2)):.3g}, max |err| {err.max():.3g}")
