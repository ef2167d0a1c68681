"""mk_attention_decode_noalloc: decode attention with no device allocation.

The no-alloc entry point serves callers that cannot allocate device memory
while they run (servers and plugins that hand all of HBM to their own pool
at start up, loops where an allocation could synchronise the device): its
split-KV scratch is a fixed array inside the library.  These tests call it
through the C ABI on two calls in a row and check

  - its attention output against the float64 oracle's single-pass
    attention over the same query, cached rows and appended row, and the
    rows it appends against the oracle's bf16 rounding of the rotated key
    and the value, at tolerances that fit one fp32 op;
  - the same outputs against a graph holding the same attention op run
    through mk_decode_step, within the tolerances the other parity tests use;
  - that a call (after the first, which looks the array up) leaves the
    device's free memory unchanged;
  - that sizes beyond the fixed scratch are refused before any device work.

This file is collected last, so a run that stops at the first failure has
run every other test before it.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import forward as of

pytestmark = pytest.mark.gpu

B, HQ, HKV, D = 3, 32, 8, 128
G = HQ // HKV
LEN0 = [100, 700, 2000]
CAP = 2100
THETA = 5e5
# graph vs no-alloc: the end-to-end tolerances of the parity tests
ATOL, RTOL_L2 = 3e-2, 1e-2
# one attention op, fp32 on the GPU vs float64: scores are 128-term dot
# products of O(1) values and the output a weighted mean of <= 2101 bf16
# rows, so fp32 rounding stays near 1e-6 of the O(1) outputs; 1e-4 absolute
# and 2e-5 relative L2 leave room for the f32 sums and nothing for a wrong
# key, head, position or rotation (errors of order 0.1)
OP_ATOL, OP_RTOL_L2 = 1e-4, 2e-5


def _close(a, b, atol, rtol_l2):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = np.abs(a - b).max()
    assert d <= atol, f"max |delta| {d}"
    rel = np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel <= rtol_l2, f"relative L2 {rel}"


def _codes(t):
    """bf16 tensor -> uint16 codes (numpy)."""
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def _oracle_call(kc, vc, qkv, pos):
    """Oracle step of the attention op on float64 qkv [B, (Hq + 2 Hkv) D]:
    append the rotated key and the value at pos (bf16 via f32, in the
    uint16 caches kc / vc [B, Hkv, cap, D]) and attend over keys 0..pos."""
    out = np.zeros((B, HQ * D))
    for s in range(B):
        p = pos[s]
        q = qkv[s, : HQ * D].reshape(HQ, D)
        k = qkv[s, HQ * D:(HQ + HKV) * D].reshape(HKV, D)
        v = qkv[s, (HQ + HKV) * D:].reshape(HKV, D)
        kc[s, :, p, :] = of.round_to_bf16_via_f32(of.rope(k, p, THETA))
        vc[s, :, p, :] = of.round_to_bf16_via_f32(v)
        qr = of.rope(q, p, THETA)
        for g in range(HKV):
            o = of.attention_single(qr[g * G:(g + 1) * G], of.bf16_to_f64(kc[s, g, : p + 1]),
                                    of.bf16_to_f64(vc[s, g, : p + 1]))
            out[s, g * G * D:(g + 1) * G * D] = o.reshape(-1)
    return out


def test_noalloc_attention_matches_oracle_and_graph_on_two_calls():
    from task_graph_interpreter_gb300 import _lib as L
    from task_graph_interpreter_gb300.graph import Graph

    dev = torch.device("cuda")
    nq = (HQ + 2 * HKV) * D
    gen = torch.Generator(device=dev).manual_seed(7)
    qkvs = [torch.randn(B, nq, device=dev, generator=gen) for _ in range(2)]
    kc0 = synth.kv_cache_torch("layer0.k_cache", B, HKV, CAP, D, LEN0, 0, device=dev)
    vc0 = synth.kv_cache_torch("layer0.v_cache", B, HKV, CAP, D, LEN0, 0, device=dev)

    # existing entry point: a graph holding one attention op
    g = Graph(B, device=dev)
    qkv_buf = torch.empty(B, nq, device=dev)
    kc_a, vc_a = kc0.clone(), vc0.clone()
    q = g.register(qkv_buf)
    kb = g.register(kc_a, B * HKV, CAP * D)
    vb = g.register(vc_a, B * HKV, CAP * D)
    att = g.attention(q, kb, vb, HQ, HKV, D, CAP, LEN0, 0, THETA)
    g.state[:, 1] = torch.tensor(LEN0, dtype=torch.int32, device=dev)
    g.lower()
    g.upload()

    # the no-alloc entry point on its own copies of the same inputs
    kc_b, vc_b = kc0.clone(), vc0.clone()
    out_b = torch.empty(B, HQ * D, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    # the oracle's caches (bf16 codes) start from the same rows
    kc_o, vc_o = _codes(kc0).copy(), _codes(vc0).copy()

    for call in range(2):
        pos = [l + call for l in LEN0]
        qkv_buf.copy_(qkvs[call])
        g.state[:, 1] = torch.tensor(pos, dtype=torch.int32, device=dev)
        g.step()
        code, task = g.status()
        assert code == 0, (code, task)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        L.mk_attention_decode_noalloc(stream, qkvs[call].data_ptr(), kc_b.data_ptr(), vc_b.data_ptr(),
                                      out_b.data_ptr(), B, HQ, HKV, D, CAP, pos, LEN0, 0, THETA)
        torch.cuda.synchronize()
        if call == 1:
            # the first call looked the scratch array up; later calls allocate nothing
            assert torch.cuda.mem_get_info(dev)[0] == free_before

        want = _oracle_call(kc_o, vc_o, qkvs[call].double().cpu().numpy(), pos)
        _close(out_b.double().cpu().numpy(), want, OP_ATOL, OP_RTOL_L2)
        _close(out_b.double().cpu().numpy(), att.tensor.double().cpu().numpy(), ATOL, RTOL_L2)
        for s in range(B):
            for cache_g, cache_b, cache_o in ((kc_a, kc_b, kc_o), (vc_a, vc_b, vc_o)):
                rb = cache_b[s, :, pos[s], :].double().cpu().numpy()
                ro = of.bf16_to_f64(cache_o[s, :, pos[s], :])
                ra = cache_g[s, :, pos[s], :].double().cpu().numpy()
                # one bf16 step at most: the kernel rounds an f32 rotation
                assert np.all(np.abs(rb - ro) <= np.abs(ro) * 2.0 ** -7 + 1e-30)
                assert np.all(np.abs(rb - ra) <= np.abs(ra) * 2.0 ** -7 + 1e-30)
    # rows other than the appended ones are untouched by both paths
    assert torch.equal(kc_b[:, :, :LEN0[0]], kc0[:, :, :LEN0[0]])
    assert torch.equal(vc_b[:, :, :LEN0[0]], vc0[:, :, :LEN0[0]])
    g.close()


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    from task_graph_interpreter_gb300 import _lib as L
    dev = torch.device("cuda")
    # the limit is checked on the host before any device access: small
    # placeholders stand in for the caches and activations
    dummy = torch.zeros(64, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    # 8 sequences x 8 kv heads x 64 one-thousand-key chunks need 8.5 M floats
    with pytest.raises(L.MkError) as e:
        L.mk_attention_decode_noalloc(stream, dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(), dummy.data_ptr(),
                                      8, HQ, HKV, D, 70000, [64000] * 8, [64000] * 8, 1000, THETA)
    assert e.value.code == L.MK_ERR_LIMIT
