"""mk_attention_decode_noalloc against the existing attention entry point.

The no-alloc entry point serves callers that cannot allocate device memory
while they run (servers and plugins that hand all of HBM to their own pool
at start up, loops where an allocation could synchronise the device): its
split-KV scratch is a fixed array inside the library.  This test calls it
through the C ABI and checks, on two calls in a row, that its attention
output and the KV rows it appends match what a graph holding the same
attention op produces through mk_decode_step, within the tolerances the
other parity tests use.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

B, HQ, HKV, D = 3, 32, 8, 128
LEN0 = [100, 700, 2000]
CAP = 2100
THETA = 5e5
ATOL, RTOL_L2 = 3e-2, 1e-2


def _close(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    assert np.abs(a - b).max() <= ATOL
    assert np.linalg.norm(a - b) <= RTOL_L2 * np.linalg.norm(b)


def test_noalloc_attention_matches_graph_attention_on_two_calls():
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

    for call in range(2):
        pos = [l + call for l in LEN0]
        qkv_buf.copy_(qkvs[call])
        g.state[:, 1] = torch.tensor(pos, dtype=torch.int32, device=dev)
        g.step()
        code, task = g.status()
        assert code == 0, (code, task)
        L.mk_attention_decode_noalloc(stream, qkvs[call].data_ptr(), kc_b.data_ptr(), vc_b.data_ptr(),
                                      out_b.data_ptr(), B, HQ, HKV, D, CAP, pos, LEN0, 0, THETA)
        torch.cuda.synchronize()
        _close(out_b, att.tensor)
        for s in range(B):
            for cache_a, cache_b in ((kc_a, kc_b), (vc_a, vc_b)):
                ra = cache_a[s, :, pos[s], :].float()
                rb = cache_b[s, :, pos[s], :].float()
                assert torch.all((ra - rb).abs() <= ra.abs() * 2.0 ** -7 + 1e-30)
    # rows other than the appended ones are untouched by both paths
    assert torch.equal(kc_b[:, :, :LEN0[0]], kc0[:, :, :LEN0[0]])
    g.close()


def test_noalloc_rejects_sizes_beyond_its_fixed_scratch():
    from task_graph_interpreter_gb300 import _lib as L
    dev = torch.device("cuda")
    nq = (HQ + 2 * HKV) * D
    qkv = torch.zeros(8, nq, device=dev)
    kc = torch.zeros(8, HKV, 70000, D, dtype=torch.bfloat16, device=dev)
    out = torch.empty(8, HQ * D, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    # 8 sequences x 8 kv heads x 64 one-thousand-key chunks need 8.5 M floats
    with pytest.raises(L.MkError) as e:
        L.mk_attention_decode_noalloc(stream, qkv.data_ptr(), kc.data_ptr(), kc.data_ptr(), out.data_ptr(), 8, HQ,
                                      HKV, D, 70000, [64000] * 8, [64000] * 8, 1000, THETA)
    assert e.value.code == L.MK_ERR_LIMIT
