"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks an oracle function against something it does not share
code with: a brute-force loop, a closed form, an invariant, a library
routine on a special case, or a value printed on the pages (tests/golden).
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import forward as of
from oracle import lowering as ol
from oracle.graph import llama_decode_spec
from oracle.validate import validate, ValidationError, levels
from tests.common import NpWeights, oracle_state, read_golden
from tests import naive_llama

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------- number formats
def test_bf16_widen_and_round_match_torch():
    x = np.concatenate([RNG.standard_normal(20000) * 3.0,
                        [0.0, -0.0, 1.0, 1.00390625, 1.0078125, 1.01171875, -2.5e-30, 65504.0]])
    codes = of.round_to_bf16_via_f32(x)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codes, ref)
    back = of.bf16_to_f64(codes)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_bf16_round_ties_to_even():
    # 1 + 2^-8 lies halfway between bf16 1.0 and 1 + 2^-7: ties go to the even code
    assert of.round_to_bf16_via_f32(np.array([1.0 + 2 ** -8]))[0] == 0x3F80
    assert of.round_to_bf16_via_f32(np.array([1.0 + 3 * 2 ** -8]))[0] == 0x3F82


# ------------------------------------------------------------- RMSNorm
def test_rmsnorm_closed_form_unit_rms():
    x = RNG.standard_normal((3, 257)) * 5.0
    eps = 1e-5
    y = of.rmsnorm(x, np.ones(257), eps)
    ms = np.mean(x * x, axis=-1)
    # before gamma, rms(y) = sqrt(ms / (ms + eps)) exactly
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), np.sqrt(ms / (ms + eps)), rtol=1e-14)


def test_rmsnorm_scale_invariance_eps0_and_gamma():
    x = RNG.standard_normal(64)
    g = RNG.standard_normal(64)
    a = of.rmsnorm(x, g, 0.0)
    b = of.rmsnorm(37.5 * x, g, 0.0)
    assert np.allclose(a, b, rtol=1e-13)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x)[None], (64,), torch.from_numpy(g), eps=1e-5)
    assert np.allclose(of.rmsnorm(x, g, 1e-5), ref.numpy()[0], rtol=1e-13)


# ------------------------------------------------------------- RoPE
def test_rope_position_zero_is_identity():
    v = RNG.standard_normal((5, 128))
    assert np.array_equal(of.rope(v, 0, 5e5), v)


def test_rope_preserves_pair_norms_and_matches_complex_rotation():
    D, theta, pos = 64, 1e4, 777
    v = RNG.standard_normal(D)
    r = of.rope(v, pos, theta)
    for i in range(D // 2):
        z = complex(v[i], v[i + D // 2]) * np.exp(1j * pos * theta ** (-2 * i / D))
        assert abs(r[i] - z.real) < 1e-12 and abs(r[i + D // 2] - z.imag) < 1e-12
        assert abs(math.hypot(r[i], r[i + D // 2]) - math.hypot(v[i], v[i + D // 2])) < 1e-12


def test_rope_first_pair_rotates_by_position_radians():
    # inv_freq_0 = theta^0 = 1: the first pair turns by exactly pos radians
    v = np.zeros(8); v[0] = 1.0
    r = of.rope(v, 3, 1e4)
    assert abs(r[0] - math.cos(3)) < 1e-15 and abs(r[4] - math.sin(3)) < 1e-15


def test_rope_scores_depend_only_on_relative_position():
    D, theta = 128, 5e5
    q, k = RNG.standard_normal(D), RNG.standard_normal(D)
    a = of.rope(q, 100, theta) @ of.rope(k, 40, theta)
    b = of.rope(q, 1060, theta) @ of.rope(k, 1000, theta)
    assert abs(a - b) < 1e-9


# ------------------------------------------------------------- SiLU
def test_silu_limits_and_library():
    assert of.silu(np.array([0.0]))[0] == 0.0
    assert abs(of.silu(np.array([40.0]))[0] - 40.0) < 1e-12
    assert abs(of.silu(np.array([-40.0]))[0]) < 1e-15
    z = RNG.standard_normal(1000) * 6
    assert np.allclose(of.silu(z), torch.nn.functional.silu(torch.from_numpy(z)).numpy(), rtol=1e-14)


# ------------------------------------------------------------- attention
def _brute_attention(q, K, V):
    out = np.zeros_like(q)
    D = q.shape[1]
    for h in range(q.shape[0]):
        s = [sum(q[h, d] * K[j, d] for d in range(D)) / math.sqrt(D) for j in range(K.shape[0])]
        mx = max(s)
        e = [math.exp(x - mx) for x in s]
        for j in range(K.shape[0]):
            out[h] += e[j] / sum(e) * V[j]
    return out


def test_attention_single_vs_brute_force_and_sdpa():
    q = RNG.standard_normal((4, 16)); K = RNG.standard_normal((9, 16)); V = RNG.standard_normal((9, 16))
    o = of.attention_single(q, K, V)
    assert np.allclose(o, _brute_attention(q, K, V), rtol=1e-12, atol=1e-13)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None, None].expand(1, 4, 9, 16),
        torch.from_numpy(V)[None, None].expand(1, 4, 9, 16))
    assert np.allclose(o, ref[0, :, 0].numpy(), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("n,P", [(1, 1), (7, 1), (7, 7), (5, 8), (129, 4), (300, 16), (1000, 3)])
def test_split_kv_combine_equals_single_pass(n, P):
    q = RNG.standard_normal((4, 32)) * 2; K = RNG.standard_normal((n, 32)); V = RNG.standard_normal((n, 32))
    parts = [of.attention_partial(q, K[a:b], V[a:b]) for (a, b) in of.chunk_bounds(n, P)]
    assert any(p[1][0] == 0 for p in parts) == (P > n or any(a == b for a, b in of.chunk_bounds(n, P)))
    assert np.allclose(of.attention_combine(parts), of.attention_single(q, K, V), rtol=1e-12, atol=1e-13)


def test_split_kv_random_chunkings_with_empty_chunks():
    q = RNG.standard_normal((4, 8)); K = RNG.standard_normal((50, 8)); V = RNG.standard_normal((50, 8))
    for _ in range(20):
        cuts = sorted(RNG.integers(0, 51, size=int(RNG.integers(1, 8))))
        bounds = list(zip([0] + cuts, cuts + [50]))
        parts = [of.attention_partial(q, K[a:b], V[a:b]) for a, b in bounds]
        assert np.allclose(of.attention_combine(parts), of.attention_single(q, K, V), rtol=1e-12)


def test_chunk_bounds_partition():
    for L in (1, 2, 5, 129, 4097):
        for P in (1, 2, 3, 16, 32):
            b = of.chunk_bounds(L, P)
            assert len(b) == P and b[0][0] == 0 and b[-1][1] == L
            assert all(b[i][1] == b[i + 1][0] for i in range(P - 1))
            assert all(0 <= y - x <= -(-L // P) for x, y in b)


# ------------------------------------------------------------- whole step
def test_tiny_forward_matches_brute_force_loops():
    w = synth.workload("tiny")
    m = w.model
    W = NpWeights(m)
    st = oracle_state(w)
    kc = [st.kcache[l][0].copy() for l in range(m.L)]
    vc = [st.vcache[l][0].copy() for l in range(m.L)]
    tok, pos = int(st.token[0]), int(st.pos[0])
    res = of.decode_step(m, W, st)
    logits, hidden, best = naive_llama.decode_step(m, W, tok, pos, kc, vc)
    assert np.allclose(res.logits[0], logits, rtol=1e-10, atol=1e-10)
    for l in range(m.L):
        assert np.allclose(res.hidden[l][0], hidden[l], rtol=1e-10, atol=1e-10)
    assert res.tokens[0] == best
    for l in range(m.L):
        assert np.array_equal(st.kcache[l][0], kc[l]) and np.array_equal(st.vcache[l][0], vc[l])
    # state update: next token at the next position, recorded in the history
    assert st.pos[0] == pos + 1 and st.token[0] == best and st.history[0, pos + 1] == best


def test_greedy_argmax_first_index_on_ties():
    assert of.argmax_first(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    assert of.top2_margin(np.array([1.0, 3.0, 3.0])) == 0.0


def test_generator_numpy_and_torch_cpu_agree():
    a = synth.normal_bf16_np("w", (333, 77), 0.0, 0.02, seed=3)
    b = synth.normal_bf16_torch("w", (333, 77), 0.0, 0.02, seed=3)
    assert np.array_equal(a, b.view(torch.int16).numpy().view(np.uint16))
    k = synth.kv_cache_np("kc", 2, 2, 50, 64, [40, 7], seed=1)
    kt = synth.kv_cache_torch("kc", 2, 2, 50, 64, [40, 7], seed=1)
    assert np.array_equal(k, kt.view(torch.int16).numpy().view(np.uint16))
    # capacity-independent values
    k2 = synth.kv_cache_np("kc", 2, 2, 90, 64, [40, 7], seed=1)
    assert np.array_equal(k2[:, :, :50], k)
    f = of.bf16_to_f64(synth.normal_bf16_np("w", (200000,), 0.0, 0.02))
    assert abs(f.mean()) < 3e-4 and abs(f.std() - 0.02) < 3e-4


# ------------------------------------------------------------- lowering
def test_descriptor_dtype_matches_struct_listing():
    rows = read_golden("descriptor_layout.txt")
    for name, off, size in rows:
        if name == "SIZE":
            assert ol.TASK_DTYPE.itemsize == int(off)
            continue
        f = ol.TASK_DTYPE.fields[name]
        assert f[1] == int(off), name
        assert f[0].itemsize == int(size), name
    assert ol.TASK_DTYPE.fields["remaining_deps"][1] % 4 == 0


def test_opids_and_flags_match_pages():
    ids = dict((n, int(v)) for n, v in read_golden("opids.txt"))
    assert ids["GEMV"] == ol.OP_GEMV and ids["SAMPLE"] == ol.OP_SAMPLE
    assert ids["MEMCPY"] == ol.OP_MEMCPY and ids["ATTENTION_APPEND"] == ol.OP_ATT_APPEND
    assert ids["ATTENTION_PARTIAL"] == ol.OP_ATT_PARTIAL and ids["ATTENTION_COMBINE"] == ol.OP_ATT_COMBINE
    fl = dict((n, int(v)) for n, v in read_golden("flags.txt"))
    assert fl == {"SILU_MUL": ol.F_SILU_MUL, "ADD_RESIDUAL": ol.F_ADD_RESIDUAL,
                  "RMS_NORM_INPUT": ol.F_RMS_NORM_INPUT}


def test_tile_rule_reproduces_worked_example():
    (n, tt, al, ntask, w), = read_golden("tile_example.txt")
    t = ol.tiles(int(n), int(tt), int(al))
    assert len(t) == int(ntask) and all(c == int(w) for _, c in t)
    assert synth.LLAMA_1B.n_qkv == int(n)


def test_tile_rule_covers_columns_with_short_last_tile():
    for n in (1, 15, 16, 1000, 6144, 14336, 128256):
        for tt in (1, 7, 152):
            t = ol.tiles(n, tt, 16)
            assert t[0][0] == 0 and sum(c for _, c in t) == n and len(t) <= tt
            assert all(c0 % 16 == 0 for c0, _ in t)


def _spec(name, num_ctas=152):
    w = synth.workload(name)
    return w, llama_decode_spec(w.model, w.B, w.kv_len, w.capacity, w.chunk, num_ctas)


@pytest.mark.parametrize("name", synth.WORKLOADS)
def test_lowered_graph_validates(name):
    w, spec = _spec(name)
    tasks, edges = ol.lower(spec)
    st = validate(tasks, edges, check_hazards=name in ("tiny", "1b", "8b"))
    m = w.model
    # every layer's tasks, the lm_head tiles and SAMPLE are present (a timed
    # step that skips layers or the lm_head would not contain them)
    n_gemv = int((tasks["op_id"] == ol.OP_GEMV).sum())

    def T(n, k, flags):  # GEMV tasks of an op: tiles, or row blocks x K splits
        _, nb, S = ol.ksplit_plan(n, k, flags, w.B, 152, 16)
        return nb * S
    per_layer = (T(m.n_qkv, m.H, ol.F_RMS_NORM_INPUT) + T(m.H, m.Hq * m.D, ol.F_ADD_RESIDUAL)
                 + T(m.F, m.H, ol.F_RMS_NORM_INPUT | ol.F_SILU_MUL) + T(m.H, m.F, ol.F_ADD_RESIDUAL))
    assert n_gemv == m.L * per_layer + T(m.V, m.H, ol.F_RMS_NORM_INPUT | ol.F_ARGMAX_EPI)
    assert int((tasks["op_id"] == ol.OP_SAMPLE).sum()) == w.B
    assert int((tasks["op_id"] == ol.OP_ATT_APPEND).sum()) == m.L * w.B * m.Hkv
    assert st["levels"] > 0


def test_long_context_chunking_gives_32_partials():
    w, spec = _spec("8b_long")
    tasks, _ = ol.lower(spec)
    part = tasks[tasks["op_id"] == ol.OP_ATT_PARTIAL]
    # 32768 cached keys in chunks of 1024: 32 partials per (sequence, kv head)
    assert len(part) == 32 * 4 * 8 * w.model.L
    assert set(int(r >> 16) for r in part["reserved"][:, 3]) == {32}


def test_level_rule_on_a_chain():
    w, spec = _spec("tiny")
    tasks, edges = ol.lower(spec)
    lv = levels(tasks, edges)
    # embed tasks have no parents (level 0); qkv tiles depend on them (level 1)
    assert lv[0] == 0 and lv[1] == 1
    cnt = tasks["num_dependents"]; off = tasks["dependents_offset"]
    for t in range(len(tasks)):
        for c in edges[off[t]: off[t] + cnt[t]]:
            assert lv[c] >= lv[t] + 1


# ------------------------------------------------------------- planted mistakes
def _tiny_lowered():
    _, spec = _spec("tiny")
    return ol.lower(spec)


def test_validator_rejects_backward_edge():
    tasks, edges = _tiny_lowered()
    e = edges.copy()
    t = int(np.nonzero(tasks["num_dependents"] > 0)[0][5])
    e[tasks["dependents_offset"][t]] = 0
    with pytest.raises(ValidationError):
        validate(tasks, e)


def test_validator_rejects_wrong_dependency_count():
    tasks, edges = _tiny_lowered()
    t2 = tasks.copy()
    t2["remaining_deps"][10] += 1
    with pytest.raises(ValidationError):
        validate(t2, edges)


def test_validator_catches_a_dropped_dependency_as_a_race():
    tasks, edges = _tiny_lowered()
    # drop the edge from the first qkv tile to its first child
    t = 1
    n = int(tasks["num_dependents"][t]); o = int(tasks["dependents_offset"][t])
    child = int(edges[o])
    e = np.delete(edges, o)
    t2 = tasks.copy()
    t2["num_dependents"][t] = n - 1
    t2["dependents_offset"][t + 1:] -= 1
    t2["remaining_deps"][child] -= 1
    with pytest.raises(ValidationError):
        validate(t2, e)


def test_oracle_lowering_planted_tile_bug_is_caught():
    # a lowering that drops the last tile of the 512-column ops (qkv and
    # gate_up in the tiny model) leaves columns that later tasks read unwritten
    _, spec = _spec("tiny")
    orig = ol.tiles
    try:
        ol.tiles = lambda n, tt, al: orig(n, tt, al)[:-1] if n == 512 else orig(n, tt, al)
        tasks, edges = ol.lower(spec)
    finally:
        ol.tiles = orig
    with pytest.raises(ValidationError):
        validate(tasks, edges)


def test_auto_chunking_fits_one_wave_with_the_smallest_chunk():
    """Automatic split-KV chunking (our reading): the chunk count fits the
    CTAs whenever one chunk per sequence does, with the smallest chunk
    length that achieves it (never below max(128, average share))."""
    import numpy as np
    from oracle.lowering import partials_per_sequence, ceil_div
    rng = np.random.default_rng(5)
    for _ in range(200):
        B = int(rng.integers(1, 9))
        Hkv = int(rng.choice([1, 2, 8]))
        ctas = int(rng.integers(8, 200))
        lens = [int(x) for x in rng.integers(0, 9000, size=B)]
        P = partials_per_sequence(lens, Hkv, 0, ctas)
        assert all(p >= 1 for p in P)
        floor = max(128, ceil_div(Hkv * sum(lens), ctas))
        E = max(max(ceil_div(l, p) for l, p in zip(lens, P)), floor)
        if Hkv * B <= ctas:
            assert Hkv * sum(P) <= ctas
            if E > floor:  # one key less per chunk would overflow the wave
                assert Hkv * sum(max(1, ceil_div(l, E - 1)) for l in lens) > ctas
        assert all(p == max(1, ceil_div(l, E)) or ceil_div(l, p) <= E for l, p in zip(lens, P))


def _chunk_inputs(T, seed=5):
    import copy
    w = synth.custom(synth.TINY, 2, [40, 120], T, name="tiny_chunk")
    W = NpWeights(w.model)
    st = oracle_state(w)
    rng = np.random.default_rng(seed)
    toks = np.concatenate([st.token[:, None], rng.integers(0, w.model.V, size=(w.B, T - 1))], axis=1)
    return w, W, st, copy.deepcopy(st), toks


def test_chunk_step_equals_steps_with_the_inputs_fixed():
    # T tokens through one chunk step = T single-token steps fed the same
    # inputs (each step's argmax replaced by the next given token)
    T = 4
    w, W, st_chunk, st_seq, toks = _chunk_inputs(T)
    res = of.chunk_step(w.model, W, st_chunk, toks)
    for i in range(T):
        if i:
            st_seq.token[:] = toks[:, i]
        r = of.decode_step(w.model, W, st_seq)
        np.testing.assert_allclose(res.logits[:, i], r.logits, rtol=1e-12, atol=1e-12)
        for l in range(w.model.L):
            np.testing.assert_allclose(res.hidden[l][:, i], r.hidden[l], rtol=1e-12, atol=1e-12)
    for l in range(w.model.L):
        assert np.array_equal(st_chunk.kcache[l], st_seq.kcache[l])
        assert np.array_equal(st_chunk.vcache[l], st_seq.vcache[l])
    assert np.array_equal(st_chunk.pos, st_seq.pos) and np.array_equal(st_chunk.token, st_seq.token)
    for s in range(w.B):
        p = int(st_chunk.pos[s])
        assert np.array_equal(st_chunk.history[s, p - T + 1: p], toks[s, 1:])
        assert st_chunk.history[s, p] == st_seq.history[s, p]


def test_chunk_step_is_causal_and_one_token_is_a_decode_step():
    # a later token of the chunk never changes an earlier row's logits, and a
    # one-token chunk is exactly a decode step
    T = 3
    w, W, st_a, st_b, toks = _chunk_inputs(T)
    other = toks.copy()
    other[:, -1] = (other[:, -1] + 17) % w.model.V
    ra = of.chunk_step(w.model, W, st_a, toks)
    rb = of.chunk_step(w.model, W, st_b, other)
    assert np.array_equal(ra.logits[:, :-1], rb.logits[:, :-1])
    assert not np.allclose(ra.logits[:, -1], rb.logits[:, -1])
    w, W, st_c, st_d, toks = _chunk_inputs(1)
    rc = of.chunk_step(w.model, W, st_c, toks)
    rd = of.decode_step(w.model, W, st_d)
    assert np.array_equal(rc.logits[:, 0], rd.logits) and np.array_equal(rc.tokens, rd.tokens)
