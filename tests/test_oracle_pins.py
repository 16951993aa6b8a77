"""Pins of the CPU oracle against things other than itself (CPU only).

Each test fixes the oracle to a closed form, a brute-force enumeration, an
independent library routine, an invariant, or a value the pages print, so that a
plausible mistake in it (a dropped bias, a wrong sign in an exponent, a swapped
operand, an unstable tie-break, an off-by-one offset) fails at least one.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import testgen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _layer(d, f, E, act, rng, router=None, b_router=None, identical=False, integer=False, top_k=2, gate_mode=0,
           shared=False):
    def draw(shape, scale):
        if integer:
            return rng.integers(-2, 3, size=shape).astype(np.float32)
        return (rng.standard_normal(shape) * scale).astype(np.float32)

    wr = draw((E, d), 1 / math.sqrt(d)) if router is None else router.astype(np.float32)
    n = 1 if identical else E
    w1 = [draw((f, d), 1 / math.sqrt(d)) for _ in range(n)]
    w2 = [draw((d, f), 1 / math.sqrt(f)) for _ in range(n)]
    w3 = [draw((f, d), 1 / math.sqrt(d)) for _ in range(n)] if act == oracle.ACT_SWIGLU else None
    b1 = [draw((f,), 0.1) for _ in range(n)] if act == oracle.ACT_RELU_BIAS else None
    b2 = [draw((d,), 0.1) for _ in range(n)] if act == oracle.ACT_RELU_BIAS else None
    if identical:
        w1, w2 = w1 * E, w2 * E
        w3 = None if w3 is None else w3 * E
        b1 = None if b1 is None else b1 * E
        b2 = None if b2 is None else b2 * E
    sh = None
    if shared:
        sh = dict(w1=draw((f, d), 1 / math.sqrt(d)), w2=draw((d, f), 1 / math.sqrt(f)),
                  w3=draw((f, d), 1 / math.sqrt(d)) if act == oracle.ACT_SWIGLU else None,
                  b1=draw((f,), 0.1) if act == oracle.ACT_RELU_BIAS else None,
                  b2=draw((d,), 0.1) if act == oracle.ACT_RELU_BIAS else None)
    return oracle.OracleLayer(d, f, E, act, wr, w1, w2, w3=w3, b_router=b_router, b1=b1, b2=b2, top_k=top_k,
                              gate_mode=gate_mode, shared=sh)


def _numpy_ffn(layer, e, x):
    """Expert FFN written with numpy matmuls (an independent routine); e = "shared" for the shared expert."""
    x = x.astype(np.float64)
    if e == "shared":
        sh = layer._shared
        W1, W2, W3, B1, B2 = sh["w1"], sh["w2"], sh.get("w3"), sh.get("b1"), sh.get("b2")
    else:
        W1, W2 = layer._w1[e], layer._w2[e]
        W3 = None if layer._w3 is None else layer._w3[e]
        B1 = None if layer._b1 is None else layer._b1[e]
        B2 = None if layer._b2 is None else layer._b2[e]
    W1, W2 = W1.astype(np.float64), W2.astype(np.float64)
    if layer.act == oracle.ACT_RELU_BIAS:
        h = np.maximum(x @ W1.T + B1, 0.0)
        return h @ W2.T + B2
    g = x @ W1.T
    u = x @ W3.astype(np.float64).T
    silu = g * 0.5 * (1.0 + np.tanh(0.5 * g))  # z * sigmoid(z) through tanh: a different formula
    return (silu * u) @ W2.T


# ------------------------------------------------------------------ generator
def test_generator_is_counter_based_and_normal():
    a = testgen.normal_f32(0, 7, (100000,), 1.0)
    b = testgen.normal_f32(0, 7, (50000,), 1.0, offset=50000)
    assert np.array_equal(a[50000:], b)                      # element i depends on i only
    assert not np.array_equal(a, testgen.normal_f32(1, 7, (100000,), 1.0))
    assert not np.array_equal(a, testgen.normal_f32(0, 8, (100000,), 1.0))
    big = testgen.normal_f32(0, 3, (2_000_000,), 1.0).astype(np.float64)
    assert abs(big.mean()) < 5e-3 and abs(big.std() - 1.0) < 5e-3
    assert abs(np.mean(big ** 4) - 3.0) < 0.05               # Gaussian kurtosis
    s = testgen.normal_f32(0, 3, (100000,), 0.25)
    assert abs(s.std() - 0.25) < 3e-3


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -7, -2.5, 0.0, 3.0e38], dtype=np.float32)
    bits = testgen.f32_to_bf16_bits(vals)
    # 1+2^-8 is halfway between 1 and 1+2^-7: ties to the even mantissa (1.0);
    # 1+3*2^-8 is halfway between 1+2^-7 and 1+2^-6: ties to even (1+2^-6)
    assert list(bits[:6]) == [0x3F80, 0x3F80, 0x3F82, 0x3F81, 0xC020, 0x0000]
    back = testgen.bf16_bits_to_f32(bits)
    assert back[3] == np.float32(1.0 + 2 ** -7)
    x = testgen.normal_f32(0, 1, (10000,), 1.0)
    r = testgen.bf16_bits_to_f32(testgen.f32_to_bf16_bits(x))
    assert np.all(np.abs(r - x) <= np.abs(x) * 2.0 ** -8)


def test_workload_shapes():
    s = testgen.CONFIGS["mixtral-prefill"]
    assert (s.T, s.d_model, s.d_ff, s.num_experts, s.dtype) == (8192, 4096, 14336, 8, "bf16")
    b = testgen.zipf_router_bias(16)
    assert b[0] == 0.0 and np.all(np.diff(b) < 0)
    assert abs(float(b[15]) - 1.5 * math.log(1 / 16)) < 1e-6


# ------------------------------------------------------------------ router logits
def test_logits_equal_independent_dot_and_bias():
    rng = np.random.default_rng(1)
    d, E = 96, 6
    br = rng.standard_normal(E).astype(np.float32)
    L = _layer(d, 16, E, oracle.ACT_SWIGLU, rng, b_router=br)
    x = rng.standard_normal((40, d)).astype(np.float32)
    ref = x.astype(np.float64) @ L._wr.astype(np.float64).T + br.astype(np.float64)
    np.testing.assert_allclose(L.router_logits(x), ref, rtol=0, atol=1e-12)


def test_logits_of_unit_vectors_are_router_columns():
    rng = np.random.default_rng(2)
    d, E = 32, 5
    L = _layer(d, 8, E, oracle.ACT_SWIGLU, rng)
    x = np.eye(d, dtype=np.float32)
    assert np.array_equal(L.router_logits(x), L._wr.T.astype(np.float64))


# ------------------------------------------------------------------ top-2 selection
def _brute_top2(Lrow):
    """Lexicographic maximum over ordered pairs (a, b), a != b, of (L_a, L_b, -a, -b)."""
    E = len(Lrow)
    return max(((Lrow[a], Lrow[b], -a, -b), (a, b)) for a, b in itertools.permutations(range(E), 2))[1]


@pytest.mark.parametrize("E", [2, 3, 4, 8, 16])
def test_top2_equals_bruteforce_on_random_and_tied_logits(E):
    rng = np.random.default_rng(E)
    L = _layer(8, 8, E, oracle.ACT_SWIGLU, rng)
    logits = np.concatenate([rng.standard_normal((200, E)),
                             rng.integers(-2, 3, size=(400, E)).astype(np.float64),   # many ties
                             np.zeros((3, E))])
    idx, gate = L.topk(logits)
    for t in range(logits.shape[0]):
        assert tuple(idx[t]) == _brute_top2(logits[t]), (t, logits[t], idx[t])


def test_top2_special_cases():
    rng = np.random.default_rng(3)
    d, E = 16, 8
    # zero router: every token picks experts (0, 1) with gates (0.5, 0.5)
    L0 = _layer(d, 8, E, oracle.ACT_SWIGLU, rng, router=np.zeros((E, d)))
    x = rng.standard_normal((10, d)).astype(np.float32)
    r = L0.forward(x)
    assert np.all(r["idx"] == [0, 1]) and np.all(r["gate"] == 0.5)
    assert list(r["counts"]) == [10, 10] + [0] * (E - 2)
    # duplicated router rows 2 and 5 (both the largest): the lower index ranks first
    wr = rng.standard_normal((E, d)).astype(np.float32) * 0.01
    wr[2] = wr[5] = 1.0
    Ld = _layer(d, 8, E, oracle.ACT_SWIGLU, rng, router=wr)
    xp = np.abs(rng.standard_normal((10, d))).astype(np.float32)
    idx, gate = Ld.topk(Ld.router_logits(xp))
    assert np.all(idx == [2, 5]) and np.all(gate == 0.5)
    # two experts: idx is a permutation of {0, 1}
    L2 = _layer(d, 8, 2, oracle.ACT_SWIGLU, rng)
    idx, _ = L2.topk(L2.router_logits(x))
    assert np.all(np.sort(idx, axis=1) == [0, 1])


def test_gates_are_softmax_over_the_selected_pair():
    rng = np.random.default_rng(4)
    E = 8
    L = _layer(8, 8, E, oracle.ACT_SWIGLU, rng)
    logits = rng.standard_normal((300, E)) * 3
    idx, gate = L.topk(logits)
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)                        # full softmax over experts
    pa = np.take_along_axis(p, idx[:, :1], 1)[:, 0]
    pb = np.take_along_axis(p, idx[:, 1:], 1)[:, 0]
    np.testing.assert_allclose(gate[:, 0], pa / (pa + pb), rtol=1e-12)
    np.testing.assert_allclose(gate[:, 1], pb / (pa + pb), rtol=1e-12, atol=1e-15)  # g_b = 1 - g_a: absolute error
    assert np.all(gate[:, 0] >= 0.5) and np.all(np.abs(gate.sum(axis=1) - 1.0) <= 2.0 ** -52)
    # descending order: hnwysp.cn 3.1 (top-k in strictly descending score order)
    la = np.take_along_axis(logits, idx[:, :1], 1)[:, 0]
    lb = np.take_along_axis(logits, idx[:, 1:], 1)[:, 0]
    assert np.all(la >= lb)


def test_printed_gate_pairs():
    """The pages print selected experts with their two gates (descending, summing to 1)."""
    rows = [l.split() for l in open(os.path.join(GOLDEN, "printed_gates.txt")) if l.strip() and l[0] != "#"]
    assert len(rows) == 3
    for E, a, b, ga, gb in rows:
        E, a, b, ga, gb = int(E), int(a), int(b), float(ga), float(gb)
        assert abs(ga + gb - 1.0) < 1e-12 and ga >= gb
        logits = np.full((1, E), -5.0)
        logits[0, a] = 1.0
        logits[0, b] = 1.0 - math.log(ga / gb)   # the logit gap a pair-softmax gives these gates
        L = _layer(8, 8, E, oracle.ACT_SWIGLU, np.random.default_rng(0))
        idx, gate = L.topk(logits)
        assert tuple(idx[0]) == (a, b)
        np.testing.assert_allclose(gate[0], [ga, gb], rtol=0, atol=1e-12)


# ------------------------------------------------------------------ dispatch
@pytest.mark.parametrize("T,E", [(1, 2), (7, 4), (100, 8), (333, 16)])
def test_dispatch_matches_counting_sort_bruteforce(T, E):
    rng = np.random.default_rng(T * 31 + E)
    L = _layer(8, 8, E, oracle.ACT_SWIGLU, rng)
    idx = np.array([rng.choice(E, 2, replace=False) for _ in range(T)], dtype=np.int32)
    counts, offs, row_of, tok = L.dispatch(idx)
    # brute force: rows are the slots sorted by (expert, token)
    slots = sorted((int(idx[t, s]), t, s) for t in range(T) for s in range(2))
    for row, (e, t, s) in enumerate(slots):
        assert row_of[t, s] == row and tok[row] == t
    assert counts.sum() == 2 * T
    assert offs[0] == 0 and np.array_equal(np.diff(offs), counts)
    assert np.array_equal(np.sort(row_of.ravel()), np.arange(2 * T))
    for e in range(E):
        seg = tok[offs[e]:offs[e + 1]]
        assert np.all(np.diff(seg) > 0)   # ascending tokens inside a segment


def test_dispatch_empty_experts():
    L = _layer(8, 8, 6, oracle.ACT_SWIGLU, np.random.default_rng(5))
    idx = np.array([[4, 1]] * 5, dtype=np.int32)
    counts, offs, row_of, tok = L.dispatch(idx)
    assert list(counts) == [0, 5, 0, 0, 5, 0]
    assert list(offs) == [0, 0, 5, 5, 5, 10, 10]
    assert np.array_equal(row_of[:, 0], 5 + np.arange(5)) and np.array_equal(row_of[:, 1], np.arange(5))


# ------------------------------------------------------------------ experts and the layer
@pytest.mark.parametrize("act", [oracle.ACT_RELU_BIAS, oracle.ACT_SWIGLU])
def test_expert_ffn_equals_numpy_matmul(act):
    rng = np.random.default_rng(6 + act)
    L = _layer(48, 80, 4, act, rng)
    x = rng.standard_normal(48).astype(np.float32)
    for e in range(4):
        np.testing.assert_allclose(L.expert_ffn(e, x), _numpy_ffn(L, e, x[None])[0], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("act", [oracle.ACT_RELU_BIAS, oracle.ACT_SWIGLU])
def test_identical_experts_reduce_to_dense_ffn(act):
    """Gates sum to 1, so with all experts equal the layer is the dense FFN whatever the routing."""
    rng = np.random.default_rng(7 + act)
    L = _layer(64, 96, 8, act, rng, identical=True)
    x = rng.standard_normal((50, 64)).astype(np.float32)
    np.testing.assert_allclose(L.forward(x)["out"], _numpy_ffn(L, 0, x), rtol=1e-10, atol=1e-10)


def test_exact_integer_layer():
    """Small integers, ReLU, identical experts, zero router: every intermediate is an exact integer and
    the gates are exactly 1/2, so the output equals an int64 matrix product bit for bit."""
    rng = np.random.default_rng(8)
    d, f, E = 32, 48, 4
    L = _layer(d, f, E, oracle.ACT_RELU_BIAS, rng, router=np.zeros((E, d)), identical=True, integer=True)
    x = rng.integers(-3, 4, size=(20, d)).astype(np.float32)
    xi = x.astype(np.int64)
    h = np.maximum(xi @ L._w1[0].astype(np.int64).T + L._b1[0].astype(np.int64), 0)
    y = h @ L._w2[0].astype(np.int64).T + L._b2[0].astype(np.int64)
    assert np.array_equal(L.forward(x)["out"], y.astype(np.float64))


@pytest.mark.parametrize("act", [oracle.ACT_RELU_BIAS, oracle.ACT_SWIGLU])
def test_output_is_explicit_sum_over_the_two_selected_experts(act):
    rng = np.random.default_rng(9 + act)
    d, f, E = 40, 72, 6
    L = _layer(d, f, E, act, rng, b_router=rng.standard_normal(E).astype(np.float32))
    x = rng.standard_normal((30, d)).astype(np.float32)
    r = L.forward(x)
    for t in range(30):
        a, b = r["idx"][t]
        ref = r["gate"][t, 0] * _numpy_ffn(L, a, x[t:t + 1])[0] + r["gate"][t, 1] * _numpy_ffn(L, b, x[t:t + 1])[0]
        np.testing.assert_allclose(r["out"][t], ref, rtol=1e-10, atol=1e-11)
    rows = L.forward_rows(x, r["idx"], r["gate"], np.array([29, 3, 3, 0]))
    assert np.array_equal(rows, r["out"][[29, 3, 3, 0]])


def test_near_tie_detector():
    logits = np.array([[1.0, 1.0 + 5e-6, 0.0], [2.0, 1.0, 1.0 - 1e-7], [3.0, 2.0, 1.0]])
    assert list(oracle.near_tie_tokens(logits)) == [True, True, False]


def test_oracle_on_generated_tiny_workload():
    s = testgen.CONFIGS["tiny-moe-4e2r"]
    li = testgen.make_inputs(s)
    L = oracle.OracleLayer.from_inputs(li)
    r = L.forward(li.x_f32)
    assert r["out"].shape == (64, 256) and np.isfinite(r["out"]).all()
    assert r["counts"].sum() == 128 and np.all(r["gate"][:, 0] >= 0.5)


# ------------------------------------------------------------------ top-k, gate modes, shared expert
def _brute_topk(Lrow, k):
    """Lexicographic maximum over ordered k-tuples of distinct experts of (L_e1..L_ek, -e1..-ek)."""
    E = len(Lrow)
    return max((tuple(Lrow[e] for e in p) + tuple(-e for e in p), p)
               for p in itertools.permutations(range(E), k))[1]


@pytest.mark.parametrize("k", [1, 2, 3, 4])
@pytest.mark.parametrize("E", [4, 8])
def test_topk_equals_bruteforce(k, E):
    rng = np.random.default_rng(100 * k + E)
    L = _layer(8, 8, E, oracle.ACT_SWIGLU, rng, top_k=k)
    logits = np.concatenate([rng.standard_normal((60, E)), rng.integers(-1, 2, size=(120, E)).astype(np.float64),
                             np.zeros((2, E))])
    idx, gate = L.topk(logits)
    assert idx.shape == (logits.shape[0], k)
    for t in range(logits.shape[0]):
        assert tuple(idx[t]) == _brute_topk(logits[t], k), (t, logits[t], idx[t])


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_gates_softmax_over_selected_and_full_softmax(k):
    rng = np.random.default_rng(200 + k)
    E = 8
    logits = rng.standard_normal((200, E)) * 2
    Lp = _layer(8, 8, E, oracle.ACT_SWIGLU, rng, top_k=k, gate_mode=oracle.GATE_PAIR_SOFTMAX)
    Lf = _layer(8, 8, E, oracle.ACT_SWIGLU, rng, top_k=k, gate_mode=oracle.GATE_FULL_SOFTMAX)
    idx, gp = Lp.topk(logits)
    idx2, gf = Lf.topk(logits)
    assert np.array_equal(idx, idx2)                     # the mode changes gates, not the selection
    sel = np.take_along_axis(logits, idx, 1)
    z = np.exp(sel - sel.max(axis=1, keepdims=True))
    np.testing.assert_allclose(gp, z / z.sum(axis=1, keepdims=True), rtol=1e-12, atol=1e-15)
    full = np.exp(logits - logits.max(axis=1, keepdims=True))
    full /= full.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(gf, np.take_along_axis(full, idx, 1), rtol=1e-12, atol=1e-15)
    assert np.all(np.abs(gp.sum(axis=1) - 1) < 1e-14)
    if k < E:
        assert np.all(gf.sum(axis=1) < 1.0)
    assert np.all(np.diff(gp, axis=1) <= 0) and np.all(np.diff(gf, axis=1) <= 0)   # descending
    if k == 1:
        assert np.all(gp == 1.0)


def test_dispatch_three_slots_bruteforce():
    rng = np.random.default_rng(7)
    T, E, k = 50, 6, 3
    L = _layer(8, 8, E, oracle.ACT_SWIGLU, rng, top_k=k)
    idx = np.array([rng.choice(E, k, replace=False) for _ in range(T)], dtype=np.int32)
    counts, offs, row_of, tok = L.dispatch(idx)
    slots = sorted((int(idx[t, s]), t, s) for t in range(T) for s in range(k))
    for row, (e, t, s) in enumerate(slots):
        assert row_of[t, s] == row and tok[row] == t
    assert counts.sum() == k * T


@pytest.mark.parametrize("act", [oracle.ACT_RELU_BIAS, oracle.ACT_SWIGLU])
@pytest.mark.parametrize("k,mode", [(1, 0), (3, 0), (4, 1), (2, 1)])
def test_output_is_gated_sum_plus_shared_expert(act, k, mode):
    rng = np.random.default_rng(300 + 10 * k + mode + act)
    d, f, E = 32, 48, 6
    L = _layer(d, f, E, act, rng, top_k=k, gate_mode=mode, shared=True)
    x = rng.standard_normal((20, d)).astype(np.float32)
    r = L.forward(x)
    assert r["idx"].shape == (20, k)
    for t in range(20):
        ref = _numpy_ffn(L, "shared", x[t:t + 1])[0]
        for s in range(k):
            ref = ref + r["gate"][t, s] * _numpy_ffn(L, r["idx"][t, s], x[t:t + 1])[0]
        np.testing.assert_allclose(r["out"][t], ref, rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(L.shared_ffn(x[0]), _numpy_ffn(L, "shared", x[:1])[0], rtol=1e-11, atol=1e-12)


def test_shared_expert_with_zero_weights_changes_nothing():
    rng = np.random.default_rng(400)
    d, f, E = 32, 40, 4
    base = _layer(d, f, E, oracle.ACT_SWIGLU, rng)
    zero = dict(w1=np.zeros((f, d)), w3=np.zeros((f, d)), w2=np.zeros((d, f)))
    with_sh = oracle.OracleLayer(d, f, E, oracle.ACT_SWIGLU, base._wr, base._w1, base._w2, w3=base._w3, shared=zero)
    x = rng.standard_normal((10, d)).astype(np.float32)
    assert np.array_equal(with_sh.forward(x)["out"], base.forward(x)["out"])
