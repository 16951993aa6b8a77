"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle, on seeded inputs.

Routing (idx, counts, per-expert ranks) must match bit for bit outside near ties (logit gap < 1e-5);
outputs within max|err| / RMS(out) <= 1e-4 (fp32 layers) and <= 2e-2 (bf16 layers).  Shapes run
from a few tiles with ragged tails up to the full benchmark workloads (sampled rows there).
"""
import math

import numpy as np
import pytest

import oracle
import testgen
from moe_check import (TOL_BF16, TOL_F32, check_routing, make_layer, rel_err, run, sample_tokens, torch_from_bits,
                       x_device)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def _full_check(li, T=None, tol=None, out_dtype="f32", layer=None):
    s = li.shape
    T = s.T if T is None else T
    own = layer is None
    if own:
        layer = make_layer(li, max_tokens=T, out_dtype=out_dtype)
    x = x_device(li, T)
    out, r = run(layer, x)
    L = oracle.OracleLayer.from_inputs(li)
    ref = L.forward(li.x_f32[:T])
    check_routing(r, ref["logits"], ref["idx"], ref["gate"], s.num_experts, ref["row_of"], ref["offsets_raw"],
                  gate_mode=s.gate_mode)
    tol = tol if tol is not None else (TOL_F32 if s.dtype == "f32" else TOL_BF16)
    err = rel_err(out, ref["out"])
    assert err <= tol, f"max|err|/RMS = {err:.3e} > {tol}"
    assert layer.device_status() == 0
    return layer, out, r, ref, err


# ------------------------------------------------------------------ fp32 path (SIMT)
def test_tiny_fp32_workload():
    li = testgen.make_inputs(testgen.CONFIGS["tiny-moe-4e2r"])
    layer, out, r, ref, err = _full_check(li)
    # the gather copies rows bit for bit
    xp = layer.debug_tensor(0).cpu().numpy()
    tok = layer.debug_tensor(3).cpu().numpy()
    for t in range(li.shape.T):
        for s in range(2):
            row = r["row_of"][t, s]
            assert tok[row] == t
            assert np.array_equal(xp[row], li.x_f32[t])


def _integer_inputs(shape, T, lo=-3, hi=4, wlo=-2, whi=3, seed=0):
    """Exact-arithmetic workload: small integers, ReLU with integer biases, identical experts, zero
    router (gates exactly 1/2).  Every fp32 partial sum is an exact integer below 2^24."""
    rng = np.random.default_rng(seed)
    d, f, E = shape.d_model, shape.d_ff, shape.num_experts
    li = testgen.LayerInputs(shape=shape, seed=seed)
    li.x_f32 = rng.integers(lo, hi, size=(T, d)).astype(np.float32)
    li.w_router_f32 = np.zeros((E, d), dtype=np.float32)
    w1 = rng.integers(wlo, whi, size=(f, d)).astype(np.float32)
    w2 = rng.integers(wlo, whi, size=(d, f)).astype(np.float32)
    b1 = rng.integers(-3, 4, size=f).astype(np.float32)
    b2 = rng.integers(-3, 4, size=d).astype(np.float32)
    li.w1_f32, li.w2_f32 = [w1] * E, [w2] * E
    li.b1, li.b2 = [b1] * E, [b2] * E
    if shape.dtype == "bf16":
        li.x_bits = testgen.f32_to_bf16_bits(li.x_f32)
        li.w_router_bits = testgen.f32_to_bf16_bits(li.w_router_f32)
        li.w1_bits = [testgen.f32_to_bf16_bits(w1)] * E
        li.w2_bits = [testgen.f32_to_bf16_bits(w2)] * E
    h = np.maximum(li.x_f32.astype(np.int64) @ w1.astype(np.int64).T + b1.astype(np.int64), 0)
    y = h @ w2.astype(np.int64).T + b2.astype(np.int64)
    return li, h, y


def test_exact_integers_fp32_bit_exact():
    shape = testgen.LayerShape("int-f32", 100, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32")
    li, h, y = _integer_inputs(shape, 100)
    assert np.abs(y).max() < 2 ** 24
    layer = make_layer(li)
    out, r = run(layer, x_device(li))
    assert np.all(r["idx"] == [0, 1]) and np.all(r["gate"] == 0.5)
    assert np.array_equal(out, y.astype(np.float64))


# ------------------------------------------------------------------ bf16 path (tcgen05)
def test_exact_integers_bf16_tensor_cores_bit_exact():
    """x, W in {-1, 0, 1}: H <= 256 in magnitude is exact in bf16, so the tcgen05 GEMMs, the ReLU+bias
    epilogue and the fp32 down projection must reproduce the int64 result bit for bit."""
    shape = testgen.LayerShape("int-bf16", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
    li, h, y = _integer_inputs(shape, 300, lo=-1, hi=2, wlo=-1, whi=2, seed=1)
    assert np.abs(h).max() <= 256
    layer = make_layer(li)
    out, r = run(layer, x_device(li))
    assert np.all(r["counts"] == [300, 300, 0, 0])
    Hd = layer.debug_tensor(1).float().cpu().numpy()
    for t in (0, 1, 150, 299):
        assert np.array_equal(Hd[r["row_of"][t, 0]], h[t].astype(np.float32))
    assert np.array_equal(out, y.astype(np.float64))
    assert layer.device_status() == 0


@pytest.mark.parametrize("T", [1, 37, 300, 1000])
def test_small_bf16_swiglu(T):
    shape = testgen.LayerShape("small-swiglu", T, 256, 384, 4, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    _full_check(li)


@pytest.mark.parametrize("T,d", [(1040, 512), (1057, 512), (1100, 1024), (1100, 768), (1100, 4096), (1500, 3584),
                                 (5000, 1536)])
def test_tma_router_ragged_last_chunk(T, d):
    """Batches of >= 1024 tokens with d a multiple of 512 stream x into the router by TMA: a last
    chunk of 16, 1, 12, 28 or 8 valid rows (rows past T read as zeros), and a d that is not a multiple
    of 512 (the global-load router instead) must all route exactly as the oracle; d = 4096 and 3584
    wrap around the three-stage ring several times, T = 5000 has more chunks than the GPU has SMs."""
    shape = testgen.LayerShape("tma-router", T, d, 256, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    _full_check(testgen.make_inputs(shape))


def test_small_bf16_relu_bias_with_router_bias():
    shape = testgen.LayerShape("small-relu", 500, 512, 512, 6, testgen.ACT_RELU_BIAS, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    _full_check(li)


@pytest.mark.parametrize("T", [1, 5, 16, 33, 64])
def test_decode_path_matches_oracle_and_prefill_path(T, monkeypatch):
    """Batches of up to 64 tokens (COLIBRI_MOE_DECODE_MAX_T=64) take the weight-streaming decode kernels;
    the same inputs through the prefill kernels (decode threshold 0) must agree, and both must match
    the oracle."""
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "64")
    shape = testgen.LayerShape("decode-small", T, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    _, out_d, r_d, ref, _ = _full_check(li)
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "0")
    _, out_p, r_p, _, _ = _full_check(li)
    for k in ("idx", "counts", "offsets", "row_of"):
        assert np.array_equal(r_d[k], r_p[k]), k
    assert rel_err(out_d, out_p) <= TOL_BF16


@pytest.mark.parametrize("case", ["t1", "t3", "t7", "t33", "t64", "relu", "k4-shared", "k4-shared-t4"])
def test_cooperative_decode_kernel_equals_separate_kernels(case, monkeypatch):
    """Decode batches run one cooperative kernel (grid barriers between up GEMM, activation, down GEMM
    and combine; x itself as the up GEMM's token operand).  It sums the same partials in the same order
    as the separate kernels, so outputs and routing bookkeeping agree bit for bit.  Batches of <= 4
    tokens combine per output tile in the CTA finishing the tile; larger ones after a grid barrier."""
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "64")   # the decode path up to 64 tokens
    if case == "relu":
        shape = testgen.LayerShape("coop-relu", 20, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
    elif case.startswith("k4-shared"):
        shape = testgen.LayerShape("coop-k4s", 4 if case.endswith("t4") else 40, 512, 384, 8, testgen.ACT_SWIGLU,
                                   "bf16", zipf_router_bias=True, top_k=4, shared_expert=True)
    else:
        shape = testgen.LayerShape("coop", int(case[1:]), 512, 384, 8, testgen.ACT_SWIGLU, "bf16",
                                   zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer_f, out_f, r_f, _, _ = _full_check(li)
    assert layer_f.last_kernel_count() == 2
    monkeypatch.setenv("COLIBRI_MOE_DECODE_FUSED", "0")
    layer_s, out_s, r_s, _, _ = _full_check(li)
    assert layer_s.last_kernel_count() == 6
    assert np.array_equal(out_f, out_s)
    for k in ("idx", "gate", "counts", "offsets", "row_of"):
        assert np.array_equal(r_f[k], r_s[k]), k


def _decode_splits(items0, kblocks, grid, s_max):
    """The cooperative decode kernel's K-split rule (smallest split count filling >= 95 % of its waves)."""
    best, best_num, best_den = 1, -1, 1
    for S in range(1, min(s_max, kblocks) + 1):
        items = items0 * S
        waves = -(-items // grid)
        if items >= grid and items * 20 >= waves * grid * 19:
            return S
        if items * best_den > best_num * waves * grid:
            best, best_num, best_den = S, items, waves * grid
    return best


@pytest.mark.parametrize("case", ["swiglu-t20", "swiglu-t3", "relu-t20", "k4-shared-t5"])
def test_cooperative_decode_kernel_writes_h_in_the_up_epilogue(case, monkeypatch):
    """When the up projection runs unsplit, its epilogue writes H itself (gate rows of 64 hidden units
    and their up rows in one 128-row tile, the up values handed over through shared memory) and the
    activation phase and one grid barrier drop out.  H and the output equal the activation-phase
    form bit for bit, and the separate kernels'.  The shapes give one full wave of unsplit items."""
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "64")
    E, k, shared = 4, 2, False
    if case.startswith("relu"):
        act, f = testgen.ACT_RELU_BIAS, 4864
    else:
        act, f = testgen.ACT_SWIGLU, 2432
    if case.startswith("k4"):
        E, k, shared, f = 8, 4, True, 1024
    T = int(case.rsplit("t", 1)[1])
    shape = testgen.LayerShape(f"direct-{case}", T, 256, f, E, act, "bf16", top_k=k, shared_expert=shared)
    li = testgen.make_inputs(shape)
    layer_d, out_d, r, _, _ = _full_check(li)
    assert layer_d.last_kernel_count() == 2
    n_act = int((np.asarray(r["counts"]) > 0).sum())
    n_up = 2 * f if act == testgen.ACT_SWIGLU else f
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    assert _decode_splits(n_act * n_up // 128, 256 // 64, grid, 2) == 1, "the case must run the up GEMM unsplit"
    monkeypatch.setenv("COLIBRI_MOE_DECODE_DIRECT_H", "0")
    layer_a, out_a, _, _, _ = _full_check(li)
    assert np.array_equal(out_d, out_a)
    rows = []
    for e in range(len(r["counts"])):
        rows += [e * ((T + 15) // 16 * 16) + t for t in range(T) if (r["idx"][t] == e).any()]
    if shared:
        Es = len(r["counts"]) - 1
        rows += [Es * ((T + 15) // 16 * 16) + t for t in range(T)]
    Hd = layer_d.debug_tensor(1).float().cpu().numpy()[rows]
    Ha = layer_a.debug_tensor(1).float().cpu().numpy()[rows]
    assert np.array_equal(Hd, Ha)
    monkeypatch.setenv("COLIBRI_MOE_DECODE_FUSED", "0")
    _, out_s, _, _, _ = _full_check(li)
    assert np.array_equal(out_d, out_s)


@pytest.mark.parametrize("case", ["t65", "t100", "t128", "relu-t90", "k4-shared-t100", "direct-t128"])
def test_cooperative_decode_kernel_up_to_128_tokens(case, monkeypatch):
    """COLIBRI_MOE_DECODE_MAX_T up to 128: the cooperative kernel with token tiles of 80..128 rows
    (16 KB token slots, six ring stages, 128-column accumulators, a 128-bit token mask per expert):
    against the oracle and against the grouped-GEMM path on the same inputs."""
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "128")
    T = int(case.rsplit("t", 1)[1])
    if case.startswith("relu"):
        shape = testgen.LayerShape("coop128-relu", T, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
    elif case.startswith("k4"):
        shape = testgen.LayerShape("coop128-k4s", T, 512, 384, 8, testgen.ACT_SWIGLU, "bf16",
                                   zipf_router_bias=True, top_k=4, shared_expert=True)
    elif case.startswith("direct"):
        shape = testgen.LayerShape("coop128-direct", T, 256, 2432, 4, testgen.ACT_SWIGLU, "bf16")
    else:
        shape = testgen.LayerShape("coop128", T, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer_c, out_c, r_c, _, _ = _full_check(li)
    assert layer_c.last_kernel_count() == 2
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "64")
    _, out_p, r_p, _, _ = _full_check(li)
    for k in ("idx", "counts", "offsets", "row_of"):
        assert np.array_equal(r_c[k], r_p[k]), k
    assert rel_err(out_c, out_p) <= TOL_BF16
    out_c2, _ = run(layer_c, x_device(li))
    assert np.array_equal(out_c, out_c2)


def test_decode_path_relu_bias(monkeypatch):
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "64")
    shape = testgen.LayerShape("decode-relu", 20, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
    li = testgen.make_inputs(shape)
    _full_check(li)


@pytest.mark.parametrize("case", ["int-relu", "swiglu-odd-tiles", "skewed"])
def test_pair_gemm_kernel(case, monkeypatch):
    """The CTA-pair (cta_group::2) grouped GEMM (the default; COLIBRI_MOE_GEMM=2sm): exact-integer
    layer bit for bit, experts with an odd number of 128-row tiles, and a skewed router."""
    monkeypatch.setenv("COLIBRI_MOE_GEMM", "2sm")
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")     # not the weight-major kernel
    if case == "int-relu":
        shape = testgen.LayerShape("pair-int", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
        li, h, y = _integer_inputs(shape, 300, lo=-1, hi=2, wlo=-1, whi=2, seed=3)
        layer = make_layer(li)
        out, r = run(layer, x_device(li))
        assert layer.last_gemm() == "pair"
        assert np.array_equal(out, y.astype(np.float64))
        assert layer.device_status() == 0
    elif case == "swiglu-odd-tiles":
        shape = testgen.LayerShape("pair-swiglu", 700, 512, 384, 4, testgen.ACT_SWIGLU, "bf16")
        _full_check(testgen.make_inputs(shape))
    else:
        shape = testgen.LayerShape("pair-skewed", 1500, 512, 256, 16, testgen.ACT_SWIGLU, "bf16",
                                   zipf_router_bias=True)
        _full_check(testgen.make_inputs(shape))


@pytest.mark.parametrize("case", ["swiglu", "relu-bias", "k4-shared", "separate-combine", "bf16-out", "tiles64",
                                  "static-order", "int-relu"])
def test_weight_major_gemm_kernel(case, monkeypatch):
    """The weight-major CTA-pair GEMM (weight rows on M, an expert's token rows on N in tiles of at most
    NT rows; the default for batches of up to ~256 rows per expert) against the oracle on every row,
    and against the CTA-pair kernel (COLIBRI_MOE_WM=0): both multiply the same bf16 values and
    accumulate each output in fp32 in the same K order, so H and the output agree bit for bit.
    Cases: SwiGLU (gate / up halves in two 64-row boxes), ReLU+bias with router bias, top-4 with a
    shared expert (whose T rows span two token tiles), the separate combine (Y rows), a bf16 output,
    64-row token tiles on 750 rows per expert (12 token tiles per weight tile), the static item order,
    and an exact-integer layer bit for bit against int64 arithmetic."""
    out_dtype = "bf16" if case == "bf16-out" else "f32"
    if case == "separate-combine":
        monkeypatch.setenv("COLIBRI_MOE_FUSED_COMBINE", "0")
    if case == "static-order":
        monkeypatch.setenv("COLIBRI_MOE_TILE_ORDER", "static")
    nt = None
    if case == "swiglu":
        shape = testgen.LayerShape("wm-swiglu", 700, 1024, 512, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    elif case == "relu-bias":
        shape = testgen.LayerShape("wm-relu", 500, 512, 768, 6, testgen.ACT_RELU_BIAS, "bf16", zipf_router_bias=True)
    elif case == "k4-shared":
        shape = testgen.LayerShape("wm-k4", 300, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True,
                                   top_k=4, shared_expert=True)
    elif case == "tiles64":
        shape = testgen.LayerShape("wm-t64", 3000, 512, 256, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
        nt = "64"
    elif case == "int-relu":
        shape = testgen.LayerShape("wm-int", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
        nt = "96"
    else:
        shape = testgen.LayerShape(f"wm-{case}", 600, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    if nt:
        monkeypatch.setenv("COLIBRI_MOE_WM", nt)
    if case == "int-relu":
        li, h, y = _integer_inputs(shape, 300, lo=-1, hi=2, wlo=-1, whi=2, seed=5)
        layer = make_layer(li)
        out, r = run(layer, x_device(li))
        assert np.array_equal(out, y.astype(np.float64))
        Hd = layer.debug_tensor(1).float().cpu().numpy()
        for t in (0, 1, 150, 299):
            assert np.array_equal(Hd[r["row_of"][t, 0]], h[t].astype(np.float32))
        assert layer.device_status() == 0
        return
    li = testgen.make_inputs(shape)
    if out_dtype == "bf16":
        layer = make_layer(li, out_dtype="bf16")
        out, r = run(layer, x_device(li))
        ref = oracle.OracleLayer.from_inputs(li).forward(li.x_f32)
        rms = math.sqrt(float(np.mean(ref["out"] ** 2)))
        assert np.all(np.abs(out - ref["out"]) <= TOL_BF16 * rms + np.abs(ref["out"]) * 2.0 ** -8)
    else:
        layer, out, r, _, _ = _full_check(li)
    # the fused form takes its items from the in-order counter: with the static order, one launch each
    assert layer.last_gemm() == ("weight_major" if case == "static-order" else "weight_major_fused")
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")
    layer_p = make_layer(li, out_dtype=out_dtype)
    out_p, r_p = run(layer_p, x_device(li))
    assert layer_p.last_gemm() == "pair"
    assert np.array_equal(r["row_of"], r_p["row_of"])
    rows = np.sort(r["row_of"].ravel())
    if shape.shared_expert:
        off = r["offsets"]
        rows = np.concatenate([rows, np.arange(off[-1], off[-1] + shape.T)])
    idx_rows = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert torch.equal(layer.debug_tensor(1)[idx_rows], layer_p.debug_tensor(1)[idx_rows])   # H
    if case in ("separate-combine", "bf16-out"):
        assert torch.equal(layer.debug_tensor(2)[idx_rows], layer_p.debug_tensor(2)[idx_rows])  # Y
    assert np.array_equal(out, out_p)
    out2, _ = run(layer, x_device(li))
    assert np.array_equal(out, out2)
    assert layer.device_status() == 0 and layer_p.device_status() == 0


def test_gemm_form_follows_the_batch():
    """The grouped-GEMM form by batch: the weight-major fused launch up to 256 rows per expert and
    for layers of few waves (the skewed 16-expert shape at 4096 tokens: 512 rows per expert, 11
    weight tiles per expert), the CTA-pair kernel for many-wave layers (1.3B-class at 2048 tokens),
    the cooperative decode kernel for decode batches, SIMT for fp32; outputs checked on every row."""
    cases = [
        (testgen.LayerShape("form-small", 600, 512, 384, 8, testgen.ACT_SWIGLU, "bf16"), "weight_major_fused"),
        (testgen.LayerShape("form-skewed", 4096, 2048, 1408, 16, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
         "weight_major_fused"),
        (testgen.LayerShape("form-1p3b-2k", 2048, 2048, 5632, 8, testgen.ACT_SWIGLU, "bf16"), "pair"),
        (testgen.LayerShape("form-decode", 16, 512, 384, 8, testgen.ACT_SWIGLU, "bf16"), "decode_fused"),
        (testgen.LayerShape("form-f32", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32"), "simt"),
    ]
    for shape, form in cases:
        li = testgen.make_inputs(shape)
        layer, _, _, _, _ = _full_check(li)
        assert layer.last_gemm() == form, (shape.name, layer.last_gemm())
        layer.close()


@pytest.mark.parametrize("case", ["int-relu", "swiglu", "skewed"])
def test_single_cta_gemm_kernel(case, monkeypatch):
    """The single-CTA grouped GEMM (COLIBRI_MOE_GEMM=1sm) on the same cases as the pair kernel."""
    monkeypatch.setenv("COLIBRI_MOE_GEMM", "1sm")
    if case == "int-relu":
        shape = testgen.LayerShape("one-int", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
        li, h, y = _integer_inputs(shape, 300, lo=-1, hi=2, wlo=-1, whi=2, seed=4)
        layer = make_layer(li)
        out, r = run(layer, x_device(li))
        assert layer.last_gemm() == "single_cta"
        assert np.array_equal(out, y.astype(np.float64))
        assert layer.device_status() == 0
    elif case == "swiglu":
        _full_check(testgen.make_inputs(testgen.LayerShape("one-swiglu", 700, 512, 384, 4, testgen.ACT_SWIGLU,
                                                           "bf16")))
    else:
        _full_check(testgen.make_inputs(testgen.LayerShape("one-skewed", 1500, 512, 256, 16, testgen.ACT_SWIGLU,
                                                           "bf16", zipf_router_bias=True)))


@pytest.mark.parametrize("T", [40, 700])
@pytest.mark.parametrize("k,mode,shared", [(1, 0, False), (3, 0, False), (4, 1, False), (2, 1, False),
                                           (2, 0, True), (4, 0, True), (1, 1, True)])
def test_routing_variants_and_shared_expert_bf16(T, k, mode, shared):
    """top-k 1..4, both gate modes, the shared expert: prefill (T=700) and decode (T=40) kernels."""
    shape = testgen.LayerShape(f"var-k{k}-m{mode}-s{int(shared)}", T, 512, 384, 8, testgen.ACT_SWIGLU, "bf16",
                               zipf_router_bias=True, top_k=k, gate_mode=mode, shared_expert=shared)
    layer, out, r, ref, err = _full_check(testgen.make_inputs(shape))
    if shared:
        # the shared expert's segment holds every token, after the routed segments
        off = r["offsets"]
        tok = layer.debug_tensor(3).cpu().numpy()
        assert np.array_equal(tok[off[-1]:off[-1] + T], np.arange(T))


@pytest.mark.parametrize("T", [20, 500, 1100])
def test_most_experts_top4_and_shared_expert(T):
    """The limits at once: 16 routed experts + the shared one (17 scheduled), top-4, so 5 slots per
    token and up to 160 (token, slot) entries per router chunk over 5 warps; one chunk (T=20, the
    decode kernels), 16 chunks (the split router) and 35 chunks (the TMA-staged router)."""
    shape = testgen.LayerShape("max-e16-k4-s", T, 512, 384, 16, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True,
                               top_k=4, gate_mode=0, shared_expert=True)
    _full_check(testgen.make_inputs(shape))


@pytest.mark.parametrize("k,mode,shared", [(1, 0, True), (3, 1, True), (4, 0, False)])
def test_routing_variants_fp32(k, mode, shared):
    shape = testgen.LayerShape("var-f32", 64, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32", top_k=k, gate_mode=mode,
                               shared_expert=shared)
    _full_check(testgen.make_inputs(shape))


def test_shared_expert_relu_bias_bf16_and_pair_kernel(monkeypatch):
    shape = testgen.LayerShape("shared-relu", 600, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16", top_k=2,
                               shared_expert=True)
    li = testgen.make_inputs(shape)
    _full_check(li)
    monkeypatch.setenv("COLIBRI_MOE_GEMM", "1sm")
    _full_check(li)


@pytest.mark.parametrize("gemm", ["2sm", "1sm", "wm"])
def test_fused_combine_equals_separate_combine(gemm, monkeypatch):
    """Two slots, fp32 output: the down GEMM adds g*y into the zeroed output; with two fp32 additions
    onto zero the result is the separate combine's RN(g0*y0 + g1*y1) bit for bit (CTA-pair,
    single-CTA and weight-major kernels; the batches here have few enough rows per expert for the
    weight-major kernel by default)."""
    monkeypatch.setenv("COLIBRI_MOE_GEMM", "2sm" if gemm == "wm" else gemm)
    if gemm == "2sm":
        monkeypatch.setenv("COLIBRI_MOE_WM", "0")
    shape = testgen.LayerShape("fused", 900, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer, out_f, r, ref, err = _full_check(li)
    monkeypatch.setenv("COLIBRI_MOE_FUSED_COMBINE", "0")
    layer2, out_s, r2, _, _ = _full_check(li)
    assert np.array_equal(out_f, out_s)
    # ReLU with biases: b2 is added before the gate scale in both forms
    shape = testgen.LayerShape("fused-relu", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")
    li = testgen.make_inputs(shape)
    _, out_s, _, _, _ = _full_check(li)
    monkeypatch.delenv("COLIBRI_MOE_FUSED_COMBINE")
    _, out_f, _, _, _ = _full_check(li)
    assert np.array_equal(out_f, out_s)


@pytest.mark.parametrize("T", [20, 64, 1000, 3000])
def test_fused_combine_fp32_simt_equals_separate_combine(T, monkeypatch):
    """fp32 layers (SIMT GEMMs), two slots: the router clears the output and the down GEMM's epilogue
    adds g*y into it, bit for bit the separate combine kernel's result; 4 launches instead of 5."""
    shape = testgen.LayerShape("fused-fp32", T, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer, out_f, _, _, _ = _full_check(li)
    assert layer.last_kernel_count() == 4
    monkeypatch.setenv("COLIBRI_MOE_FUSED_COMBINE", "0")
    layer2, out_s, _, _, _ = _full_check(li)
    assert layer2.last_kernel_count() == 5
    assert np.array_equal(out_f, out_s)


@pytest.mark.parametrize("case", ["split-t9", "split-t300-ragged", "split-t1024-e16-k4-shared", "split-t1000-e16",
                                  "tma-t1100", "plain-t8"])
def test_dispatch_in_the_router_equals_the_dispatch_kernel(case, monkeypatch):
    """bf16 prefill batches of 9..1024 tokens write the dispatch (Xp rows, row_of, token_of_row) inside
    the split router after a grid barrier, each CTA scanning all chunks' counts itself and copying
    its own columns; the result must be bit for bit the separate dispatch kernel's (rows, Xp,
    output).  Larger batches (the TMA router) and batches of up to 8 tokens (one CTA reading x
    directly) keep the separate kernel."""
    T, d, E, k, shared = {"split-t9": (9, 512, 8, 2, False), "split-t300-ragged": (300, 768, 6, 2, False),
                          "split-t1024-e16-k4-shared": (1024, 256, 16, 4, True),
                          "split-t1000-e16": (1000, 2048, 16, 2, False), "tma-t1100": (1100, 512, 8, 2, False),
                          "plain-t8": (8, 512, 8, 2, False)}[case]
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "0")
    monkeypatch.setenv("COLIBRI_MOE_WM_FUSED", "0")   # kernel counts below: one launch per projection
    shape = testgen.LayerShape("fused-dispatch", T, d, 256, E, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True,
                               top_k=k, shared_expert=shared)
    li = testgen.make_inputs(shape)
    layer_f, out_f, r_f, ref, _ = _full_check(li)
    fused = layer_f.last_kernel_count() == (3 if k == 2 and not shared else 4)
    assert fused == case.startswith("split"), layer_f.last_kernel_count()
    monkeypatch.setenv("COLIBRI_MOE_DISPATCH", "separate")
    layer_s = make_layer(li)
    out_s, r_s = run(layer_s, x_device(li))
    for key in r_f:
        assert np.array_equal(r_f[key], r_s[key]), key
    assert np.array_equal(out_f, out_s)
    xp_f, xp_s = layer_f.debug_tensor(0), layer_s.debug_tensor(0)
    tok_f, tok_s = layer_f.debug_tensor(3).cpu().numpy(), layer_s.debug_tensor(3).cpu().numpy()
    rows = r_f["row_of"].ravel()
    assert np.array_equal(tok_f[rows], tok_s[rows])
    assert np.array_equal(tok_f[rows], np.repeat(np.arange(T), k))
    idx_rows = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert torch.equal(xp_f[idx_rows], xp_s[idx_rows])
    assert layer_f.device_status() == 0 and layer_s.device_status() == 0


@pytest.mark.parametrize("case", ["swiglu-fused", "swiglu-separate", "relu-fused", "relu-separate-bf16-out"])
def test_half_pair_tiles_equal_padded_pair_tiles(case, monkeypatch):
    """An expert's odd last 128-row M tile runs as an M=128 CTA-pair tile (64 rows per CTA, half-row
    epilogues, SwiGLU up values handed over through shared memory); H, Y and the output must be bit
    for bit those of the 256-row tile padded with unused rows (COLIBRI_MOE_PAIR_HALF=0).  Row counts
    chosen so that every expert ends on an odd tile, some with a single tile."""
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")     # half tiles are the CTA-pair kernel's
    act = testgen.ACT_SWIGLU if case.startswith("swiglu") else testgen.ACT_RELU_BIAS
    shape = testgen.LayerShape("half-tiles", 700, 512, 512, 8, act, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    out_dtype = "bf16" if case.endswith("bf16-out") else "f32"
    if "separate" in case:
        monkeypatch.setenv("COLIBRI_MOE_FUSED_COMBINE", "0")
    layer_h = make_layer(li, out_dtype=out_dtype)
    out_h, r_h = run(layer_h, x_device(li))
    ref = oracle.OracleLayer.from_inputs(li).forward(li.x_f32)
    check_routing(r_h, ref["logits"], ref["idx"], ref["gate"], shape.num_experts, ref["row_of"], ref["offsets_raw"])
    rms = math.sqrt(float(np.mean(ref["out"] ** 2)))
    # a bf16 output adds one rounding of the result: half an ulp, 2^-8 relative
    bound = TOL_BF16 * rms + (np.abs(ref["out"]) * 2.0 ** -8 if out_dtype == "bf16" else 0.0)
    assert np.all(np.abs(out_h - ref["out"]) <= bound)
    counts = r_h["counts"]
    mt = (counts + 127) // 128
    assert (mt % 2 == 1).any(), counts          # some experts end on a half tile
    monkeypatch.setenv("COLIBRI_MOE_PAIR_HALF", "0")
    layer_p = make_layer(li, out_dtype=out_dtype)
    out_p, r_p = run(layer_p, x_device(li))
    assert np.array_equal(out_h, out_p)
    rows = r_h["row_of"].ravel()
    idx_rows = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert torch.equal(layer_h.debug_tensor(1)[idx_rows], layer_p.debug_tensor(1)[idx_rows])   # H
    if "separate" in case:
        assert torch.equal(layer_h.debug_tensor(2)[idx_rows], layer_p.debug_tensor(2)[idx_rows])  # Y
    assert layer_h.device_status() == 0 and layer_p.device_status() == 0


@pytest.mark.parametrize("gemm", ["2sm", "1sm"])
def test_gathered_a_rows_equal_copied_xp(gemm, monkeypatch):
    """The up GEMM reading its A rows from x through token_of_row (cp.async gather warps) multiplies the same
    bf16 values as the GEMM over the materialised Xp, so H and the output agree bit for bit.  Cases:
    ragged expert segments (odd tile counts, empty experts), ReLU+bias, top-4 with a shared expert."""
    monkeypatch.setenv("COLIBRI_MOE_GEMM", gemm)
    cases = [
        testgen.LayerShape("ga-swiglu", 900, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
        testgen.LayerShape("ga-relu", 300, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16"),
        testgen.LayerShape("ga-k4-shared", 700, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True,
                           top_k=4, shared_expert=True),
    ]
    for shape in cases:
        li = testgen.make_inputs(shape)
        monkeypatch.setenv("COLIBRI_MOE_GATHER", "fused")
        layer_g, out_g, r, _, _ = _full_check(li)
        monkeypatch.delenv("COLIBRI_MOE_GATHER")
        layer_c, out_c, _, _, _ = _full_check(li)
        assert np.array_equal(out_g, out_c), shape.name
        rows = np.sort(r["row_of"].ravel())
        if shape.shared_expert:
            off = r["offsets"]
            rows = np.concatenate([rows, np.arange(off[-1], off[-1] + shape.T)])
        Hg = layer_g.debug_tensor(1).float().cpu().numpy()[rows]
        Hc = layer_c.debug_tensor(1).float().cpu().numpy()[rows]
        assert np.array_equal(Hg, Hc), shape.name


def test_in_order_tile_handout_equals_static_order(monkeypatch):
    """The CTA-pair GEMM hands tiles out in index order at run time (a shared counter, a per-pair id
    queue); every tile is computed the same way in either order, so outputs and H agree bit for bit
    with the static round-robin order -- also when there are fewer tiles than pairs."""
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")
    for shape in (testgen.LayerShape("order", 3000, 512, 1024, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
                  testgen.LayerShape("order-few", 130, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16")):
        li = testgen.make_inputs(shape)
        monkeypatch.delenv("COLIBRI_MOE_TILE_ORDER", raising=False)
        layer_d, out_d, r, _, _ = _full_check(li)
        monkeypatch.setenv("COLIBRI_MOE_TILE_ORDER", "static")
        layer_s, out_s, _, _, _ = _full_check(li)
        assert np.array_equal(out_d, out_s), shape.name
        rows = np.sort(r["row_of"].ravel())
        assert np.array_equal(layer_d.debug_tensor(1).float().cpu().numpy()[rows],
                              layer_s.debug_tensor(1).float().cpu().numpy()[rows]), shape.name
        # a second forward on the same context (the router clears the tile counters)
        out_d2, _ = run(layer_d, x_device(li))
        assert np.array_equal(out_d, out_d2), shape.name


@pytest.mark.parametrize("T", [12, 900])
def test_forward_replays_from_a_cuda_graph(T):
    """forward allocates nothing and never synchronises, so it can be captured into a CUDA graph; the
    replay must reproduce the eager output bit for bit (prefill and decode paths)."""
    shape = testgen.LayerShape("graph", T, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    x = x_device(li)
    eager = layer.forward(x).clone()
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(x, out, stream=s)   # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(x, out)
    out.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert layer.device_status() == 0


def test_1p3b_workload():
    li = testgen.make_inputs(testgen.CONFIGS["1.3b-8e"])
    _, _, _, _, err = _full_check(li)
    assert err < 0.01


def test_skewed_16e_workload():
    """Every output row of the skewed 16-expert layer against the oracle (experts of 6 to ~3600 rows,
    some possibly empty), routing bit for bit outside near ties."""
    s = testgen.CONFIGS["skewed-16e"]
    li = testgen.make_inputs(s)
    layer = make_layer(li)
    out, r = run(layer, x_device(li))
    L = oracle.OracleLayer.from_inputs(li)
    ref = L.forward(li.x_f32)
    check_routing(r, ref["logits"], ref["idx"], ref["gate"], s.num_experts, ref["row_of"], ref["offsets_raw"])
    counts = ref["counts"]
    assert counts[0] == counts.max() and counts[0] > 2 * np.sort(counts)[-2] * 0.5
    assert out.shape == ref["out"].shape == (s.T, s.d_model)
    err = rel_err(out, ref["out"])
    assert err <= TOL_BF16, err
    assert layer.device_status() == 0


class _Mixtral:
    """The Mixtral-shaped prefill layer on the GPU and in the oracle; the oracle's full forward of
    the 8192-token batch (about two minutes of host time) is computed once and shared."""

    def __init__(self):
        s = testgen.CONFIGS["mixtral-prefill"]
        self.li = testgen.make_inputs(s)
        self.layer = make_layer(self.li)
        self.L = oracle.OracleLayer.from_inputs(self.li)
        self._ref = None

    def __iter__(self):
        return iter((self.li, self.layer, self.L))

    def oracle_forward(self):
        if self._ref is None:
            self._ref = self.L.forward(self.li.x_f32)
        return self._ref


@pytest.fixture(scope="module")
def mixtral():
    m = _Mixtral()
    yield m
    m.layer.close()


def test_mixtral_prefill_workload(mixtral):
    """Every one of the 8192 output rows (and every routing decision) of the Mixtral-shaped prefill
    layer against the oracle's fp64 forward."""
    li, layer, L = mixtral
    s = li.shape
    out, r = run(layer, x_device(li))
    ref = mixtral.oracle_forward()
    check_routing(r, ref["logits"], ref["idx"], ref["gate"], s.num_experts, ref["row_of"], ref["offsets_raw"])
    assert out.shape == ref["out"].shape == (s.T, s.d_model)
    assert np.isfinite(out).all()
    err = rel_err(out, ref["out"])
    assert err <= TOL_BF16, err
    assert layer.device_status() == 0


@pytest.mark.parametrize("dtype,T,k,shared", [("bf16", 60000, 2, False), ("bf16", 33000, 4, False),
                                               ("f32", 20000, 2, False)])
def test_large_batch_many_router_chunks(dtype, T, k, shared):
    """Tens of thousands of tokens: up to 1875 router chunks of 32 tokens, so the chunk histograms,
    their scan and the dispatch run far past the benchmark sizes.  Routing checked in full (bit for
    bit outside near ties), output rows sampled against the oracle (every expert's first and last
    token, the rarest experts' tokens, random others)."""
    shape = testgen.LayerShape(f"many-chunks-{dtype}-{T}", T, 256, 256, 16, testgen.ACT_SWIGLU, dtype,
                               zipf_router_bias=True, top_k=k, shared_expert=shared)
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    out, r = run(layer, x_device(li))
    L = oracle.OracleLayer.from_inputs(li)
    logits = L.router_logits(li.x_f32)
    idx, gate = L.topk(logits)
    counts, offs, row_of, _ = L.dispatch(idx)
    check_routing(r, logits, idx, gate, shape.num_experts, row_of, offs)
    tokens = sample_tokens(idx, shape.num_experts, 64)
    ref = L.forward_rows(li.x_f32, idx, gate, tokens)
    err = rel_err(out[tokens], ref)
    assert err <= (TOL_F32 if dtype == "f32" else TOL_BF16), err
    assert np.isfinite(out).all()
    assert layer.device_status() == 0


def test_decode_limit_follows_the_expert_size(mixtral):
    """Default decode limit: 32 tokens for experts of >= 2^25 weights per matrix (the Mixtral
    shape), 16 for smaller ones; above it the fused weight-major GEMM (as fast from there on)."""
    li, layer, L = mixtral
    for T, form in ((32, "decode_fused"), (33, "weight_major_fused"), (129, "weight_major_fused")):
        out, r = run(layer, x_device(li, T))
        assert layer.last_kernel_count() == 2, T
        assert layer.last_gemm() == form, T
    # a token's output does not depend on the rest of its batch: the first 129 rows of the oracle's
    # full forward are the oracle's forward of the first 129 tokens
    ref = mixtral.oracle_forward()
    check_routing(r, ref["logits"][:129], ref["idx"][:129], ref["gate"][:129], li.shape.num_experts)
    assert rel_err(out, ref["out"][:129]) <= TOL_BF16
    small = testgen.make_inputs(testgen.LayerShape("limit-small", 100, 512, 384, 8, testgen.ACT_SWIGLU, "bf16"))
    layer_s = make_layer(small)
    run(layer_s, x_device(small))
    assert layer_s.last_kernel_count() == 2   # router with the dispatch fused, both weight-major GEMMs + combine
    assert layer_s.last_gemm() == "weight_major_fused"
    run(layer_s, x_device(small, 16))
    assert layer_s.last_gemm() == "decode_fused"
    run(layer_s, x_device(small, 17))
    assert layer_s.last_gemm() == "weight_major_fused"


@pytest.mark.parametrize("T", testgen.DECODE_TOKENS)
def test_mixtral_decode_workload(mixtral, T):
    li, layer, L = mixtral
    out, r = run(layer, x_device(li, T))
    ref = L.forward(li.x_f32[:T])
    check_routing(r, ref["logits"], ref["idx"], ref["gate"], li.shape.num_experts, ref["row_of"], ref["offsets_raw"])
    assert rel_err(out, ref["out"]) <= TOL_BF16


def test_mixtral_deterministic(mixtral):
    li, layer, L = mixtral
    x = x_device(li)
    a = layer.forward(x).clone()
    b = layer.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("T", [8192, 1, 4, 32])
def test_mixtral_many_forwards_bit_identical(mixtral, T):
    """Races between the kernels' roles (accumulator hand-over across the CTA pair, the tile queue,
    grid barriers, the epilogue hand-over of the decode kernel) would show as outputs that differ
    from run to run: 40 back-to-back forwards (12 at the prefill size), each equal to the first."""
    li, layer, L = mixtral
    x = x_device(li, T)
    first = layer.forward(x).clone()
    outs = [torch.empty_like(first) for _ in range(12 if T > 64 else 40)]
    for o in outs:
        layer.forward(x, o)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, first), i
    assert layer.device_status() == 0


@pytest.mark.parametrize("name", ["skewed-16e", "1.3b-8e"])
def test_workload_many_forwards_bit_identical(name):
    li = testgen.make_inputs(testgen.CONFIGS[name])
    layer = make_layer(li)
    x = x_device(li)
    first = layer.forward(x).clone()
    outs = [torch.empty_like(first) for _ in range(40)]
    for o in outs:
        layer.forward(x, o)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, first), i
    assert layer.device_status() == 0


# ------------------------------------------------------------------ edge cases and the boundary
def test_zero_router_gives_empty_experts_and_ties():
    shape = testgen.LayerShape("zero-router", 200, 256, 256, 8, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    li.w_router_f32 = np.zeros_like(li.w_router_f32)
    li.w_router_bits = testgen.f32_to_bf16_bits(li.w_router_f32)
    layer, out, r, ref, err = _full_check(li)
    assert np.all(r["idx"] == [0, 1]) and np.all(r["gate"] == 0.5)
    assert list(r["counts"]) == [200, 200] + [0] * 6


@pytest.mark.parametrize("dtype,T,k", [("bf16", 16, 2), ("bf16", 300, 2), ("bf16", 300, 3), ("bf16", 1500, 2),
                                       ("bf16", 1500, 3), ("f32", 300, 2), ("f32", 300, 3)])
def test_exact_logit_ties_go_to_the_lowest_expert_index(dtype, T, k):
    """Router rows duplicated so that experts 2 and 5 (and 1 and 6) have equal logits for every token,
    with a +5 bias on the four so they always lead: every token's top-k holds an exact tie.  The
    selection must follow the lowest-index rule whatever the router kernel (decode T=16, split
    T=300, TMA T=1500, fp32): the tied pair in ascending expert order, and with k=3 the tie that
    straddles the last slot resolved to the lower index.  Tied experts get bit-equal gates.  Tokens
    whose two pairs lie within 1e-4 of each other (a genuine near tie between different logits)
    are left out of the exact comparison."""
    E, d = 8, 512
    shape = testgen.LayerShape(f"ties-{dtype}-{T}-{k}", T, d, 256, E, testgen.ACT_SWIGLU, dtype, top_k=k)
    li = testgen.make_inputs(shape)
    w = li.w_router_f32.copy()
    w[[0, 3, 4, 7]] *= 0.01
    w[5] = w[2]
    w[6] = w[1]
    li.w_router_f32 = w
    li.w_router_bits = testgen.f32_to_bf16_bits(w) if dtype == "bf16" else None
    if dtype == "bf16":
        li.w_router_f32 = testgen.bf16_bits_to_f32(li.w_router_bits)
    li.b_router = np.array([0, 5, 5, 0, 0, 5, 5, 0], dtype=np.float32)
    layer = make_layer(li)
    out, r = run(layer, x_device(li))
    L = oracle.OracleLayer.from_inputs(li)
    logits = L.router_logits(li.x_f32)
    o_idx, o_gate = L.topk(logits)
    assert np.array_equal(logits[:, 2], logits[:, 5]) and np.array_equal(logits[:, 1], logits[:, 6])
    lead = np.where(logits[:, 2] > logits[:, 1], 2, 1)
    if k == 3:
        # the leading pair ascending, then the lower index of the other pair
        want = np.stack([lead, np.where(lead == 2, 5, 6), np.where(lead == 2, 1, 2)], axis=1)
    else:
        want = np.stack([lead, np.where(lead == 2, 5, 6)], axis=1)
    clear = np.abs(logits[:, 2] - logits[:, 1]) >= 1e-4
    assert clear.sum() >= T * 0.9
    assert np.array_equal(o_idx[clear], want[clear])                  # the oracle follows the rule
    assert np.array_equal(r["idx"][clear], want[clear])               # so does the GPU
    g = r["gate"][clear]
    assert np.array_equal(g[:, 0], g[:, 1])                           # the tied pair's gates
    np.testing.assert_allclose(g, o_gate[clear], rtol=0, atol=1e-5)
    ref = L.forward(li.x_f32)
    assert rel_err(out[clear], ref["out"][clear]) <= (TOL_F32 if dtype == "f32" else TOL_BF16)
    assert layer.device_status() == 0


def test_t0_is_noop_and_max_tokens():
    shape = testgen.LayerShape("edge", 256, 256, 256, 4, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    layer = make_layer(li, max_tokens=256)
    out = torch.full((0, 256), 7.0, device="cuda")
    layer.forward(x_device(li, 0), out)
    _full_check(li, T=256, layer=layer)


def test_forward_host_matches_device_forward():
    shape = testgen.LayerShape("host", 300, 256, 256, 4, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    x = x_device(li)
    dev = layer.forward(x).cpu()
    xh = torch_from_bits(li.x_bits).pin_memory()
    oh = torch.empty((300, 256), dtype=torch.float32).pin_memory()
    layer.forward_host(xh, oh)
    assert torch.equal(dev, oh)


def test_bf16_output_dtype():
    shape = testgen.LayerShape("bf16-out", 400, 256, 256, 4, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    layer = make_layer(li, out_dtype="bf16")
    out, r = run(layer, x_device(li))
    ref = oracle.OracleLayer.from_inputs(li).forward(li.x_f32)["out"]
    rms = math.sqrt(float(np.mean(ref ** 2)))
    # fp32 tolerance plus one bf16 rounding of the result (half an ulp, 2^-8 relative)
    bound = TOL_BF16 * rms + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(out - ref) <= bound)


def test_error_paths():
    from mixture_experts_gemm_gb300 import ColibriError, MoELayer
    shape = testgen.LayerShape("err", 64, 256, 256, 4, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    fresh = MoELayer(256, 256, 4, 64)
    x = x_device(li)
    with pytest.raises(ColibriError) as e:
        fresh.forward(x)
    assert e.value.code == -5   # weights not loaded
    with pytest.raises(ColibriError) as e:
        fresh.get_routing(4)
    assert e.value.code == -5
    layer = make_layer(li)
    big = torch.zeros((65, 256), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ColibriError) as e:
        layer.forward(big)
    assert e.value.code == -1   # T > max_tokens
    with pytest.raises(ColibriError) as e:
        layer.forward(x.cpu())
    assert e.value.code == -1   # host pointer where a device pointer is required
    buf = torch.zeros((64 * 256 * 3,), dtype=torch.bfloat16, device="cuda")
    xa = buf[: 64 * 256].view(64, 256)
    with pytest.raises(ColibriError) as e:
        layer.forward(xa, out=buf[64 * 128: 64 * 128 + 64 * 256 * 2].view(torch.float32).view(64, 256))
    assert e.value.code == -1   # x and out overlap
    with pytest.raises(ColibriError) as e:
        MoELayer(256, 256, 4, 64, act="swiglu").load_weights(li.w_router_bits, [None] * 4, [None] * 4)
    assert e.value.code == -3   # missing expert weights
    with pytest.raises(ColibriError) as e:
        MoELayer(250, 256, 4, 64)
    assert e.value.code == -6   # d not a multiple of 8


def test_pipelined_host_forward_matches_device_forward():
    """forward_host_async: calls overlap their copies with the neighbouring forwards through two
    staging slots; every result must equal the device forward of its own input bit for bit, also
    when a synchronous forward_host call is interleaved."""
    shape = testgen.LayerShape("async", 600, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True)
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    xs = [x_device(li)]
    for sd in (1, 2, 3):
        _, bits = testgen.make_x(shape, seed=sd, want_f32=False)
        xs.append(torch_from_bits(bits).cuda())
    refs = [layer.forward(x).cpu() for x in xs]
    xh = [x.cpu().pin_memory() for x in xs]
    oh = [torch.empty_like(r).pin_memory() for r in refs]
    for rep in range(2):
        for i in range(len(xs)):
            layer.forward_host_async(xh[i], oh[i])
        if rep == 0:
            o_sync = torch.empty_like(refs[0]).pin_memory()
            layer.forward_host(xh[2], o_sync)
            assert torch.equal(o_sync, refs[2])
        layer.host_sync()
        for i in range(len(xs)):
            assert torch.equal(oh[i], refs[i]), (rep, i)
            oh[i].zero_()
    assert layer.device_status() == 0


def test_last_kernel_count_matches_the_path(monkeypatch):
    shape = testgen.LayerShape("count", 300, 512, 384, 8, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    assert layer.last_kernel_count() == 0
    x = x_device(li)
    layer.forward(x)
    assert layer.last_kernel_count() == 2          # router with the dispatch, both weight-major GEMMs + combine
    assert layer.last_gemm() == "weight_major_fused"
    monkeypatch.setenv("COLIBRI_MOE_WM_FUSED", "0")
    layer_s = make_layer(li)
    layer_s.forward(x)
    assert layer_s.last_kernel_count() == 3        # router with the dispatch, up GEMM, down GEMM + combine
    assert layer_s.last_gemm() == "weight_major"
    monkeypatch.delenv("COLIBRI_MOE_WM_FUSED")
    layer.forward(x[:12].contiguous())
    assert layer.last_kernel_count() == 2          # decode: router + one cooperative kernel
    assert layer.last_gemm() == "decode_fused"
    layer.forward(x[:0])
    assert layer.last_kernel_count() == 0
    assert layer.last_gemm() == "none"
    monkeypatch.setenv("COLIBRI_MOE_FUSED_COMBINE", "0")
    monkeypatch.setenv("COLIBRI_MOE_DECODE_FUSED", "0")
    layer2 = make_layer(li)
    layer2.forward(x)
    assert layer2.last_kernel_count() == 3        # router with the dispatch, both GEMMs, combine
    layer2.forward(x[:12].contiguous())
    assert layer2.last_kernel_count() == 6        # router, dispatch, 2 x (GEMM, reduction), combine
    assert layer2.last_gemm() == "decode_split"
    monkeypatch.setenv("COLIBRI_MOE_DISPATCH", "separate")
    layer3 = make_layer(li)
    layer3.forward(x)
    assert layer3.last_kernel_count() == 4        # router, dispatch, both GEMMs, combine
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")
    layer4 = make_layer(li)
    layer4.forward(x)
    assert layer4.last_kernel_count() == 5        # router, dispatch, up GEMM (CTA pairs), down GEMM, combine
    assert layer4.last_gemm() == "pair"
    torch.cuda.synchronize()


def test_two_contexts_on_two_streams_concurrently():
    """Contexts share no device state: two layers (one on the grouped-GEMM path, one on the
    cooperative decode path) forward on two streams at once, several times over without a host
    synchronisation in between, and each output equals its own sequential run bit for bit."""
    la = testgen.make_inputs(testgen.LayerShape("conc-a", 900, 512, 384, 8, testgen.ACT_SWIGLU, "bf16",
                                                zipf_router_bias=True))
    lb = testgen.make_inputs(testgen.LayerShape("conc-b", 12, 512, 768, 16, testgen.ACT_SWIGLU, "bf16",
                                                top_k=4, shared_expert=True))
    layer_a, layer_b = make_layer(la), make_layer(lb)
    xa, xb = x_device(la), x_device(lb)
    ref_a = layer_a.forward(xa).clone()
    ref_b = layer_b.forward(xb).clone()
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs_a = [torch.empty_like(ref_a) for _ in range(4)]
    outs_b = [torch.empty_like(ref_b) for _ in range(4)]
    for i in range(4):
        layer_a.forward(xa, outs_a[i], stream=sa)
        layer_b.forward(xb, outs_b[i], stream=sb)
    torch.cuda.synchronize()
    for i in range(4):
        assert torch.equal(outs_a[i], ref_a), i
        assert torch.equal(outs_b[i], ref_b), i
    assert layer_a.device_status() == 0 and layer_b.device_status() == 0


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    """Failure detection without a fault: the probe runs the kernels' bounded mbarrier wait on a
    barrier nothing arrives on; after its time limit the wait gives up, the status bit is reported
    (and cleared by the read), and the same context then runs a forward that matches the oracle."""
    import time
    import mixture_experts_gemm_gb300 as moe
    li = testgen.make_inputs(testgen.LayerShape("probe", 300, 256, 512, 4, testgen.ACT_SWIGLU, "bf16"))
    layer = make_layer(li)
    assert layer.device_status() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    layer.probe_wait_timeout(20000)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.019 <= waited < 1.0, waited
    assert layer.device_status() == moe.STATUS_WAIT_PROBE
    assert layer.device_status() == 0              # reading clears it
    for bad in (0, -5, 1000001):
        with pytest.raises(RuntimeError):
            layer.probe_wait_timeout(bad)
    _full_check(li, layer=layer)                   # device_status() == 0 asserted inside


def test_stage_events_time_every_stage():
    shape = testgen.LayerShape("events", 512, 512, 512, 8, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    layer = make_layer(li)
    n = layer.num_stages()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    layer.set_stage_events(ev)
    layer.forward(x_device(li))
    torch.cuda.synchronize()
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
    assert all(t > 0 for t in times)
    layer.set_stage_events(None)
