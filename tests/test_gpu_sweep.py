"""GPU parity on a seeded sweep of layer shapes, each against the fp64 CPU oracle.

Every case draws, from its own seed: dtype (fp32 SIMT or bf16 tensor-core path), activation, model
and hidden widths within what the path supports, the number of experts (2..16), top-k (1..4),
gate mode, an optional shared expert, a Zipf-like router bias, the output dtype and the token count
(decode-sized batches through the cooperative kernel, larger ones through the grouped GEMMs, with
ragged tails).  The checks are those of the fixed cases: routing bit for bit outside near ties,
output within the dtype's tolerance (a bf16 output also gets half an ulp of its own rounding per
element), a clean device status word, and a repeat forward equal bit for bit (determinism).
"""
import numpy as np
import pytest

import testgen
from moe_check import TOL_BF16, TOL_F32, bf16_h_bound, check_routing, make_layer, rel_err, run, x_device

import oracle

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

N_CASES = 64
FLOP_BUDGET = 4e9  # oracle work per case (fp64 multiply-adds x 2), so the sweep runs in about a minute


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def draw_case(i: int):
    rng = np.random.default_rng(1000 + i)
    bf16 = bool(rng.integers(0, 4))  # three in four cases on the tensor-core path
    act = int(rng.integers(0, 2))
    if bf16:
        d = int(rng.choice([256, 512]))
        f = int(rng.choice([128, 256, 384, 512, 640])) if act == testgen.ACT_SWIGLU else int(rng.choice([256, 512]))
    else:
        d = int(rng.choice([64, 136, 256]))
        f = int(rng.choice([64, 200, 512]))
    E = int(rng.integers(2, 17))
    k = int(rng.integers(1, min(4, E) + 1))
    shared = bool(rng.integers(0, 2)) and E < 17
    mode = int(rng.integers(0, 2))
    zipf = bool(rng.integers(0, 2))
    T = int(rng.choice([1, 3, 17, 40, 64, 65, 200, 513, 777, 1500]))
    n_mats = 3 if act == testgen.ACT_SWIGLU else 2
    while T > 1 and 2.0 * T * (k + shared) * n_mats * d * f > FLOP_BUDGET:
        T //= 2
    out_dtype = "bf16" if bf16 and rng.integers(0, 4) == 0 else "f32"
    name = f"sweep{i}-{'bf16' if bf16 else 'f32'}-{'swiglu' if act else 'relu'}-d{d}-f{f}-E{E}-k{k}" \
           f"{'-s' if shared else ''}-m{mode}{'-z' if zipf else ''}-T{T}-{out_dtype}"
    shape = testgen.LayerShape(name, T, d, f, E, act, "bf16" if bf16 else "f32", zipf_router_bias=zipf, top_k=k,
                               gate_mode=mode, shared_expert=shared)
    return shape, out_dtype


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_layer_shape(i):
    shape, out_dtype = draw_case(i)
    li = testgen.make_inputs(shape)
    layer = make_layer(li, out_dtype=out_dtype)
    x = x_device(li)
    out, r = run(layer, x)
    L = oracle.OracleLayer.from_inputs(li)
    ref = L.forward(li.x_f32)
    check_routing(r, ref["logits"], ref["idx"], ref["gate"], shape.num_experts, ref["row_of"], ref["offsets_raw"],
                  gate_mode=shape.gate_mode)
    tol = TOL_F32 if shape.dtype == "f32" else TOL_BF16
    if out_dtype == "bf16":
        # the layer's tolerance plus the one rounding of the result to bf16 (half an ulp: 2^-8 relative)
        ref_out = ref["out"]
        rms = float(np.sqrt(np.mean(ref_out ** 2)))
        excess = np.abs(out - ref_out) - (tol * rms + np.abs(ref_out) * 2.0 ** -8)
        assert np.all(excess <= 0), f"{shape.name}: bf16 output off by {excess.max():.3e} beyond its bound"
    else:
        err = rel_err(out, ref["out"])
        assert err <= tol, f"{shape.name}: max|err|/RMS = {err:.3e} > {tol}"
    assert layer.device_status() == 0, shape.name
    out2, _ = run(layer, x)
    assert np.array_equal(out, out2), shape.name


N_WM_CASES = 40


def draw_wm_case(i: int):
    """A bf16 layer for the weight-major GEMM: widths with 256-row weight tiles, 2..16 experts, top-1..4,
    gate mode, shared expert, Zipf bias, and a token count from 1 to ~3000 (ragged token tiles)."""
    rng = np.random.default_rng(5000 + i)
    act = int(rng.integers(0, 2))
    d = int(rng.choice([256, 512, 768]))
    f = int(rng.choice([128, 256, 384, 640])) if act == testgen.ACT_SWIGLU else int(rng.choice([256, 512, 768]))
    E = int(rng.integers(2, 17))
    k = int(rng.integers(1, min(4, E) + 1))
    shared = bool(rng.integers(0, 2))
    mode = int(rng.integers(0, 2))
    zipf = bool(rng.integers(0, 2))
    T = int(rng.choice([1, 5, 31, 33, 97, 200, 450, 1000, 3000]))
    n_mats = 3 if act == testgen.ACT_SWIGLU else 2
    while T > 1 and 2.0 * T * (k + shared) * n_mats * d * f > FLOP_BUDGET:
        T //= 2
    nt = str(int(rng.choice([0, 32, 64, 96, 160, 256])))  # 0: the default token tile for the batch
    out_dtype = "bf16" if rng.integers(0, 4) == 0 else "f32"
    fused = bool(rng.integers(0, 4))  # one in four cases as two launches
    name = f"wm{i}-{'swiglu' if act else 'relu'}-d{d}-f{f}-E{E}-k{k}{'-s' if shared else ''}-m{mode}" \
           f"{'-z' if zipf else ''}-T{T}-nt{nt}-{out_dtype}{'' if fused else '-2launch'}"
    shape = testgen.LayerShape(name, T, d, f, E, act, "bf16", zipf_router_bias=zipf, top_k=k, gate_mode=mode,
                               shared_expert=shared)
    return shape, out_dtype, nt, fused


@pytest.mark.parametrize("i", range(N_WM_CASES))
def test_random_weight_major_layer(i, monkeypatch):
    """The weight-major GEMM on random shapes, decode path off: against the oracle (routing bit for bit
    outside near ties, output within tolerance) and bit for bit against the CTA-pair kernel on the same
    inputs (H, out), in its fused form or as two launches."""
    shape, out_dtype, nt, fused = draw_wm_case(i)
    monkeypatch.setenv("COLIBRI_MOE_DECODE_MAX_T", "0")
    if nt != "0":
        monkeypatch.setenv("COLIBRI_MOE_WM", nt)
    if not fused:
        monkeypatch.setenv("COLIBRI_MOE_WM_FUSED", "0")
    li = testgen.make_inputs(shape)
    layer = make_layer(li, out_dtype=out_dtype)
    x = x_device(li)
    out, r = run(layer, x)
    form = layer.last_gemm()
    L = oracle.OracleLayer.from_inputs(li)
    ref = L.forward(li.x_f32)
    n_tie = check_routing(r, ref["logits"], ref["idx"], ref["gate"], shape.num_experts, ref["row_of"],
                          ref["offsets_raw"], gate_mode=shape.gate_mode)
    keep = ~oracle.near_tie_tokens(ref["logits"], k=shape.top_k) if n_tie else np.ones(shape.T, dtype=bool)
    ref_out = ref["out"][keep]
    rms = float(np.sqrt(np.mean(ref_out ** 2)))
    # the bf16 tolerance, plus what the one bf16 rounding of H can add to an element (this only
    # matters for output outliers), plus half an ulp of a bf16 output's own rounding
    h_bound = bf16_h_bound(li, ref["idx"], ref["gate"])[keep]
    half_ulp_out = np.abs(ref_out) * 2.0 ** -8 if out_dtype == "bf16" else 0.0
    excess = np.abs(out[keep] - ref_out) - (TOL_BF16 * rms + h_bound + half_ulp_out)
    assert np.all(excess <= 0), f"{shape.name}: beyond its bound by {excess.max() / rms:.3e} x RMS"
    assert layer.device_status() == 0, shape.name
    monkeypatch.setenv("COLIBRI_MOE_WM", "0")
    layer_p = make_layer(li, out_dtype=out_dtype)
    out_p, r_p = run(layer_p, x)
    assert layer_p.last_gemm() == "pair", shape.name
    assert np.array_equal(out, out_p), (shape.name, form)
    rows = np.sort(r["row_of"].ravel())
    if shape.shared_expert:
        off = r["offsets"]
        rows = np.concatenate([rows, np.arange(off[-1], off[-1] + shape.T)])
    idx_rows = torch.from_numpy(rows.astype(np.int64)).cuda()
    assert torch.equal(layer.debug_tensor(1)[idx_rows], layer_p.debug_tensor(1)[idx_rows]), (shape.name, form)
    out2, _ = run(layer, x)
    assert np.array_equal(out, out2), shape.name
