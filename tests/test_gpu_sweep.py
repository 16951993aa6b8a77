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
from moe_check import TOL_BF16, TOL_F32, check_routing, make_layer, rel_err, run, x_device

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
