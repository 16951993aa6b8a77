"""colibri_moe_route_noalloc: routing for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a host framework's memory pool owns the GPU, a real-time loop
cannot take cudaMalloc's implicit synchronisation, or the device-memory budget is fixed at
start-up).  This entry point keeps its scratch in a fixed array inside the library instead; its
results must equal the oracle's routing and the routing the context-based forward reports, call
after call, from a single token up to the largest batch the fixed array holds.
"""
import ctypes

import numpy as np
import pytest

import oracle
import testgen
from moe_check import NEAR_TIE, check_routing, make_layer, torch_from_bits, x_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _route_noalloc(lib, x, wr, br, T, shape, dtype_code, stream):
    dev = x.device
    E = shape.num_experts
    out = dict(idx=torch.full((T, 2), -7, dtype=torch.int32, device=dev),
               gate=torch.full((T, 2), -7.0, dtype=torch.float32, device=dev),
               counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
               offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
               row_of=torch.full((T, 2), -7, dtype=torch.int32, device=dev))
    rc = lib.colibri_moe_route_noalloc(x.data_ptr(), wr.data_ptr(), None if br is None else br.data_ptr(), T,
                                       shape.d_model, E, dtype_code, out["idx"].data_ptr(), out["gate"].data_ptr(),
                                       out["counts"].data_ptr(), out["offsets"].data_ptr(), out["row_of"].data_ptr(),
                                       stream)
    return rc, out


_CASES = [
    # forward routes these 1000 tokens with the split router, route_noalloc with the plain one
    testgen.LayerShape("noalloc-bf16", 1000, 512, 256, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
    testgen.LayerShape("noalloc-f32", 77, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32"),
    # one 32-token chunk (its summary written by the chunk itself) and a single token
    testgen.LayerShape("noalloc-one-chunk-e16", 32, 256, 256, 16, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
    testgen.LayerShape("noalloc-t1", 1, 256, 256, 8, testgen.ACT_SWIGLU, "bf16"),
    # the largest batch: every histogram row of the fixed scratch array in use
    testgen.LayerShape("noalloc-max-t", 65536, 256, 256, 16, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
]


@pytest.mark.parametrize("shape", _CASES, ids=[c.name for c in _CASES])
def test_route_noalloc_matches_oracle_and_forward_routing(cuda_lib, shape):
    """Two calls in a row: each equals the oracle's routing (bit for bit outside near ties, gates
    within 1e-5) and the routing the context-based forward reports; the second equals the first."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_gemm_gb300 as moe
    lib = moe.lib()
    li = testgen.make_inputs(shape)
    T, E = shape.T, shape.num_experts
    L = oracle.OracleLayer.from_inputs(li)
    logits = L.router_logits(li.x_f32)
    o_idx, o_gate = L.topk(logits)
    _, o_offs, o_row_of, _ = L.dispatch(o_idx)
    tie = oracle.near_tie_tokens(logits, NEAR_TIE)

    layer = make_layer(li)
    x = x_device(li)
    layer.forward(x)
    ref = {k: v.cpu().numpy() for k, v in layer.get_routing(T).items()}
    torch.cuda.synchronize()
    layer.close()

    bf = shape.dtype == "bf16"
    wr = (torch_from_bits(li.w_router_bits) if bf else torch.from_numpy(li.w_router_f32)).cuda()
    br = None if li.b_router is None else torch.from_numpy(li.b_router).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    first = None
    for call in range(2):
        rc, got = _route_noalloc(lib, x, wr, br, T, shape, 1 if bf else 0, stream)
        assert rc == 0, moe.strerror(rc)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in got.items()}
        check_routing(got, logits, o_idx, o_gate, E, o_row_of, o_offs)
        # the existing entry point's routing: the same decisions wherever rounding cannot flip one
        assert np.array_equal(got["idx"][~tie], ref["idx"][~tie]), call
        np.testing.assert_allclose(got["gate"], ref["gate"], rtol=0, atol=1e-5)
        if not tie.any():
            for k in ("idx", "counts", "offsets", "row_of"):
                assert np.array_equal(got[k], ref[k]), (call, k)
        if first is None:
            first = got
        else:
            for k in got:
                assert np.array_equal(got[k], first[k]), k


def test_route_noalloc_rejects_oversize_batches(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mixture_experts_gemm_gb300 as moe
    lib = moe.lib()
    d, E, T = 256, 4, 65537
    x = torch.zeros((T, d), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((E, d), dtype=torch.bfloat16, device="cuda")
    shape = testgen.LayerShape("noalloc-big", T, d, 256, E, testgen.ACT_SWIGLU, "bf16")
    rc, _ = _route_noalloc(lib, x, wr, None, T, shape, 1, torch.cuda.current_stream().cuda_stream)
    assert rc == -1
