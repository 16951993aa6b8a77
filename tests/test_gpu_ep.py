"""Expert parallelism through the C ABI on one GPU: ep_size ranks emulated in one process (each rank a
context holding its own experts; the all-to-alls done as copies between the ranks' buffers), so the
kernels of ep_dispatch / ep_experts / ep_combine run exactly as on separate GPUs.

Every rank's output must equal the ordinary forward of its batch on a context holding all experts,
bit for bit where that forward runs the grouped GEMMs (the expert ranks always do), and the oracle
within the layer's tolerance everywhere."""
import ctypes

import numpy as np
import pytest

import oracle
import testgen
from moe_check import TOL_BF16, TOL_F32, check_routing, host_weights, make_layer, rel_err, torch_from_bits

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_lib):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    torch.cuda.synchronize()


def _ep_layers(li, n, max_tokens, max_recv_rows=None):
    from mixture_experts_gemm_gb300 import MoELayer
    s = li.shape
    w = host_weights(li)
    layers = []
    for r in range(n):
        L = MoELayer(s.d_model, s.d_ff, s.num_experts, max_tokens, dtype=s.dtype,
                     act="swiglu" if s.act == testgen.ACT_SWIGLU else "relu_bias",
                     has_router_bias=li.b_router is not None, out_dtype="f32", top_k=s.top_k, gate_mode=s.gate_mode,
                     ep_rank=r, ep_size=n, max_recv_rows=max_recv_rows)
        # only this rank's experts are read: pass None for the others
        El = s.num_experts // n
        own = lambda lst: None if lst is None else [t if r * El <= e < (r + 1) * El else None
                                                    for e, t in enumerate(lst)]
        L.load_weights(w["w_router"], own(w["w1"]), own(w["w2"]), w3=own(w["w3"]), b_router=w["b_router"],
                       b1=own(w["b1"]), b2=own(w["b2"]))
        layers.append(L)
    return layers


def _xs(li, sizes):
    bf = li.shape.dtype == "bf16"
    full = torch_from_bits(li.x_bits) if bf else torch.from_numpy(li.x_f32)
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    return [full[a:a + n].contiguous().cuda() for a, n in zip(starts, sizes)], starts


CASES = {
    # name: (shape over all ranks' tokens, per-rank batch sizes)
    "bf16-swiglu-2": (testgen.LayerShape("ep2", 1000, 512, 384, 8, testgen.ACT_SWIGLU, "bf16", zipf_router_bias=True),
                      [300, 700]),
    "bf16-swiglu-4-empty-rank": (testgen.LayerShape("ep4", 1166, 512, 384, 8, testgen.ACT_SWIGLU, "bf16",
                                                    zipf_router_bias=True), [1000, 0, 37, 129]),
    "bf16-relu-1": (testgen.LayerShape("ep1", 500, 256, 512, 4, testgen.ACT_RELU_BIAS, "bf16"), [500]),
    "f32-relu-2": (testgen.LayerShape("ep-f32", 128, 256, 512, 4, testgen.ACT_RELU_BIAS, "f32"), [64, 64]),
    "bf16-top4-full-softmax-2": (testgen.LayerShape("ep-k4", 600, 512, 256, 8, testgen.ACT_SWIGLU, "bf16",
                                                    zipf_router_bias=True, top_k=4, gate_mode=1), [250, 350]),
    "bf16-16-experts-8-ranks": (testgen.LayerShape("ep8", 1600, 256, 256, 16, testgen.ACT_SWIGLU, "bf16",
                                                   zipf_router_bias=True), [200] * 8),
}


@pytest.mark.parametrize("case", list(CASES))
def test_expert_parallel_step_equals_forward_and_oracle(case):
    from mixture_experts_gemm_gb300 import ep
    shape, sizes = CASES[case]
    n = len(sizes)
    li = testgen.make_inputs(shape)
    xs, starts = _xs(li, sizes)
    layers = _ep_layers(li, n, max(max(sizes), 1))
    outs = ep.ep_forward_local([ep.LayerEP(L) for L in layers], xs)
    torch.cuda.synchronize()
    full = make_layer(li, max_tokens=max(max(sizes), 1))
    L = oracle.OracleLayer.from_inputs(li)
    tol = TOL_F32 if shape.dtype == "f32" else TOL_BF16
    for r, (x, out) in enumerate(zip(xs, outs)):
        T = sizes[r]
        assert out.shape == (T, shape.d_model)
        if T == 0:
            continue
        got = out.cpu().numpy().astype(np.float64)
        ref_fwd = full.forward(x)
        torch.cuda.synchronize()
        grouped = full.last_gemm() not in ("decode_fused", "decode_split")   # the decode path sums in another order
        if grouped:
            assert np.array_equal(got, ref_fwd.cpu().numpy().astype(np.float64)), (case, r)
            if shape.dtype == "bf16":   # the ranks' GEMMs: weight-major or CTA pairs, the same result
                assert layers[r].last_gemm() in ("weight_major_fused", "weight_major", "pair"), layers[r].last_gemm()
        a = int(starts[r])
        ref = L.forward(li.x_f32[a:a + T])
        assert rel_err(got, ref["out"]) <= tol, (case, r)
        # the routing the dispatch kept: the oracle's (outside near ties); row_of = rows of send_rows
        g = {k: v.cpu().numpy() for k, v in layers[r].get_routing(T).items()}
        torch.cuda.synchronize()
        check_routing(dict(g, offsets=_padded(g["counts"]), row_of=_as_padded(g, shape.num_experts)), ref["logits"],
                      ref["idx"], ref["gate"], shape.num_experts, ref["row_of"], ref["offsets_raw"],
                      gate_mode=shape.gate_mode)
    for Lr in layers:
        assert Lr.device_status() == 0
        Lr.close()
    full.close()


def _padded(counts):
    pad = (counts + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(pad)]).astype(np.int32)


def _as_padded(g, E):
    """get_routing's row_of on an expert-parallel context is the row of send_rows (unpadded, experts
    in order): the same rank inside the expert, moved onto 128-row padded segments for the check."""
    counts = g["counts"].astype(np.int64)
    raw = np.concatenate([[0], np.cumsum(counts)])
    return (g["row_of"] - raw[g["idx"]] + _padded(g["counts"])[g["idx"]]).astype(np.int32)


def test_expert_parallel_mixtral_shape_two_ranks_equals_forward():
    """The benchmark's Mixtral-shaped layer split over two ranks of 4096 tokens each (4 experts per
    rank): each rank's output equals the single-context forward of its batch bit for bit."""
    from mixture_experts_gemm_gb300 import ep
    s = testgen.CONFIGS["mixtral-prefill"]
    li = testgen.make_inputs(s)
    sizes = [4096, 4096]
    xs, _ = _xs(li, sizes)
    layers = _ep_layers(li, 2, 4096)
    outs = ep.ep_forward_local([ep.LayerEP(L) for L in layers], xs)
    torch.cuda.synchronize()
    for L in layers:
        assert L.device_status() == 0
        L.close()
    full = make_layer(li, max_tokens=4096)
    for x, out in zip(xs, outs):
        ref = full.forward(x)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    full.close()


def test_expert_parallel_error_paths():
    import mixture_experts_gemm_gb300 as moe
    lib = moe.lib()
    cfg = moe.Config(256, 256, 8, 2, 64, moe.DTYPE_BF16, moe.ACT_SWIGLU, 0, moe.DTYPE_F32, 0, 0)
    h = ctypes.c_void_p()
    assert lib.colibri_moe_ep_create(ctypes.byref(cfg), 0, 3, 128, 0, ctypes.byref(h)) == -1   # 8 % 3
    assert lib.colibri_moe_ep_create(ctypes.byref(cfg), 2, 2, 128, 0, ctypes.byref(h)) == -1   # rank >= size
    assert lib.colibri_moe_ep_create(ctypes.byref(cfg), 0, 0, 128, 0, ctypes.byref(h)) == -1
    assert lib.colibri_moe_ep_create(ctypes.byref(cfg), 0, 2, 0, 0, ctypes.byref(h)) == -1     # no rows
    cfg_sh = moe.Config(256, 256, 8, 2, 64, moe.DTYPE_BF16, moe.ACT_SWIGLU, 0, moe.DTYPE_F32, 0, 1)
    assert lib.colibri_moe_ep_create(ctypes.byref(cfg_sh), 0, 2, 128, 0, ctypes.byref(h)) == -6  # shared expert
    shape = testgen.LayerShape("ep-err", 64, 256, 256, 8, testgen.ACT_SWIGLU, "bf16")
    li = testgen.make_inputs(shape)
    L = _ep_layers(li, 2, 64, max_recv_rows=100)[0]
    x = torch_from_bits(li.x_bits).cuda()
    out = torch.empty((64, 256), dtype=torch.float32, device="cuda")
    assert lib.colibri_moe_forward(L.handle, x.data_ptr(), out.data_ptr(), 64, None) == -6
    assert lib.colibri_moe_ep_combine(L.handle, out.data_ptr(), out.data_ptr(), None) == -5   # before dispatch
    rows = torch.empty((101, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((101, 256), dtype=torch.float32, device="cuda")
    too_many = np.array([[51, 0, 0, 0], [50, 0, 0, 0]], dtype=np.int32)
    assert lib.colibri_moe_ep_experts(L.handle, rows.data_ptr(), too_many.ctypes.data, y.data_ptr(), None) == -1
    neg = np.array([[1, -1, 0, 0], [0, 0, 0, 0]], dtype=np.int32)
    assert lib.colibri_moe_ep_experts(L.handle, rows.data_ptr(), neg.ctypes.data, y.data_ptr(), None) == -1
    host = np.zeros((64, 256), dtype=np.float32)
    sc = torch.empty(8, dtype=torch.int32, device="cuda")
    assert lib.colibri_moe_ep_dispatch(L.handle, host.ctypes.data, 64, rows.data_ptr(), sc.data_ptr(), None) == -1
    # an ordinary context refuses the expert-parallel calls
    full = make_layer(li)
    assert lib.colibri_moe_ep_dispatch(full.handle, x.data_ptr(), 64, rows.data_ptr(), sc.data_ptr(), None) == -6
    full.close()
    L.close()
