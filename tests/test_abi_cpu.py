"""The C-ABI library without a GPU: it builds for sm_103a, loads, exports every function the header
declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "colibri_moe.h")


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"COLIBRI_API\s+[\w\s\*]+?\b(colibri_moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("colibri_moe_create", "colibri_moe_load_weights", "colibri_moe_forward",
                     "colibri_moe_destroy", "colibri_moe_get_routing", "colibri_moe_strerror"):
        assert required in names


def test_library_exports_every_declared_symbol(cuda_lib):
    import mixture_experts_gemm_gb300 as m
    names = declared_functions()
    assert set(names) == set(m.EXPORTED)
    raw = ctypes.CDLL(m.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_strerror_covers_every_code(cuda_lib):
    import mixture_experts_gemm_gb300 as m
    codes = [int(v) for v in re.findall(r"#define COLIBRI_(?:OK|ERR_\w+)\s+\(?(-?\d+)\)?", open(HEADER).read())]
    assert sorted(codes) == [-7, -6, -5, -4, -3, -2, -1, 0]
    texts = {m.strerror(c) for c in codes}
    assert len(texts) == len(codes) and "unknown status code" not in texts
    assert m.strerror(12345) == "unknown status code"


def _cfg(m, **kw):
    base = dict(d_model=256, d_ff=256, num_experts=4, top_k=2, max_tokens=64, dtype=1, act=1,
                has_router_bias=0, out_dtype=0)
    base.update(kw)
    return m.Config(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(top_k=0), -1), (dict(top_k=5), -1), (dict(num_experts=2, top_k=3), -1), (dict(gate_mode=2), -1),
    (dict(has_shared_expert=2), -1), (dict(num_experts=1), -1), (dict(num_experts=17), -1), (dict(max_tokens=0), -1),
    (dict(d_model=0), -1), (dict(dtype=5), -1), (dict(act=9), -1), (dict(out_dtype=3), -1),
    (dict(has_router_bias=2), -1), (dict(d_model=260), -6), (dict(d_ff=200), -6),
    (dict(act=0, d_ff=384), -6), (dict(dtype=0, d_model=12), -6),
])
def test_create_rejects_bad_configs_without_a_device(cuda_lib, kw, code):
    import mixture_experts_gemm_gb300 as m
    h = ctypes.c_void_p(1234)
    rc = m.lib().colibri_moe_create(ctypes.byref(_cfg(m, **kw)), 0, ctypes.byref(h))
    assert rc == code and h.value is None


def test_null_arguments(cuda_lib):
    import mixture_experts_gemm_gb300 as m
    L = m.lib()
    assert L.colibri_moe_create(None, 0, None) == -1
    assert L.colibri_moe_forward(None, None, None, 4, None) == -1
    assert L.colibri_moe_forward_host(None, None, None, 4, None) == -1
    assert L.colibri_moe_forward_host_async(None, None, None, 4, None) == -1
    assert L.colibri_moe_host_sync(None) == -1
    assert L.colibri_moe_load_weights(None, None, None) == -1
    assert L.colibri_moe_get_routing(None, None, None, None, None, None, None) == -1
    assert L.colibri_moe_set_stage_events(None, None, 0) == -1
    n = ctypes.c_int32()
    assert L.colibri_moe_num_stages(None, ctypes.byref(n)) == -1
    assert L.colibri_moe_last_kernel_count(None, ctypes.byref(n)) == -1
    assert L.colibri_moe_last_gemm(None, ctypes.byref(n)) == -1
    assert L.colibri_moe_probe_wait_timeout(None, 1000, None) == -1
    assert L.colibri_moe_ep_dispatch(None, None, 4, None, None, None) == -1
    assert L.colibri_moe_ep_experts(None, None, None, None, None) == -1
    assert L.colibri_moe_ep_combine(None, None, None, None) == -1
    L.colibri_moe_destroy(None)  # NULL-safe


@pytest.mark.parametrize("ep_rank,ep_size,max_rows,kw,code", [
    (0, 0, 64, {}, -1),                       # no ranks
    (0, 3, 64, {}, -1),                       # 4 experts do not split over 3 ranks
    (2, 2, 64, {}, -1),                       # rank out of range
    (0, 2, 0, {}, -1),                        # no receive rows
    (0, 2, 64, {"has_shared_expert": 1}, -6),  # a shared expert would run replicated on every rank
])
def test_ep_create_rejects_bad_partitions_without_a_device(cuda_lib, ep_rank, ep_size, max_rows, kw, code):
    """Expert-parallel contexts check the partition before touching the GPU."""
    import mixture_experts_gemm_gb300 as m
    h = ctypes.c_void_p()
    rc = m.lib().colibri_moe_ep_create(ctypes.byref(_cfg(m, **kw)), ep_rank, ep_size, max_rows, 0, ctypes.byref(h))
    assert rc == code and h.value is None


def test_create_without_gpu_reports_cuda_error(cuda_lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import mixture_experts_gemm_gb300 as m
    h = ctypes.c_void_p()
    assert m.lib().colibri_moe_create(ctypes.byref(_cfg(m)), 0, ctypes.byref(h)) == -4


def test_product_has_no_cpu_fallback():
    """The package never imports the oracle or the input generator: it runs the CUDA library or fails."""
    pkg = os.path.join(ROOT, "mixture_experts_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.lower().replace("oracle.", ""), f
                assert "testgen" not in src, f


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    import mixture_experts_gemm_gb300 as m
    monkeypatch.setattr(m, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(ImportError):
        m.lib()
