"""GB300 (sm_103a) Mixture-of-Experts layer forward: Python binding of the C ABI.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
``libcolibri_moe.so`` (built in-tree by ``_build.py``).  There is no fallback:
if the library is missing or cannot run, calls raise.

    layer = MoELayer(d_model=4096, d_ff=14336, num_experts=8, max_tokens=8192)
    layer.load_weights(w_router, w1, w2, w3=w3)         # torch tensors or numpy arrays
    out = layer.forward(x)                              # x: [T, d] CUDA tensor

The C functions keep their names (``colibri_moe_*``); ``lib()`` returns the
loaded ``ctypes.CDLL`` for direct calls.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from ._build import LIB as LIB_PATH

__all__ = ["MoELayer", "ColibriError", "lib", "LIB_PATH", "DTYPE_F32", "DTYPE_BF16", "ACT_RELU_BIAS", "ACT_SWIGLU",
           "EXPORTED"]

DTYPE_F32, DTYPE_BF16 = 0, 1
ACT_RELU_BIAS, ACT_SWIGLU = 0, 1
STATUS_WAIT_PROBE = 1 << 6  # set by probe_wait_timeout when its bounded wait gives up
GATE_SOFTMAX_SELECTED, GATE_SOFTMAX_ALL = 0, 1
_GATES = {"selected": GATE_SOFTMAX_SELECTED, "pair": GATE_SOFTMAX_SELECTED, "all": GATE_SOFTMAX_ALL,
          "full": GATE_SOFTMAX_ALL}
_DTYPES = {"f32": DTYPE_F32, "fp32": DTYPE_F32, "float32": DTYPE_F32, "bf16": DTYPE_BF16, "bfloat16": DTYPE_BF16}
_ACTS = {"relu_bias": ACT_RELU_BIAS, "relu": ACT_RELU_BIAS, "swiglu": ACT_SWIGLU}

# every function include/colibri_moe.h declares
EXPORTED = ("colibri_moe_create", "colibri_moe_load_weights", "colibri_moe_forward", "colibri_moe_forward_host",
            "colibri_moe_get_routing", "colibri_moe_debug_buffer", "colibri_moe_num_stages",
            "colibri_moe_forward_host_async", "colibri_moe_host_sync",
            "colibri_moe_last_kernel_count", "colibri_moe_last_gemm", "colibri_moe_set_stage_events", "colibri_moe_device_status",
            "colibri_moe_probe_wait_timeout", "colibri_moe_route_noalloc",
            "colibri_moe_ep_create", "colibri_moe_ep_dispatch", "colibri_moe_ep_experts", "colibri_moe_ep_combine",
            "colibri_moe_destroy", "colibri_moe_strerror")


class ColibriError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {strerror(code)} ({code})")


class Config(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("max_tokens", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("act", ctypes.c_int32), ("has_router_bias", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
                ("gate_mode", ctypes.c_int32), ("has_shared_expert", ctypes.c_int32)]


class Weights(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("b_router", ctypes.c_void_p), ("w1", ctypes.c_void_p),
                ("w3", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("ws1", ctypes.c_void_p), ("ws3", ctypes.c_void_p),
                ("ws2", ctypes.c_void_p), ("bs1", ctypes.c_void_p), ("bs2", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                              f"g.build()'` (nvcc, sm_103a)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        sig = {
            "colibri_moe_create": ([ctypes.POINTER(Config), ctypes.c_int, ctypes.POINTER(vp)], ctypes.c_int),
            "colibri_moe_load_weights": ([vp, ctypes.POINTER(Weights), vp], ctypes.c_int),
            "colibri_moe_forward": ([vp, vp, vp, i32, vp], ctypes.c_int),
            "colibri_moe_forward_host": ([vp, vp, vp, i32, vp], ctypes.c_int),
            "colibri_moe_forward_host_async": ([vp, vp, vp, i32, vp], ctypes.c_int),
            "colibri_moe_host_sync": ([vp], ctypes.c_int),
            "colibri_moe_get_routing": ([vp, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "colibri_moe_debug_buffer": ([vp, i32, ctypes.POINTER(vp), ctypes.POINTER(i64)], ctypes.c_int),
            "colibri_moe_num_stages": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
            "colibri_moe_last_kernel_count": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
            "colibri_moe_last_gemm": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
            "colibri_moe_set_stage_events": ([vp, vp, i32], ctypes.c_int),
            "colibri_moe_device_status": ([vp, ctypes.POINTER(i32)], ctypes.c_int),
            "colibri_moe_probe_wait_timeout": ([vp, i32, vp], ctypes.c_int),
            "colibri_moe_route_noalloc": ([vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp], ctypes.c_int),
            "colibri_moe_ep_create": ([ctypes.POINTER(Config), i32, i32, i32, ctypes.c_int, ctypes.POINTER(vp)],
                                      ctypes.c_int),
            "colibri_moe_ep_dispatch": ([vp, vp, i32, vp, vp, vp], ctypes.c_int),
            "colibri_moe_ep_experts": ([vp, vp, vp, vp, vp], ctypes.c_int),
            "colibri_moe_ep_combine": ([vp, vp, vp, vp], ctypes.c_int),
            "colibri_moe_destroy": ([vp], None),
            "colibri_moe_strerror": ([ctypes.c_int], ctypes.c_char_p),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def strerror(code: int) -> str:
    try:
        return lib().colibri_moe_strerror(code).decode()
    except ImportError:
        return "library not loaded"


def _check(rc: int, what: str):
    if rc != 0:
        raise ColibriError(rc, what)


def _ptr(a) -> Optional[int]:
    """Address of a contiguous torch tensor or numpy array (host or device); None passes NULL."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return a.data_ptr()
    if hasattr(a, "ctypes"):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return a.ctypes.data
    raise TypeError(f"cannot take the address of {type(a)}")


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class MoELayer:
    """One MoE layer instance (a ``colibri_moe_t`` context) on one GPU.

    With ``ep_size`` > 0 the context is rank ``ep_rank`` of an expert-parallel layer (the experts
    split over ep_size GPUs): it holds experts [ep_rank*El, (ep_rank+1)*El) and runs ep_dispatch /
    ep_experts / ep_combine (see ``ep.py`` for the exchange between them) instead of forward."""

    def __init__(self, d_model: int, d_ff: int, num_experts: int, max_tokens: int, dtype="bf16", act="swiglu",
                 has_router_bias: bool = False, out_dtype="f32", device: int = 0, top_k: int = 2,
                 gate_mode="selected", shared_expert: bool = False, ep_rank: int = 0, ep_size: int = 0,
                 max_recv_rows: Optional[int] = None):
        self.cfg = Config(d_model, d_ff, num_experts, top_k, max_tokens,
                          _DTYPES[dtype] if isinstance(dtype, str) else int(dtype),
                          _ACTS[act] if isinstance(act, str) else int(act), int(bool(has_router_bias)),
                          _DTYPES[out_dtype] if isinstance(out_dtype, str) else int(out_dtype),
                          _GATES[gate_mode] if isinstance(gate_mode, str) else int(gate_mode), int(bool(shared_expert)))
        self.device = device
        self.ep_rank, self.ep_size = int(ep_rank), int(ep_size)
        self._ep_T = None
        self._h = ctypes.c_void_p()
        if self.ep_size > 0:
            if max_recv_rows is None:
                max_recv_rows = self.ep_size * max_tokens * top_k
            self.max_recv_rows = int(max_recv_rows)
            _check(lib().colibri_moe_ep_create(ctypes.byref(self.cfg), self.ep_rank, self.ep_size, self.max_recv_rows,
                                               device, ctypes.byref(self._h)), "colibri_moe_ep_create")
        else:
            _check(lib().colibri_moe_create(ctypes.byref(self.cfg), device, ctypes.byref(self._h)),
                   "colibri_moe_create")
        self._keep = []

    # -------------------------------------------------------------- properties
    @property
    def handle(self) -> int:
        return self._h.value

    @property
    def d_model(self) -> int:
        return self.cfg.d_model

    @property
    def num_experts(self) -> int:
        return self.cfg.num_experts

    def close(self):
        if self._h and self._h.value:
            lib().colibri_moe_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -------------------------------------------------------------- calls
    def load_weights(self, w_router, w1: Sequence, w2: Sequence, w3: Optional[Sequence] = None, b_router=None,
                     b1: Optional[Sequence] = None, b2: Optional[Sequence] = None, shared: Optional[dict] = None,
                     stream=None):
        """Copy weights (host or device, dtype per config; biases fp32) into the device arena.
        shared: the shared expert's tensors, dict(w1=..., w3=..., w2=..., b1=..., b2=...)."""
        E = self.cfg.num_experts

        def parr(lst):
            if lst is None:
                return None
            if len(lst) != E:
                raise ValueError(f"expected {E} per-expert tensors, got {len(lst)}")
            arr = (ctypes.c_void_p * E)(*[_ptr(t) for t in lst])
            self._keep.append(arr)
            return ctypes.cast(arr, ctypes.c_void_p).value

        sh = shared or {}
        w = Weights(_ptr(w_router), _ptr(b_router), parr(w1), parr(w3), parr(w2), parr(b1), parr(b2),
                    _ptr(sh.get("w1")), _ptr(sh.get("w3")), _ptr(sh.get("w2")), _ptr(sh.get("b1")), _ptr(sh.get("b2")))
        s = _stream_handle(stream) if stream is not None else None
        try:
            _check(lib().colibri_moe_load_weights(self._h, ctypes.byref(w), s), "colibri_moe_load_weights")
        finally:
            self._keep.clear()

    def forward(self, x, out=None, stream=None):
        """out[T, d] = layer(x[T, d]); x and out are CUDA tensors.  Asynchronous on `stream`."""
        import torch
        T = x.shape[0]
        if out is None:
            odt = torch.float32 if self.cfg.out_dtype == DTYPE_F32 else torch.bfloat16
            out = torch.empty((T, self.cfg.d_model), dtype=odt, device=x.device)
        _check(lib().colibri_moe_forward(self._h, _ptr(x), _ptr(out), T, _stream_handle(stream)),
               "colibri_moe_forward")
        return out

    def forward_ptr(self, x_ptr: int, out_ptr: int, T: int, stream_handle: Optional[int]):
        _check(lib().colibri_moe_forward(self._h, x_ptr, out_ptr, T, stream_handle), "colibri_moe_forward")

    def forward_host(self, x_host, out_host, stream=None):
        """Host buffers in and out (pinned for asynchronous copies); synchronises the stream."""
        T = x_host.shape[0]
        _check(lib().colibri_moe_forward_host(self._h, _ptr(x_host), _ptr(out_host), T, _stream_handle(stream)),
               "colibri_moe_forward_host")
        return out_host

    def forward_host_async(self, x_host, out_host, stream=None):
        """Pipelined host-buffer forward: returns at once; out_host is valid after host_sync()."""
        T = x_host.shape[0]
        _check(lib().colibri_moe_forward_host_async(self._h, _ptr(x_host), _ptr(out_host), T,
                                                    _stream_handle(stream)), "colibri_moe_forward_host_async")
        return out_host

    def host_sync(self):
        _check(lib().colibri_moe_host_sync(self._h), "colibri_moe_host_sync")

    def get_routing(self, T: int, stream=None):
        """Routing of the last forward (T tokens) as CUDA tensors."""
        import torch
        dev = torch.device("cuda", self.device)
        E, k = self.cfg.num_experts, self.cfg.top_k
        r = dict(idx=torch.empty((T, k), dtype=torch.int32, device=dev),
                 gate=torch.empty((T, k), dtype=torch.float32, device=dev),
                 counts=torch.empty(E, dtype=torch.int32, device=dev),
                 offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                 row_of=torch.empty((T, k), dtype=torch.int32, device=dev))
        _check(lib().colibri_moe_get_routing(self._h, _ptr(r["idx"]), _ptr(r["gate"]), _ptr(r["counts"]),
                                             _ptr(r["offsets"]), _ptr(r["row_of"]), _stream_handle(stream)),
               "colibri_moe_get_routing")
        return r

    # -------------------------------------------------------------- expert parallelism
    @property
    def local_experts(self) -> int:
        """El: experts this rank holds (E / ep_size), or E for an ordinary context."""
        return self.cfg.num_experts // self.ep_size if self.ep_size else self.cfg.num_experts

    def ep_dispatch(self, x, send_rows=None, send_counts=None, stream=None):
        """Route x[T, d] over all experts; returns (send_rows [T*k, d], send_counts [E] int32), CUDA tensors,
        rows grouped by expert (rank q's rows are one contiguous block)."""
        import torch
        T, d, k = x.shape[0], self.cfg.d_model, self.cfg.top_k
        if send_rows is None:
            send_rows = torch.empty((T * k, d), dtype=x.dtype, device=x.device)
        if send_counts is None:
            send_counts = torch.empty(self.cfg.num_experts, dtype=torch.int32, device=x.device)
        _check(lib().colibri_moe_ep_dispatch(self._h, _ptr(x), T, _ptr(send_rows), _ptr(send_counts),
                                             _stream_handle(stream)), "colibri_moe_ep_dispatch")
        self._ep_T = T
        return send_rows, send_counts

    def ep_experts(self, recv_rows, recv_counts, y_rows=None, stream=None):
        """Expert FFN of the rows this rank received.  recv_counts: HOST int32 [ep_size, El] (numpy or
        torch); returns y_rows [R, d] fp32 (CUDA), in the order of recv_rows."""
        import numpy as np
        import torch
        rc = np.ascontiguousarray(np.asarray(recv_counts.cpu() if hasattr(recv_counts, "cpu") else recv_counts,
                                             dtype=np.int32))
        if rc.size != self.ep_size * self.local_experts:
            raise ValueError(f"recv_counts must hold ep_size x El = {self.ep_size} x {self.local_experts} entries")
        R = int(rc.sum())
        if y_rows is None:
            y_rows = torch.empty((R, self.cfg.d_model), dtype=torch.float32, device=torch.device("cuda", self.device))
        _check(lib().colibri_moe_ep_experts(self._h, _ptr(recv_rows) if R else None, rc.ctypes.data,
                                            _ptr(y_rows) if R else None, _stream_handle(stream)),
               "colibri_moe_ep_experts")
        return y_rows

    def ep_combine(self, y_back, out=None, stream=None):
        """out[T, d] = gate-weighted sum of the returned expert outputs (T of the last ep_dispatch)."""
        import torch
        if self._ep_T is None:
            raise ColibriError(-5, "colibri_moe_ep_combine")
        if out is None:
            odt = torch.float32 if self.cfg.out_dtype == DTYPE_F32 else torch.bfloat16
            out = torch.empty((self._ep_T, self.cfg.d_model), dtype=odt, device=torch.device("cuda", self.device))
        _check(lib().colibri_moe_ep_combine(self._h, _ptr(y_back) if self._ep_T else None,
                                            _ptr(out) if self._ep_T else None, _stream_handle(stream)),
               "colibri_moe_ep_combine")
        return out

    def debug_buffer(self, which: int):
        p = ctypes.c_void_p()
        rows = ctypes.c_int64()
        _check(lib().colibri_moe_debug_buffer(self._h, which, ctypes.byref(p), ctypes.byref(rows)),
               "colibri_moe_debug_buffer")
        return p.value, rows.value

    def debug_tensor(self, which: int):
        """Copy of an internal buffer (0 Xp, 1 H, 2 Y, 3 token_of_row) as a CUDA tensor.  Synchronises."""
        import torch
        ptr, rows = self.debug_buffer(which)
        d, f = self.cfg.d_model, self.cfg.d_ff
        bf = self.cfg.dtype == DTYPE_BF16
        cols, typestr, view = {0: (d, "<i2", torch.bfloat16) if bf else (d, "<f4", None),
                               1: (f, "<i2", torch.bfloat16) if bf else (f, "<f4", None),
                               2: (d, "<f4", None), 3: (1, "<i4", None)}[which]
        torch.cuda.synchronize(self.device)
        t = torch.as_tensor(_DeviceArray(ptr, (rows, cols), typestr), device=torch.device("cuda", self.device))
        t = t.clone()
        if view is not None:
            t = t.view(view)
        return t.view(-1) if which == 3 else t

    def num_stages(self) -> int:
        n = ctypes.c_int32()
        _check(lib().colibri_moe_num_stages(self._h, ctypes.byref(n)), "colibri_moe_num_stages")
        return n.value

    def last_kernel_count(self) -> int:
        """Kernels the most recent forward enqueued."""
        n = ctypes.c_int32()
        _check(lib().colibri_moe_last_kernel_count(self._h, ctypes.byref(n)), "colibri_moe_last_kernel_count")
        return n.value

    GEMM_KINDS = ("none", "decode_fused", "decode_split", "pair", "single_cta", "simt", "weight_major",
                  "weight_major_fused")

    def last_gemm(self) -> str:
        """The grouped-GEMM form the most recent forward ran (one of GEMM_KINDS)."""
        n = ctypes.c_int32()
        _check(lib().colibri_moe_last_gemm(self._h, ctypes.byref(n)), "colibri_moe_last_gemm")
        return self.GEMM_KINDS[n.value]

    def set_stage_events(self, events):
        """events: list of num_stages()+1 torch.cuda.Event (or None to turn timing off)."""
        if not events:
            _check(lib().colibri_moe_set_stage_events(self._h, None, 0), "colibri_moe_set_stage_events")
            self._events = None
            return
        for e in events:
            e.record()  # makes torch create the underlying cudaEvent_t
        arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
        self._events = (events, arr)
        _check(lib().colibri_moe_set_stage_events(self._h, ctypes.cast(arr, ctypes.c_void_p), len(events)),
               "colibri_moe_set_stage_events")

    def device_status(self) -> int:
        v = ctypes.c_int32()
        _check(lib().colibri_moe_device_status(self._h, ctypes.byref(v)), "colibri_moe_device_status")
        return v.value

    def probe_wait_timeout(self, timeout_us: int, stream=None) -> None:
        """Enqueue one bounded wait that runs out after timeout_us (sets STATUS_WAIT_PROBE)."""
        _check(lib().colibri_moe_probe_wait_timeout(self._h, int(timeout_us), _stream_handle(stream)),
               "colibri_moe_probe_wait_timeout")


class _DeviceArray:
    """Zero-copy view of raw device memory through the CUDA array interface (debug views only)."""

    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 2, "strides": None}
