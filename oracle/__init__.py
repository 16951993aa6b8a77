"""CPU oracle of one MoE layer forward -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper over ``colibri_oracle.c`` (plain C, fp64).  Only ``tests/``,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import it;
the product library never does.  It shares no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "colibri_oracle.c")
_HDR = os.path.join(_HERE, "colibri_oracle.h")
_LIB = os.path.join(_HERE, "libcolibri_oracle.so")

ACT_RELU_BIAS = 0
ACT_SWIGLU = 1
GATE_PAIR_SOFTMAX = 0
GATE_FULL_SOFTMAX = 1


def build_lib(force: bool = False) -> str:
    """Compile the oracle with gcc: C11, -O2, OpenMP over independent tokens, no FMA contraction."""
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Cfg(ctypes.Structure):
    _fields_ = [("d_model", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("num_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("act", ctypes.c_int32), ("gate_mode", ctypes.c_int32),
                ("has_shared", ctypes.c_int32)]


class _W(ctypes.Structure):
    _fields_ = [("w_router", ctypes.c_void_p), ("b_router", ctypes.c_void_p), ("w1", ctypes.c_void_p),
                ("w3", ctypes.c_void_p), ("w2", ctypes.c_void_p), ("b1", ctypes.c_void_p),
                ("b2", ctypes.c_void_p), ("ws1", ctypes.c_void_p), ("ws3", ctypes.c_void_p),
                ("ws2", ctypes.c_void_p), ("bs1", ctypes.c_void_p), ("bs2", ctypes.c_void_p)]


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_lib())
        vp, i32 = ctypes.c_void_p, ctypes.c_int32
        for name, args in {
            "oracle_router_logits": [vp, vp, vp, i32, vp],
            "oracle_topk": [vp, vp, i32, vp, vp],
            "oracle_shared_ffn": [vp, vp, vp, vp],
            "oracle_dispatch": [vp, vp, i32, vp, vp, vp, vp],
            "oracle_expert_ffn": [vp, vp, i32, vp, vp],
            "oracle_forward": [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp],
            "oracle_forward_rows": [vp, vp, vp, i32, vp, vp, vp, i32, vp],
        }.items():
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = args
        _lib = lib
    return _lib


def _f32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc != 0:
        raise OracleError(f"{what} returned {rc}")


class OracleLayer:
    """One MoE layer's parameters held as fp32 host arrays, plus the oracle's entry points."""

    def __init__(self, d_model: int, d_ff: int, num_experts: int, act: int, w_router,
                 w1: Sequence, w2: Sequence, w3: Optional[Sequence] = None, b_router=None,
                 b1: Optional[Sequence] = None, b2: Optional[Sequence] = None, top_k: int = 2,
                 gate_mode: int = GATE_PAIR_SOFTMAX, shared: Optional[dict] = None):
        """shared: dict(w1=[f,d], w3=[f,d] or None, w2=[d,f], b1=[f] or None, b2=[d] or None)."""
        self.d, self.f, self.E, self.act = d_model, d_ff, num_experts, act
        self.k = top_k
        self.cfg = _Cfg(d_model, d_ff, num_experts, top_k, act, gate_mode, int(shared is not None))
        self._shared = None if shared is None else {k: _f32(v) for k, v in shared.items()}
        # keep every array alive for as long as the struct points into it
        self._wr = _f32(w_router)
        self._br = _f32(b_router)
        self._w1 = [_f32(a) for a in w1]
        self._w2 = [_f32(a) for a in w2]
        self._w3 = None if w3 is None else [_f32(a) for a in w3]
        self._b1 = None if b1 is None else [_f32(a) for a in b1]
        self._b2 = None if b2 is None else [_f32(a) for a in b2]

        def parr(lst):
            if lst is None:
                return None
            arr = (ctypes.c_void_p * len(lst))(*[a.ctypes.data for a in lst])
            return arr

        self._p1, self._p2 = parr(self._w1), parr(self._w2)
        self._p3, self._pb1, self._pb2 = parr(self._w3), parr(self._b1), parr(self._b2)
        addr = lambda p: None if p is None else ctypes.cast(p, ctypes.c_void_p).value
        sh = self._shared or {}
        self.w = _W(_ptr(self._wr), _ptr(self._br), addr(self._p1), addr(self._p3), addr(self._p2),
                    addr(self._pb1), addr(self._pb2), _ptr(sh.get("w1")), _ptr(sh.get("w3")), _ptr(sh.get("w2")),
                    _ptr(sh.get("b1")), _ptr(sh.get("b2")))

    @classmethod
    def from_inputs(cls, li) -> "OracleLayer":
        """Build from a ``testgen.LayerInputs`` (its fp32 views)."""
        s = li.shape
        shared = None
        if getattr(s, "shared_expert", False):
            shared = dict(w1=li.ws1_f32, w3=li.ws3_f32, w2=li.ws2_f32, b1=li.bs1, b2=li.bs2)
        return cls(s.d_model, s.d_ff, s.num_experts, s.act, li.w_router_f32, li.w1_f32, li.w2_f32,
                   w3=li.w3_f32 or None, b_router=li.b_router, b1=li.b1 or None, b2=li.b2 or None,
                   top_k=s.top_k, gate_mode=getattr(s, "gate_mode", GATE_PAIR_SOFTMAX), shared=shared)

    def _args(self):
        return ctypes.byref(self.cfg), ctypes.byref(self.w)

    def router_logits(self, x) -> np.ndarray:
        x = _f32(x)
        T = x.shape[0]
        L = np.empty((T, self.E), dtype=np.float64)
        _check(_L().oracle_router_logits(*self._args(), _ptr(x), T, _ptr(L)), "oracle_router_logits")
        return L

    def topk(self, logits):
        logits = np.ascontiguousarray(logits, dtype=np.float64)
        T = logits.shape[0]
        idx = np.empty((T, self.k), dtype=np.int32)
        gate = np.empty((T, self.k), dtype=np.float64)
        _check(_L().oracle_topk(ctypes.byref(self.cfg), _ptr(logits), T, _ptr(idx), _ptr(gate)), "oracle_topk")
        return idx, gate

    top2 = topk

    def dispatch(self, idx):
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        T = idx.shape[0]
        counts = np.empty(self.E, dtype=np.int32)
        offs = np.empty(self.E + 1, dtype=np.int32)
        row_of = np.empty((T, self.k), dtype=np.int32)
        tok = np.empty(max(self.k * T, 1), dtype=np.int32)
        _check(_L().oracle_dispatch(ctypes.byref(self.cfg), _ptr(idx), T, _ptr(counts), _ptr(offs),
                                    _ptr(row_of), _ptr(tok)), "oracle_dispatch")
        return counts, offs, row_of, tok[:self.k * T]

    def expert_ffn(self, e: int, x_t) -> np.ndarray:
        x_t = _f32(x_t)
        y = np.empty(self.d, dtype=np.float64)
        _check(_L().oracle_expert_ffn(*self._args(), e, _ptr(x_t), _ptr(y)), "oracle_expert_ffn")
        return y

    def shared_ffn(self, x_t) -> np.ndarray:
        x_t = _f32(x_t)
        y = np.empty(self.d, dtype=np.float64)
        _check(_L().oracle_shared_ffn(*self._args(), _ptr(x_t), _ptr(y)), "oracle_shared_ffn")
        return y

    def forward(self, x):
        """Returns dict(out, idx, gate, counts, offsets_raw, row_of, logits)."""
        x = _f32(x)
        T = x.shape[0]
        out = np.empty((T, self.d), dtype=np.float64)
        idx = np.empty((T, self.k), dtype=np.int32)
        gate = np.empty((T, self.k), dtype=np.float64)
        counts = np.empty(self.E, dtype=np.int32)
        offs = np.empty(self.E + 1, dtype=np.int32)
        row_of = np.empty((T, self.k), dtype=np.int32)
        L = np.empty((T, self.E), dtype=np.float64)
        _check(_L().oracle_forward(*self._args(), _ptr(x), T, _ptr(out), _ptr(idx), _ptr(gate), _ptr(counts),
                                   _ptr(offs), _ptr(row_of), _ptr(L)), "oracle_forward")
        return dict(out=out, idx=idx, gate=gate, counts=counts, offsets_raw=offs, row_of=row_of, logits=L)

    def forward_rows(self, x, idx, gate, tokens) -> np.ndarray:
        x = _f32(x)
        idx = np.ascontiguousarray(idx, dtype=np.int32)
        gate = np.ascontiguousarray(gate, dtype=np.float64)
        tokens = np.ascontiguousarray(tokens, dtype=np.int32)
        out = np.empty((len(tokens), self.d), dtype=np.float64)
        _check(_L().oracle_forward_rows(*self._args(), _ptr(x), x.shape[0], _ptr(idx), _ptr(gate), _ptr(tokens),
                                        len(tokens), _ptr(out)), "oracle_forward_rows")
        return out


def near_tie_tokens(logits: np.ndarray, eps: float = 1e-5, k: int = 2) -> np.ndarray:
    """Tokens whose top-k set or slot order could flip under rounding: a gap between consecutive
    ranks 1..k+1 of the fp64 logits below ``eps``."""
    s = -np.sort(-np.asarray(logits, dtype=np.float64), axis=1)
    tie = np.zeros(s.shape[0], dtype=bool)
    for j in range(min(k, s.shape[1] - 1)):
        tie |= (s[:, j] - s[:, j + 1]) < eps
    return tie
