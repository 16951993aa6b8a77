"""Seeded synthetic inputs for the MoE layer: the five workload shapes and their tensors.

This module holds no arithmetic of the layer itself (no routing, no matmul, no
activation).  It only draws inputs (x, router weights and bias, expert weights
and biases) from the counter-based generator defined in ``testgen.c``; both the
CPU oracle and the CUDA path consume exactly these bits.

Workloads (shapes and distributions as stated for the benchmark; ``N(0, v)``
takes ``v`` as the variance):

* ``tiny-moe-4e2r``   T=64,   d=256,  E=4,  f=512,   ReLU with biases, fp32
* ``1.3b-8e``         T=512,  d=2048, E=8,  f=5632,  SwiGLU, bf16
* ``mixtral-prefill`` T=8192, d=4096, E=8,  f=14336, SwiGLU, bf16
* ``mixtral-decode``  the Mixtral weights with T in {1, 4, 16, 32}
* ``skewed-16e``      T=4096, d=2048, E=16, f=1408,  SwiGLU, bf16,
                      router bias b_r[e] = 1.5 * ln(1 / (e + 1))

x ~ N(0, 1); weights ~ N(0, 1/fan_in); biases ~ N(0, 0.01); router weights
~ N(0, 1/d).  Seed 0 throughout.  Tensor ids: x = 0, W_r = 1, b_r = 2, and for
expert e: 16 + 8e + {0: W1 (ReLU) or W_gate (SwiGLU), 1: W_up, 2: W2/W_down,
3: b1, 4: b2}; the optional shared expert: 8 + {0..4} in the same order.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "testgen.c")
_LIB = os.path.join(_HERE, "libtestgen.so")

ACT_RELU_BIAS = 0
ACT_SWIGLU = 1


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d_model: int
    d_ff: int
    num_experts: int
    act: int                 # ACT_RELU_BIAS or ACT_SWIGLU
    dtype: str               # "f32" or "bf16"
    zipf_router_bias: bool = False
    top_k: int = 2
    gate_mode: int = 0       # 0 softmax over the selected experts, 1 full softmax (unnormalised)
    shared_expert: bool = False

    def with_T(self, T: int) -> "LayerShape":
        return LayerShape(self.name, T, self.d_model, self.d_ff, self.num_experts, self.act,
                          self.dtype, self.zipf_router_bias, self.top_k, self.gate_mode, self.shared_expert)


CONFIGS = {
    "tiny-moe-4e2r": LayerShape("tiny-moe-4e2r", 64, 256, 512, 4, ACT_RELU_BIAS, "f32"),
    "1.3b-8e": LayerShape("1.3b-8e", 512, 2048, 5632, 8, ACT_SWIGLU, "bf16"),
    "mixtral-prefill": LayerShape("mixtral-prefill", 8192, 4096, 14336, 8, ACT_SWIGLU, "bf16"),
    "mixtral-decode": LayerShape("mixtral-decode", 32, 4096, 14336, 8, ACT_SWIGLU, "bf16"),
    "skewed-16e": LayerShape("skewed-16e", 4096, 2048, 1408, 16, ACT_SWIGLU, "bf16", zipf_router_bias=True),
}
DECODE_TOKENS = (1, 4, 16, 32)

TID_X, TID_WR, TID_BR = 0, 1, 2
TID_SHARED = 8  # shared expert: 8 W1/W_gate, 9 W_up, 10 W2/W_down, 11 b1, 12 b2


def tid_expert(e: int, which: int) -> int:
    """which: 0 W1/W_gate, 1 W_up, 2 W2/W_down, 3 b1, 4 b2."""
    return 16 + 8 * e + which


def build_lib(force: bool = False) -> str:
    """Compile libtestgen.so with gcc (plain C, OpenMP, no fused multiply-add contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_lib())
        u64, dbl = ctypes.c_uint64, ctypes.c_double
        vp = ctypes.c_void_p
        lib.testgen_normal_at.restype = dbl
        lib.testgen_normal_at.argtypes = [u64, u64, u64]
        lib.testgen_fill_f32.restype = None
        lib.testgen_fill_f32.argtypes = [u64, u64, u64, u64, dbl, vp]
        lib.testgen_fill_bf16.restype = None
        lib.testgen_fill_bf16.argtypes = [u64, u64, u64, u64, dbl, vp]
        lib.testgen_f32_to_bf16.restype = None
        lib.testgen_f32_to_bf16.argtypes = [vp, vp, u64]
        lib.testgen_bf16_to_f32.restype = None
        lib.testgen_bf16_to_f32.argtypes = [vp, vp, u64]
        _lib = lib
    return _lib


def normal_at(seed: int, tensor_id: int, i: int) -> float:
    return _L().testgen_normal_at(seed, tensor_id, i)


def normal_f32(seed: int, tensor_id: int, shape, std: float, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    _L().testgen_fill_f32(seed, tensor_id, offset, n, float(std), out.ctypes.data)
    return out.reshape(shape)


def normal_bf16_bits(seed: int, tensor_id: int, shape, std: float, offset: int = 0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    _L().testgen_fill_bf16(seed, tensor_id, offset, n, float(std), out.ctypes.data)
    return out.reshape(shape)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _L().testgen_f32_to_bf16(a.ctypes.data, out.ctypes.data, a.size)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float32)
    _L().testgen_bf16_to_f32(b.ctypes.data, out.ctypes.data, b.size)
    return out


@dataclass
class LayerInputs:
    """Host arrays of one layer instance.

    ``*_f32`` hold the values as fp32 (for bf16 shapes: the bf16 values widened);
    ``*_bits`` hold bf16 bit patterns (bf16 shapes only).  Either side may be
    skipped at generation time to save host memory on the large shapes.
    """
    shape: LayerShape
    seed: int
    x_f32: Optional[np.ndarray] = None
    x_bits: Optional[np.ndarray] = None
    w_router_f32: Optional[np.ndarray] = None
    w_router_bits: Optional[np.ndarray] = None
    b_router: Optional[np.ndarray] = None
    w1_f32: List[np.ndarray] = field(default_factory=list)
    w3_f32: List[np.ndarray] = field(default_factory=list)
    w2_f32: List[np.ndarray] = field(default_factory=list)
    w1_bits: List[np.ndarray] = field(default_factory=list)
    w3_bits: List[np.ndarray] = field(default_factory=list)
    w2_bits: List[np.ndarray] = field(default_factory=list)
    b1: List[np.ndarray] = field(default_factory=list)
    b2: List[np.ndarray] = field(default_factory=list)
    # shared expert (same shapes as one routed expert)
    ws1_f32: Optional[np.ndarray] = None
    ws3_f32: Optional[np.ndarray] = None
    ws2_f32: Optional[np.ndarray] = None
    ws1_bits: Optional[np.ndarray] = None
    ws3_bits: Optional[np.ndarray] = None
    ws2_bits: Optional[np.ndarray] = None
    bs1: Optional[np.ndarray] = None
    bs2: Optional[np.ndarray] = None


def _draw(seed, tid, shape, std, is_bf16, want_f32, want_bits):
    if not is_bf16:
        return normal_f32(seed, tid, shape, std), None
    bits = normal_bf16_bits(seed, tid, shape, std)
    return (bf16_bits_to_f32(bits) if want_f32 else None), (bits if want_bits else None)


def zipf_router_bias(E: int) -> np.ndarray:
    """b_r[e] = 1.5 * ln(1 / (e + 1)) in fp32: expert 0 hottest."""
    return np.array([1.5 * math.log(1.0 / (e + 1)) for e in range(E)], dtype=np.float32)


def make_weights(shape: LayerShape, seed: int = 0, want_f32: bool = True, want_bits: bool = True,
                 experts=None) -> LayerInputs:
    """Router and expert parameters (x not drawn).  ``experts`` limits which experts are drawn."""
    bf = shape.dtype == "bf16"
    d, f, E = shape.d_model, shape.d_ff, shape.num_experts
    li = LayerInputs(shape=shape, seed=seed)
    li.w_router_f32, li.w_router_bits = _draw(seed, TID_WR, (E, d), math.sqrt(1.0 / d), bf, True, want_bits)
    if shape.zipf_router_bias:
        li.b_router = zipf_router_bias(E)
    ex = range(E) if experts is None else experts
    for e in ex:
        a, b = _draw(seed, tid_expert(e, 0), (f, d), math.sqrt(1.0 / d), bf, want_f32, want_bits)
        li.w1_f32.append(a); li.w1_bits.append(b)
        if shape.act == ACT_SWIGLU:
            a, b = _draw(seed, tid_expert(e, 1), (f, d), math.sqrt(1.0 / d), bf, want_f32, want_bits)
            li.w3_f32.append(a); li.w3_bits.append(b)
        a, b = _draw(seed, tid_expert(e, 2), (d, f), math.sqrt(1.0 / f), bf, want_f32, want_bits)
        li.w2_f32.append(a); li.w2_bits.append(b)
        if shape.act == ACT_RELU_BIAS:
            li.b1.append(normal_f32(seed, tid_expert(e, 3), (f,), 0.1))
            li.b2.append(normal_f32(seed, tid_expert(e, 4), (d,), 0.1))
    if shape.shared_expert:
        li.ws1_f32, li.ws1_bits = _draw(seed, TID_SHARED + 0, (f, d), math.sqrt(1.0 / d), bf, want_f32, want_bits)
        if shape.act == ACT_SWIGLU:
            li.ws3_f32, li.ws3_bits = _draw(seed, TID_SHARED + 1, (f, d), math.sqrt(1.0 / d), bf, want_f32, want_bits)
        li.ws2_f32, li.ws2_bits = _draw(seed, TID_SHARED + 2, (d, f), math.sqrt(1.0 / f), bf, want_f32, want_bits)
        if shape.act == ACT_RELU_BIAS:
            li.bs1 = normal_f32(seed, TID_SHARED + 3, (f,), 0.1)
            li.bs2 = normal_f32(seed, TID_SHARED + 4, (d,), 0.1)
    return li


def make_x(shape: LayerShape, T: Optional[int] = None, seed: int = 0, want_f32: bool = True,
           want_bits: bool = True):
    """Activations x[T, d] ~ N(0, 1): row t is elements t*d .. t*d+d-1 of stream 0."""
    T = shape.T if T is None else T
    return _draw(seed, TID_X, (T, shape.d_model), 1.0, shape.dtype == "bf16", want_f32, want_bits)


def make_inputs(shape: LayerShape, T: Optional[int] = None, seed: int = 0, want_f32: bool = True,
                want_bits: bool = True) -> LayerInputs:
    li = make_weights(shape, seed, want_f32, want_bits)
    li.x_f32, li.x_bits = make_x(shape, T, seed, want_f32 or shape.dtype == "f32", want_bits)
    return li
