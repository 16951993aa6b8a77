"""Helpers shared by the GPU parity tests: build a layer from generated inputs, run it through the
C ABI, and compare with the oracle (bit-exact routing, tolerance-bounded outputs)."""
from __future__ import annotations

import numpy as np

import oracle
import testgen

# max |out_gpu - out_oracle| / RMS(out_oracle): fp32 layers and bf16 layers
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
NEAR_TIE = 1e-5


def torch_from_bits(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host_weights(li: testgen.LayerInputs):
    """Host tensors in the layer's dtype, in the argument order of MoELayer.load_weights."""
    import torch
    bf = li.shape.dtype == "bf16"
    conv = (lambda b, f: torch_from_bits(b)) if bf else (lambda b, f: torch.from_numpy(f))
    wr = conv(li.w_router_bits, li.w_router_f32)
    w1 = [conv(b, f) for b, f in zip(li.w1_bits or [None] * len(li.w1_f32), li.w1_f32 or [None] * len(li.w1_bits))]
    w2 = [conv(b, f) for b, f in zip(li.w2_bits or [None] * len(li.w2_f32), li.w2_f32 or [None] * len(li.w2_bits))]
    w3 = None
    if li.w3_f32 or li.w3_bits:
        w3 = [conv(b, f) for b, f in zip(li.w3_bits or [None] * len(li.w3_f32), li.w3_f32 or [None] * len(li.w3_bits))]
    br = None if li.b_router is None else torch.from_numpy(li.b_router)
    b1 = [torch.from_numpy(b) for b in li.b1] or None
    b2 = [torch.from_numpy(b) for b in li.b2] or None
    shared = None
    if li.shape.shared_expert:
        shared = dict(w1=conv(li.ws1_bits, li.ws1_f32), w2=conv(li.ws2_bits, li.ws2_f32))
        if li.shape.act == testgen.ACT_SWIGLU:
            shared["w3"] = conv(li.ws3_bits, li.ws3_f32)
        else:
            shared["b1"] = torch.from_numpy(li.bs1)
            shared["b2"] = torch.from_numpy(li.bs2)
    return dict(w_router=wr, w1=w1, w2=w2, w3=w3, b_router=br, b1=b1, b2=b2, shared=shared)


def make_layer(li: testgen.LayerInputs, max_tokens: int | None = None, out_dtype: str = "f32"):
    from mixture_experts_gemm_gb300 import MoELayer
    s = li.shape
    layer = MoELayer(s.d_model, s.d_ff, s.num_experts, max_tokens or s.T, dtype=s.dtype,
                     act="swiglu" if s.act == testgen.ACT_SWIGLU else "relu_bias",
                     has_router_bias=li.b_router is not None, out_dtype=out_dtype, top_k=s.top_k,
                     gate_mode=s.gate_mode, shared_expert=s.shared_expert)
    layer.load_weights(**host_weights(li))
    return layer


def x_device(li: testgen.LayerInputs, T: int | None = None):
    import torch
    if li.shape.dtype == "bf16":
        x = torch_from_bits(li.x_bits)
    else:
        x = torch.from_numpy(li.x_f32)
    if T is not None:
        x = x[:T]
    return x.contiguous().cuda()


def run(layer, x):
    import torch
    out = layer.forward(x)
    torch.cuda.synchronize()
    r = {k: v.cpu().numpy() for k, v in layer.get_routing(x.shape[0]).items()}
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), r


def rel_err(out, ref):
    rms = float(np.sqrt(np.mean(ref ** 2)))
    return float(np.max(np.abs(out - ref))) / rms


def check_routing(gpu: dict, logits: np.ndarray, o_idx: np.ndarray, o_gate: np.ndarray, E: int,
                  o_row_of: np.ndarray | None = None, o_offsets_raw: np.ndarray | None = None,
                  gate_mode: int = 0):
    """Bit-exact routing outside near ties; the GPU's own bookkeeping valid everywhere.

    Returns the number of near-tie tokens excluded."""
    T = logits.shape[0]
    k = o_idx.shape[1]
    tie = oracle.near_tie_tokens(logits, NEAR_TIE, k=k)
    g_idx, g_gate, g_row = gpu["idx"], gpu["gate"], gpu["row_of"]
    counts, offs = gpu["counts"], gpu["offsets"]
    keep = ~tie
    assert np.array_equal(g_idx[keep], o_idx[keep]), "routing indices differ on a non-near-tie token"
    np.testing.assert_allclose(g_gate[keep], o_gate[keep], rtol=0, atol=1e-5)
    assert np.all((g_idx >= 0) & (g_idx < E))
    assert all(len(set(row)) == k for row in g_idx.tolist())   # distinct experts per token
    if gate_mode == 0:
        assert np.all(np.abs(g_gate.sum(axis=1, dtype=np.float64) - 1.0) <= k * 2.0 ** -23)
    else:
        assert np.all(g_gate.sum(axis=1) <= 1.0 + 1e-6)
    # counts: exact after removing near-tie tokens from both sides
    gc = np.bincount(g_idx[keep].ravel(), minlength=E)
    oc = np.bincount(o_idx[keep].ravel(), minlength=E)
    assert np.array_equal(gc, oc)
    assert np.array_equal(counts, np.bincount(g_idx.ravel(), minlength=E))
    # offsets: segments start on multiples of 128 and hold their counts
    pad = (counts + 127) // 128 * 128
    assert offs[0] == 0 and np.array_equal(np.diff(offs), pad)
    # rows: row_of - offsets[e] is the token's rank among the tokens of e, ascending t
    rank = g_row - offs[g_idx]
    fill = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for s in range(k):
            e = g_idx[t, s]
            assert rank[t, s] == fill[e], (t, s, e, rank[t, s], fill[e])
            fill[e] += 1
    if not tie.any() and o_row_of is not None:
        # no near ties: ranks equal the oracle's dispatch bit for bit
        assert np.array_equal(rank, o_row_of - o_offsets_raw[o_idx])
    return int(tie.sum())


def sample_tokens(idx: np.ndarray, E: int, n_random: int, seed: int = 0):
    """Sample rows for large-batch checks: every token of each expert's first and last position, the
    tokens of the rarest experts, plus n_random others."""
    T = idx.shape[0]
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(T, size=min(n_random, T), replace=False).tolist())
    pick.update([0, T - 1])
    counts = np.bincount(idx.ravel(), minlength=E)
    for e in range(E):
        toks = np.nonzero((idx == e).any(axis=1))[0]
        if len(toks):
            pick.update([int(toks[0]), int(toks[-1])])
        if 0 < counts[e] <= 8:
            pick.update(int(t) for t in toks)
    return np.array(sorted(pick), dtype=np.int32)


def bf16_h_bound(li: testgen.LayerInputs, idx: np.ndarray, gate: np.ndarray) -> np.ndarray:
    """Per output element, what the bf16 path's one intermediate rounding can add to its error: H, the
    activation between the two projections, is stored in bf16, each element within one bf16 ulp
    (2^-8 relative, one half-ulp rounding plus fp32 accumulation ahead of it) of its exact value, so
    out[t, i] moves by at most 2^-8 * sum over t's slots of g * sum_j |W2[i, j] * H[t, j]|.  Exact H
    in fp64; routing (idx, gate: the routed slots) given; the shared expert adds with weight 1.  This
    matters beside the max|err| / RMS budget only for output outliers (top-1, unnormalised gates,
    short K), where that rounding alone can exceed 2e-2 x RMS."""
    s = li.shape
    x = li.x_f32.astype(np.float64)
    acc = np.zeros(x.shape)
    swiglu = s.act == testgen.ACT_SWIGLU

    def abs_terms(xr, w1, w3, w2, b1):
        if swiglu:
            g = xr @ w1.astype(np.float64).T
            u = xr @ w3.astype(np.float64).T
            h = g / (1.0 + np.exp(-g)) * u
        else:
            h = np.maximum(xr @ w1.astype(np.float64).T + b1, 0.0)
        return np.abs(h) @ np.abs(w2.astype(np.float64)).T

    for e in range(s.num_experts):
        toks, slots = np.nonzero(idx == e)
        if len(toks) == 0:
            continue
        a = abs_terms(x[toks], li.w1_f32[e], li.w3_f32[e] if swiglu else None, li.w2_f32[e],
                      None if swiglu else li.b1[e])
        np.add.at(acc, toks, gate[toks, slots][:, None] * a)
    if s.shared_expert:
        acc += abs_terms(x, li.ws1_f32, li.ws3_f32 if swiglu else None, li.ws2_f32, None if swiglu else li.bs1)
    return acc * 2.0 ** -8
