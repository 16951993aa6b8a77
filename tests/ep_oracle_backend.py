"""A rank's compute side for the expert-parallel exchange, written with the oracle (fp64, CPU).

Test infrastructure: it stands in for the CUDA kernels so that ``mixture_experts_gemm_gb300.ep``'s
exchange logic runs on CPU ranks (gloo) and must reproduce the single-process oracle bit for bit.
"""
from __future__ import annotations

import numpy as np

import oracle


class OracleEP:
    """dispatch / experts / combine of rank ``rank`` of ``ep_size`` with the oracle's arithmetic."""

    def __init__(self, L: "oracle.OracleLayer", rank: int, ep_size: int):
        self.L, self.rank, self.ep_size = L, rank, ep_size
        self.El = L.E // ep_size

    def dispatch(self, x):
        import torch
        xs = np.ascontiguousarray(x.numpy(), dtype=np.float32)
        T = xs.shape[0]
        if T:
            logits = self.L.router_logits(xs)
            self.idx, self.gate = self.L.topk(logits)
        else:
            self.idx = np.zeros((0, self.L.k), np.int32)
            self.gate = np.zeros((0, self.L.k))
        counts, _, self.row_of, tok = self.L.dispatch(self.idx)
        # the oracle's dispatch order: experts ascending, tokens ascending inside each
        send = xs[tok] if T else np.zeros((0, xs.shape[1]), np.float32)
        return torch.from_numpy(np.ascontiguousarray(send)), torch.from_numpy(counts.astype(np.int32))

    def experts(self, recv_rows, recv_counts):
        import torch
        rows = recv_rows.numpy()
        rc = np.asarray(recv_counts).reshape(self.ep_size, self.El)
        y = np.zeros((rows.shape[0], self.L.d), dtype=np.float64)
        i = 0
        for p in range(self.ep_size):          # source-major, each source's rows by local expert
            for j in range(self.El):
                e = self.rank * self.El + j
                for _ in range(int(rc[p, j])):
                    y[i] = self.L.expert_ffn(e, rows[i])
                    i += 1
        assert i == rows.shape[0]
        return torch.from_numpy(y)

    def combine(self, y_back):
        import torch
        yb = y_back.numpy()
        T, k = self.idx.shape
        out = np.zeros((T, self.L.d), dtype=np.float64)
        for t in range(T):
            for s in range(k):                  # slot order, as the oracle's forward sums
                out[t] += self.gate[t, s] * yb[self.row_of[t, s]]
        return torch.from_numpy(out)
