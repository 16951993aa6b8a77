"""Expert parallelism: the experts of one MoE layer split over ep_size GPUs, one process per GPU.

The articles run the whole layer on one device and describe no collective; this splits the layer's
Dispatch and Compute stages (zskr.cn/news/2272131 2.1) across GPUs.  Rank r owns experts
[r*El, (r+1)*El), El = E / ep_size, routes its own batch over all E experts, and computes the expert
FFN for every row routed to its experts by any rank.  One step:

    ep_dispatch          rows grouped by expert -> send_rows, send_counts [E]
    all-to-all           send_counts -> recv_counts [ep_size, El] (El per peer)
    all-to-all           send_rows -> recv_rows (split sizes: per-peer sums of the counts)
    ep_experts           recv_rows -> y_rows (fp32 expert outputs, same order)
    all-to-all           y_rows -> y_back (the split sizes swapped)
    ep_combine           y_back -> out (gate-weighted sum in slot order)

The kernels run in ``libcolibri_moe.so`` (``MoELayer.ep_*``); this module only sizes and issues the
exchanges, through ``torch.distributed`` (NCCL on GPUs).  Rows cross GPUs only through those
collectives, into local buffers, before any kernel reads them.

``ep_forward`` takes any object with ``dispatch / experts / combine`` methods (``LayerEP`` wraps an
expert-parallel ``MoELayer``), so the exchange logic runs the same on CPU ranks (gloo) in tests.
``ep_forward_local`` runs every rank of a step in one process on one device, with the all-to-alls
done as local copies: the same result, for checking the kernels on a single GPU.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np


def split_sizes(send_counts, recv_counts, ep_size: int) -> Tuple[List[int], List[int]]:
    """Rows this rank sends to / receives from each peer: the per-peer sums of the per-expert
    counts (send_counts [E] of this rank, recv_counts [ep_size, El] received from the peers)."""
    sc = np.asarray(send_counts, dtype=np.int64).reshape(ep_size, -1)
    rc = np.asarray(recv_counts, dtype=np.int64).reshape(ep_size, -1)
    if sc.shape != rc.shape:
        raise ValueError(f"send counts {sc.shape} and receive counts {rc.shape} disagree")
    if (sc < 0).any() or (rc < 0).any():
        raise ValueError("negative row count")
    return [int(v) for v in sc.sum(axis=1)], [int(v) for v in rc.sum(axis=1)]


class LayerEP:
    """The compute side of one rank: an expert-parallel ``MoELayer`` (ep_size > 0)."""

    def __init__(self, layer, stream=None):
        if not layer.ep_size:
            raise ValueError("LayerEP needs a MoELayer created with ep_size > 0")
        self.layer = layer
        self.stream = stream

    def dispatch(self, x):
        return self.layer.ep_dispatch(x, stream=self.stream)

    def experts(self, recv_rows, recv_counts):
        return self.layer.ep_experts(recv_rows, recv_counts, stream=self.stream)

    def combine(self, y_back):
        return self.layer.ep_combine(y_back, stream=self.stream)


def ep_forward(backend, x, group=None):
    """One expert-parallel step of this rank through torch.distributed (every rank calls it)."""
    import torch.distributed as dist
    ep_size = dist.get_world_size(group)
    send_rows, send_counts = backend.dispatch(x)
    recv_counts = send_counts.new_empty(send_counts.shape)
    dist.all_to_all_single(recv_counts, send_counts, group=group)       # El counts per peer
    sc = send_counts.cpu().numpy()
    rc = recv_counts.cpu().numpy().reshape(ep_size, -1)                  # [source, local expert]
    s_split, r_split = split_sizes(sc, rc, ep_size)
    recv_rows = send_rows.new_empty((sum(r_split), send_rows.shape[1]))
    dist.all_to_all_single(recv_rows, send_rows, r_split, s_split, group=group)
    y_rows = backend.experts(recv_rows, rc)
    y_back = y_rows.new_empty((send_rows.shape[0], y_rows.shape[1]))
    dist.all_to_all_single(y_back, y_rows, s_split, r_split, group=group)
    return backend.combine(y_back)


def ep_forward_local(backends: Sequence, xs: Sequence):
    """One step of all ep_size ranks in this process: backends[r] is rank r's compute side, xs[r] its
    batch; the all-to-alls become copies between the ranks' buffers.  Returns every rank's output."""
    import torch
    n = len(backends)
    sends = [b.dispatch(x) for b, x in zip(backends, xs)]
    counts = [sc.cpu().numpy().astype(np.int64).reshape(n, -1) for _, sc in sends]  # [dest, local expert]
    per_peer = [c.sum(axis=1) for c in counts]                                      # rows p sends to each q
    starts = [np.concatenate([[0], np.cumsum(pp)[:-1]]) for pp in per_peer]

    def block(p, q, rows):  # the rows p exchanges with q, in p's send order
        a = int(starts[p][q])
        return rows[a:a + int(per_peer[p][q])]

    y_rows = []
    for q in range(n):
        rc = np.stack([counts[p][q] for p in range(n)]).astype(np.int32)           # [source, local expert]
        recv = torch.cat([block(p, q, sends[p][0]) for p in range(n)])
        y_rows.append(backends[q].experts(recv, rc))
    outs = []
    for p in range(n):
        # rank q's outputs for p's rows sit after those of the sources before p
        pieces = []
        for q in range(n):
            before = int(sum(per_peer[s][q] for s in range(p)))
            pieces.append(y_rows[q][before:before + int(per_peer[p][q])])
        outs.append(backends[p].combine(torch.cat(pieces)))
    return outs
