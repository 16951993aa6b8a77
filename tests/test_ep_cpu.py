"""Expert parallelism on CPU ranks: the exchange of ``mixture_experts_gemm_gb300.ep`` (count and row
all-to-alls through gloo, split sizes, the return trip) with the oracle standing in for the kernels.
Each rank's output must equal the single-process oracle forward of its batch bit for bit."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import testgen
from ep_oracle_backend import OracleEP
from mixture_experts_gemm_gb300 import ep


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shape(total_T):
    # 8 experts with a Zipf router bias (some experts get few or no rows), SwiGLU
    return testgen.LayerShape("ep-cpu", total_T, 64, 96, 8, testgen.ACT_SWIGLU, "f32", zipf_router_bias=True)


def _batches(li, sizes):
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    return [li.x_f32[a:a + n] for a, n in zip(starts, sizes)]


def _worker(rank, world, port, sizes, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
        dist.init_process_group("gloo", rank=rank, world_size=world)
        li = testgen.make_inputs(_shape(sum(sizes)), want_bits=False)
        L = oracle.OracleLayer.from_inputs(li)
        x = _batches(li, sizes)[rank]
        be = OracleEP(L, rank, world)
        out = ep.ep_forward(be, torch.from_numpy(np.ascontiguousarray(x)))
        ref = L.forward(x)["out"] if len(x) else np.zeros((0, li.shape.d_model))
        q.put((rank, bool(np.array_equal(out.numpy(), ref)), out.shape[0], int(np.asarray(be.idx).size)))
        dist.barrier()
        dist.destroy_process_group()
    except Exception as e:  # report instead of hanging the parent
        q.put((rank, f"error: {e!r}", -1, -1))
        raise


@pytest.mark.parametrize("sizes", [[40, 23], [40, 0, 17, 33]], ids=["2-ranks", "4-ranks-one-empty"])
def test_gloo_ranks_reproduce_the_single_process_oracle(sizes):
    world, port = len(sizes), _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, sizes, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for rank, equal, T, n_idx in res:
        assert equal is True, (rank, equal)
        assert T == sizes[rank] and n_idx == 2 * sizes[rank]


def test_local_emulation_of_the_exchange_matches_the_oracle():
    """ep_forward_local (every rank in one process; the GPU test's driver) on the oracle stand-in."""
    sizes = [30, 12, 0, 25]
    li = testgen.make_inputs(_shape(sum(sizes)), want_bits=False)
    L = oracle.OracleLayer.from_inputs(li)
    xs = _batches(li, sizes)
    backends = [OracleEP(L, r, len(sizes)) for r in range(len(sizes))]
    outs = ep.ep_forward_local(backends, [torch.from_numpy(np.ascontiguousarray(x)) for x in xs])
    for x, out in zip(xs, outs):
        ref = L.forward(x)["out"] if len(x) else np.zeros((0, li.shape.d_model))
        assert np.array_equal(out.numpy(), ref)


def test_split_sizes():
    # 2 ranks, 4 experts (2 each): this rank routes 3, 0 rows to experts 0, 1 (rank 0) and 5, 2 to
    # experts 2, 3 (rank 1); it receives [1, 4] from rank 0 and [2, 2] from rank 1
    s, r = ep.split_sizes([3, 0, 5, 2], [[1, 4], [2, 2]], 2)
    assert s == [3, 7] and r == [5, 4]
    with pytest.raises(ValueError):
        ep.split_sizes([1, 2, 3], [[1], [2], [3]], 2)
    with pytest.raises(ValueError):
        ep.split_sizes([1, -2], [[1], [2]], 2)
