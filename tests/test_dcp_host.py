"""Host side of the decode-context-parallel top-k (CPU; gloo for the exchange).

The position bookkeeping must partition every context exactly, and the
exchange must hand every rank all ranks' candidates; the local selection and
the merge are taken here from the oracle, so that the protocol itself is
checked against the single-rank definition.
"""
import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from top_selection_dsa_gb300 import dcp  # noqa: E402


def test_ownership_partitions_every_context():
    for world, inter in ((1, 1), (2, 1), (2, 64), (4, 16), (8, 64)):
        for L in (0, 1, 63, 64, 65, 1000, 4096 + 17):
            owned = [dcp.owned_positions(L, r, world, inter).tolist() for r in range(world)]
            allp = sorted(p for o in owned for p in o)
            assert allp == list(range(L))
            for r, o in enumerate(owned):
                assert o == sorted(o)                                   # local order = global order
                assert all((p // inter) % world == r for p in o)
                assert len(o) == dcp.local_len(L, r, world, inter)
    t = torch.tensor([0, 1, 129, 5000])
    assert dcp.local_len(t, 1, 4, 64).tolist() == [dcp.local_len(int(x), 1, 4, 64) for x in t]
    assert dcp.local_to_global(torch.tensor([-1, 0, 63, 64]), 1, 4, 64).tolist() == [-1, 64, 127, 320]


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    from top_selection_dsa_gb300 import dcp as d
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(0)                         # the same rows on every rank
    T, S, k, inter = 6, 900, 50, 16
    lg = np.round(rng.standard_normal((T, S)), 1).astype(np.float32)
    L = rng.integers(1, S + 1, T).astype(np.int32)
    pos = d.owned_positions(S, rank, world, inter).numpy()
    loc = lg[:, pos]
    ln = np.array([d.local_len(int(x), rank, world, inter) for x in L], np.int32)
    top = oracle.topk(loc, np.zeros(T, np.int32), ln, k)     # local selection (oracle)
    sc = np.where(top >= 0, np.take_along_axis(loc, np.maximum(top, 0), 1), -np.inf)
    gc = d.local_to_global(torch.from_numpy(top), rank, world, inter)
    all_s, all_c = d.gather_candidates(torch.from_numpy(sc.astype(np.float32)), gc)
    assert tuple(all_s.shape) == (world, T, k) and tuple(all_c.shape) == (world, T, k)
    assert torch.equal(all_c[rank], gc)                     # rank-major: this rank's block
    flat_s = all_s.permute(1, 0, 2).reshape(T, world * k)   # row t: every rank's candidates
    flat_c = all_c.permute(1, 0, 2).reshape(T, world * k)
    merged = oracle.topk_merge(flat_s.numpy(), flat_c.numpy(), k)
    out[rank] = bool(np.array_equal(merged, oracle.topk(lg, np.zeros(T, np.int32), L, k)))
    dist.destroy_process_group()


def test_two_rank_exchange_gives_the_global_topk():
    world = 2
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] and out[1]
