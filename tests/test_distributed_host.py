"""The multi-process vocabulary-parallel path (distributed.forward /
backward) on two gloo ranks on CPU, with the oracle as the local backend:
each rank holds two shards of a vocabulary of 1000, the ranks exchange only
the per-row partials and target logits, and the loss, row losses and
every rank's dlogits must equal the unsharded fp64 definition."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

V, S = 1000, 64
SPLIT = [[0, 150, 400], [400, 700, 1000]]  # rank r's shards: columns SPLIT[r][i] .. SPLIT[r][i+1]


def _problem():
    rng = np.random.default_rng(21)
    z = rng.normal(0.0, 3.0, size=(S, V))
    y = rng.integers(0, V, size=S)
    y[[3, 17]] = -100
    y[5] = 150    # a shard edge
    y[6] = 399
    y[7] = 400    # the other rank's first column
    return z, y


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, reduction, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2")
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch
    import torch.distributed as dist

    from _dist_backend import OracleBackend
    from vocab_sharded_lm_gb300 import distributed

    dist.init_process_group("gloo", rank=rank, world_size=2)
    try:
        z, y = _problem()
        vs = SPLIT[rank]
        shards = [torch.tensor(z[:, vs[i]:vs[i + 1]].copy()) for i in range(len(vs) - 1)]
        targets = torch.tensor(y)
        be = OracleBackend()
        loss, row_loss, ws = distributed.forward(shards, vs, targets, V, reduction=reduction, backend=be)
        distributed.backward(shards, vs, targets, ws, grad_output=2.0, backend=be)
        q.put((rank, np.asarray(loss.numpy()), row_loss.numpy(), [sh.numpy() for sh in shards]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_two_ranks_match_unsharded(reduction):
    from oracle import vpce_oracle as O

    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, port, reduction, q)) for r in range(2)]
    for p in procs:
        p.start()
    # read the results before joining: a child that queued a large array
    # exits only once the queue has been drained
    out = {r: (loss, rl, d) for r, loss, rl, d in (q.get(timeout=180) for _ in range(2))}
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    z, y = _problem()
    ref = O.cross_entropy(z, y, reduction=reduction)
    dref = O.dlogits(z, y, grad=2.0, reduction=reduction)
    for r in range(2):
        loss, rl, d = out[r]
        # every rank computes the same loss and row losses, equal to the unsharded definition
        np.testing.assert_allclose(loss, ref["loss"], rtol=1e-12)
        np.testing.assert_allclose(rl, ref["row_loss"], rtol=1e-12, atol=1e-12)
        vs = SPLIT[r]
        for i, di in enumerate(d):
            np.testing.assert_allclose(di, dref[:, vs[i]:vs[i + 1]], rtol=1e-10, atol=1e-15)
    np.testing.assert_array_equal(out[0][1], out[1][1])
