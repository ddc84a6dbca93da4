"""bench.py's vocabulary-split mode (--path distributed) on CPU ranks over
gloo, with the oracle as the local backend: each rank holds its part of the
shards of one shared batch, the step runs the exchange as written (folded
partials all-gathered, target logits all-reduced), and rank 0's line reports
the loss of the whole batch, the pages' 12 bytes per token on the wire, and
the slowest rank's time."""
import argparse
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _args():
    return argparse.Namespace(workload="tiny_s64_v1000", rows=0, steps=2, warmup=3, max_buffers=4, e2e_steps=1)


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    from _dist_backend import OracleBackend

    lines = []
    bench.run_distributed(_args(), backend=OracleBackend(), device="cpu", emit=lines.append)
    q.put((rank, lines))


def _run(world):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    return got


@pytest.mark.parametrize("world", [1, 2])
def test_distributed_bench_mode_on_gloo(world):
    from oracle import vpce_oracle as O

    sys.path.insert(0, ROOT)
    from vocab_sharded_lm_gb300 import synth

    got = _run(world)
    # rank 0 alone prints its line
    assert len(got[0]) == 1 and all(got[r] == [] for r in range(1, world))
    out = json.loads(got[0][0])
    w = synth.WORKLOADS["tiny_s64_v1000"]
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    z = O.assemble(synth.shards_host(w, meta, vs), vs, w.dtype)
    ref = O.cross_entropy(z, meta.targets, w.ignore_index)
    assert out["n_gpus"] == world and out["scaling"] == "strong" and out["steps"] == 2
    # the batch is shared: tokens/s counts each of its rows once
    assert out["value"] == pytest.approx(w.s * 2 / (out["ms_per_step"] * 2e-3), rel=1e-3)
    assert out["exchange"]["bytes_per_token"] == 12
    assert out["exchange"]["bytes_sent_per_rank"] == (12 * w.s if world > 1 else 0)
    # the loss of the last timed step: the whole batch's, on the oracle's logits
    # (the step before restored them from the generated copy)
    np.testing.assert_allclose(out["loss"], ref["loss"], rtol=1e-12)
    assert out["gpu_launches"] == 0 and out["e2e"]["h2d_bytes_per_step"] == 0


def test_distributed_bench_mode_rejects_uneven_split():
    # 2 shards cannot split over 3 processes: one 'unavailable' line, exit 0
    got = _run(3)
    out = json.loads(got[0][0])
    assert "unavailable" in out and all(got[r] == [] for r in (1, 2))
