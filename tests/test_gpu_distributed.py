"""GPU parity of the local steps of the multi-process path (vpce_partials,
vpce_fold_partials, vpce_combine_partials, vpce_backward on one process's
part of the vocabulary), with two ranks played in one process: the exchange
is done here (concatenate each rank's folded pairs in rank order, sum the
target logits), as the collectives would; no kernel waits on another."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import distributed, synth, vpce

from _parity import check_dlogits, check_loss, check_row_losses, from_device, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


@pytest.mark.parametrize("name,s,split", [
    ("s8192_v128256", 48, [[0, 16032, 32064, 48096, 64128], [64128, 80160, 96192, 112224, 128256]]),
    ("s4096_v50304", 64, [[0, 12576, 25152], [25152, 37728, 50304]]),
])
def test_two_ranks_in_one_process(name, s, split):
    w = synth.WORKLOADS[name].replace(s=s)
    vs_all = sorted(set(split[0]) | set(split[1]))
    meta = synth.row_meta(w)
    host = synth.shards_host(w, meta, vs_all)
    z = O.assemble(host, vs_all, w.dtype)
    ref = O.cross_entropy(z, meta.targets, w.ignore_index)
    dref = O.dlogits(z, meta.targets, w.ignore_index, grad=1.0)
    y = torch.from_numpy(meta.targets).cuda()
    be = distributed.CudaBackend()
    per_rank = []
    for vs in split:
        idx = [vs_all.index(v) for v in vs[:-1]]
        dev = to_device([host[i] for i in idx], w.dtype)
        ws = be.new_workspace(len(dev), s, "cuda")
        part, tgt = be.partials(dev, vs, y, w.ignore_index, ws)
        per_rank.append((vs, dev, ws, part, tgt))
    folded = [be.fold(r[3]) for r in per_rank]
    # one (max, sum exp) pair per row and rank: what the all-gather moves
    assert all(f.shape == (1, s, 2) for f in folded)
    ref_fold = [O.fold_partials(r[3][:, :, 0].double().cpu().numpy(), r[3][:, :, 1].double().cpu().numpy())
                for r in per_rank]
    for f, (M, S) in zip(folded, ref_fold):
        np.testing.assert_array_equal(f[0, :, 0].cpu().numpy(), M.astype(np.float32))
        np.testing.assert_allclose(f[0, :, 1].double().cpu().numpy(), S, rtol=1e-5)
    gathered = torch.cat(folded, dim=0)
    tgt_sum = per_rank[0][4] + per_rank[1][4]
    losses = []
    for vs, dev, ws, part, tgt in per_rank:
        loss, row_loss = be.combine(gathered, tgt_sum, w.V, y, w.ignore_index, "mean", len(dev), ws)
        losses.append((float(loss), row_loss.cpu().numpy()))
        be.backward(dev, vs, y, w.ignore_index, ws, 1.0)
        torch.cuda.synchronize()
        got = O.assemble([from_device(d, w.dtype) for d in dev], [0] + list(np.cumsum(np.diff(vs))), w.dtype)
        check_dlogits(got, dref[:, vs[0]:vs[-1]], w.dtype, 1.0 / ref["n_valid"])
    for loss, rl in losses:
        check_loss(loss, ref["loss"])
        check_row_losses(rl, ref["row_loss"], ref["valid"])
    assert losses[0][0] == losses[1][0]
    np.testing.assert_array_equal(losses[0][1], losses[1][1])


def test_distributed_forward_backward_through_nccl_group_of_one():
    """distributed.forward / backward end to end on the GPU: the library's
    kernels for the local steps and NCCL for the exchange, in a process
    group of one (this run has one GPU), checked against the oracle."""
    import os
    import socket

    import torch.distributed as dist

    w = synth.WORKLOADS["s8192_v128256"].replace(s=64)
    vs = synth.even_vocab_start(w.V, w.t)
    meta = synth.row_meta(w)
    host = synth.shards_host(w, meta, vs)
    z = O.assemble(host, vs, w.dtype)
    ref = O.cross_entropy(z, meta.targets, w.ignore_index)
    dref = O.dlogits(z, meta.targets, w.ignore_index, grad=1.0)
    own = not dist.is_initialized()
    if own:
        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        dev = to_device(host, w.dtype)
        y = torch.from_numpy(meta.targets).cuda()
        loss, row_loss, ws = distributed.forward(dev, vs, y, w.V, ignore_index=w.ignore_index)
        distributed.backward(dev, vs, y, ws, ignore_index=w.ignore_index)
        torch.cuda.synchronize()
        check_loss(float(loss), ref["loss"])
        check_row_losses(row_loss.cpu().numpy(), ref["row_loss"], ref["valid"])
        got = O.assemble([from_device(d, w.dtype) for d in dev], vs, w.dtype)
        check_dlogits(got, dref, w.dtype, 1.0 / ref["n_valid"])
    finally:
        if own:
            dist.destroy_process_group()
