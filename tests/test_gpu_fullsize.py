"""Full-size workloads, in the launch configuration the benchmark times: the
device generator fills every shard, the CUDA path runs on the whole batch,
and the oracle checks sampled rows one by one (per-row loss and every element
of those rows' dlogits), plus properties that hold at any size (the reduced
loss is the fp64 mean of the per-row losses; ignored rows are exactly zero)."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

from _parity import LOSS_RTOL, check_dlogits, from_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _sample_rows(w, meta, k=10):
    rng = np.random.default_rng(w.seed)
    rows = {0, w.s - 1}
    rows.update(int(r) for r in rng.choice(w.s, size=k, replace=False))
    boosted = np.nonzero(meta.boost_col >= 0)[0]
    if boosted.size:
        rows.add(int(boosted[0]))
    ign = np.nonzero(meta.targets == w.ignore_index)[0]
    if ign.size:
        rows.add(int(ign[0]))
    return np.array(sorted(rows))


def _rows_of(dev, rows, dtype):
    idx = torch.from_numpy(rows).cuda()
    return [from_device(d.index_select(0, idx), dtype) for d in dev]


@pytest.mark.parametrize("name", list(W))
def test_full_size_sampled_rows(name):
    w = W[name]
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    dev = synth.device_shards(w, meta, vs)
    rows = _sample_rows(w, meta)

    # the device generator drew the same logits as the host generator
    host_rows = [synth.logits_rows(w, rows, vs[i], vs[i + 1], meta) for i in range(w.t)]
    got_rows = _rows_of(dev, rows, w.dtype)
    for h, g in zip(host_rows, got_rows):
        hb = h.view(np.uint16).astype(np.int64) if w.dtype == "bf16" else h.view(np.int32).astype(np.int64)
        gb = g.view(np.uint16).astype(np.int64) if w.dtype == "bf16" else g.view(np.int32).astype(np.int64)
        assert np.count_nonzero(hb != gb) <= 2 and np.abs(hb - gb).max() <= 1

    z = O.assemble(host_rows, vs, w.dtype)
    y_all = meta.targets
    n_valid = int(np.sum(y_all != w.ignore_index))
    ref = O.cross_entropy(z, y_all[rows], w.ignore_index, n_valid=n_valid)
    dref = O.dlogits(z, y_all[rows], w.ignore_index, n_valid=n_valid)

    y = torch.from_numpy(y_all).cuda()
    row_loss = torch.empty(w.s, dtype=torch.float32, device="cuda")
    loss, ws = vpce.vpce_forward(dev, y, vs, ignore_index=w.ignore_index, row_loss_out=row_loss)
    rl = row_loss.cpu().numpy()
    loss_v = float(loss)
    assert vpce.vpce_read_error_flag(ws) == 0

    valid = ref["valid"]
    err = np.abs(rl[rows][valid] - ref["row_loss"][valid]) / np.maximum(np.abs(ref["row_loss"][valid]), 1.0)
    assert err.max() <= LOSS_RTOL, err.max()
    mean = float(np.sum(rl.astype(np.float64)[y_all != w.ignore_index])) / n_valid
    assert abs(loss_v - mean) <= 1e-6 * abs(mean)
    assert np.all(rl[y_all == w.ignore_index] == 0.0)

    vpce.vpce_backward(dev, y, ws, vs, ignore_index=w.ignore_index)
    back = O.assemble(_rows_of(dev, rows, w.dtype), vs, w.dtype)
    check_dlogits(back, dref, w.dtype, 1.0 / n_valid)
    del dev
    torch.cuda.empty_cache()
