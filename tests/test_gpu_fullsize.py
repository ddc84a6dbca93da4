"""Full-size workloads, in the launch configuration the benchmark times: the
device generator fills every shard, the CUDA path runs on the whole batch
(the two-call path, and the one-call fused path that the benchmark times, on
its persistent grid with tens of rows per CTA), and the oracle checks sampled
rows one by one (per-row loss and every element of those rows' dlogits),
plus properties that hold at any size (the reduced loss is the fp64 mean of
the per-row losses; ignored rows are exactly zero).

The oracle is fed the logits the kernels saw: the sampled rows are read back
from the device before the in-place call overwrites them.  A separate check
compares those bytes with the host generator's."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

from _parity import LOSS_RTOL, check_dlogits, from_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
LONG = ["s8192_v128256", "s16384_v152064", "s32768_v256000"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _sample_rows(w, meta, k=10):
    rng = np.random.default_rng(w.seed)
    rows = {0, 1, w.s - 2, w.s - 1}
    rows.update(int(r) for r in rng.choice(w.s, size=k, replace=False))
    boosted = np.nonzero(meta.boost_col >= 0)[0]
    if boosted.size:
        rows.add(int(boosted[0]))
    ign = np.nonzero(meta.targets == w.ignore_index)[0]
    if ign.size:
        rows.add(int(ign[0]))
    # rows in the middle and at the end of a CTA's walk on the persistent
    # grid (one row per CTA at a time: rows b, b + grid, ...)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for r in (sms - 1, sms, 2 * sms + 3, w.s - sms):
        if 0 <= r < w.s:
            rows.add(r)
    return np.array(sorted(rows))


def _rows_of(dev, rows, dtype):
    idx = torch.from_numpy(rows).cuda()
    return [from_device(d.index_select(0, idx), dtype) for d in dev]


def _run_sampled(w, path):
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    dev = synth.device_shards(w, meta, vs)
    rows = _sample_rows(w, meta)

    # the oracle's input: the bytes the kernels will read
    got_rows = _rows_of(dev, rows, w.dtype)
    # the device generator drew the same logits as the host generator (its
    # float64 log / cos may differ in the last bit, so a stored value may
    # rarely differ by one ulp)
    host_rows = [synth.logits_rows(w, rows, vs[i], vs[i + 1], meta) for i in range(w.t)]
    for h, g in zip(host_rows, got_rows):
        hb = h.view(np.uint16).astype(np.int64) if w.dtype == "bf16" else h.view(np.int32).astype(np.int64)
        gb = g.view(np.uint16).astype(np.int64) if w.dtype == "bf16" else g.view(np.int32).astype(np.int64)
        assert np.count_nonzero(hb != gb) <= 2 and np.abs(hb - gb).max() <= 1

    z = O.assemble(got_rows, vs, w.dtype)
    y_all = meta.targets
    n_valid = int(np.sum(y_all != w.ignore_index))
    ref = O.cross_entropy(z, y_all[rows], w.ignore_index, n_valid=n_valid)
    dref = O.dlogits(z, y_all[rows], w.ignore_index, n_valid=n_valid)

    y = torch.from_numpy(y_all).cuda()
    row_loss = torch.empty(w.s, dtype=torch.float32, device="cuda")
    if path == "split":
        loss, ws = vpce.vpce_forward(dev, y, vs, ignore_index=w.ignore_index, row_loss_out=row_loss)
        loss_v = float(loss)
        assert vpce.vpce_read_error_flag(ws) == 0
        vpce.vpce_backward(dev, y, ws, vs, ignore_index=w.ignore_index)
    else:
        plan = vpce.vpce_fused_plan(vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32, vs, w.s)
        assert plan["kernel"] == "stream"
        # many rows per CTA (or CTA pair) on the persistent grid
        assert w.s >= 8 * (plan["grid"] // plan["cluster"])
        loss, ws = vpce.vpce_forward_backward(dev, y, vs, ignore_index=w.ignore_index, row_loss_out=row_loss)
        loss_v = float(loss)
        assert vpce.vpce_read_error_flag(ws) == 0
    rl = row_loss.cpu().numpy()

    valid = ref["valid"]
    err = np.abs(rl[rows][valid] - ref["row_loss"][valid]) / np.maximum(np.abs(ref["row_loss"][valid]), 1.0)
    assert err.max() <= LOSS_RTOL, err.max()
    mean = float(np.sum(rl.astype(np.float64)[y_all != w.ignore_index])) / n_valid
    # the batch sum runs in fp64 (two calls) or as a compensated fp32 pair
    # (fused), either well below the final rounding to fp32 (2^-24 relative);
    # a plain fp32 sum of 32768 rows would typically miss this bound
    assert abs(loss_v - mean) <= 2e-7 * abs(mean), (loss_v, mean)
    assert np.all(rl[y_all == w.ignore_index] == 0.0)
    assert np.all(np.isfinite(rl))

    back = O.assemble(_rows_of(dev, rows, w.dtype), vs, w.dtype)
    check_dlogits(back, dref, w.dtype, 1.0 / n_valid)
    # every ignored row of the whole batch is exactly zero
    ign = np.nonzero(y_all == w.ignore_index)[0]
    if ign.size:
        idx = torch.from_numpy(ign).cuda()
        for d in dev:
            assert int(torch.count_nonzero(d.index_select(0, idx))) == 0
    del dev
    torch.cuda.empty_cache()


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("name", list(W))
def test_full_size_sampled_rows(name, path):
    w = W[name]
    if path == "fused" and w.s < 8 * 152:
        pytest.skip("the persistent grid is wider than a few rows per CTA here")
    _run_sampled(w, path)


@pytest.mark.parametrize("name", LONG)
@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_full_size_fused_every_t(name, t):
    # the shard count of the workload itself is covered above
    w = W[name]
    if w.V % t or t == w.t:
        pytest.skip("t does not divide V, or is the workload's own")
    _run_sampled(w.replace(t=t), "fused")
