"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on seeded inputs.  Every workload runs with its full
vocabulary (rows reduced so the oracle finishes in seconds) at every shard
count t in {1, 2, 4, 8, 16} that divides V; each shard row spans several
6 KB pipeline chunks and ends in a partial one.  Edge cases: ragged and
unaligned shards, padded row strides, column views of one big tensor, empty
and all-ignored batches, out-of-range targets, reductions, determinism."""
import math

import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

from _parity import check_dlogits, check_full, check_loss, from_device, run_full, to_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def test_tiny_workload_whole_batch():
    check_full(run_full(W["tiny_s64_v1000"]))


@pytest.mark.parametrize("name", list(W))
@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_every_workload_every_t(name, t):
    w = W[name]
    if w.V % t:
        pytest.skip("t does not divide V")
    s = min(w.s, 40 if w.V > 100000 else 64)
    check_full(run_full(w, t=t, s=s))


@pytest.mark.parametrize("widths", [[1, 7, 500, 12577], [3, 1, 1, 2], [12577], [1] * 64])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_ragged_shard_widths(widths, dtype):
    vs = [0]
    for x in widths:
        vs.append(vs[-1] + x)
    w = synth.Workload("ragged", 9, 24, vs[-1], len(widths), dtype, 2.0, "uniform", ignore_frac=0.1)
    check_full(run_full(w, vocab_start=vs))


@pytest.mark.parametrize("t", [33, 64])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("path", ["split", "fused"])
def test_many_shards_many_rows(t, dtype, path):
    """Thousands of rows over 33 or 64 shards of uneven widths: every row's
    partials arrive from many warps at once (the forward combines a row in
    the warp that adds its last partial), and more than 32 partials per row
    take the combine's second load per lane.  Widths are multiples of 8
    elements, so the fused kernel runs too."""
    rng = np.random.default_rng(1000 + t)
    widths = (rng.integers(1, 26, size=t) * 8).tolist()
    vs = [0]
    for x in widths:
        vs.append(vs[-1] + x)
    w = synth.Workload("many", 12, 3000, vs[-1], t, dtype, 2.5, "uniform", ignore_frac=0.05)
    check_full(run_full(w, vocab_start=vs, path=path))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("misalign", [1, 3])
def test_unaligned_shard_pointers(dtype, misalign):
    w = synth.Workload("unaligned", 10, 20, 20011, 3, dtype, 3.0, "uniform")
    check_full(run_full(w, misalign=misalign))


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_padded_row_stride(dtype):
    # odd row stride: every row starts at a different offset from a 16-byte line
    w = synth.Workload("padded", 11, 33, 3 * 4001, 3, dtype, 2.0, "uniform", ignore_frac=0.1)
    check_full(run_full(w, ld=4001 + 5))


def test_column_views_of_one_tensor():
    w = W["s4096_v50304"].replace(s=48)
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    full_host = synth.shards_host(w, meta, [0, w.V])[0]
    big = to_device([full_host], w.dtype)[0]
    views = [big[:, vs[i]:vs[i + 1]] for i in range(w.t)]
    y = torch.from_numpy(meta.targets).cuda()
    loss, ws = vpce.vpce_forward(views, y, vs)
    z = O.assemble([full_host], [0, w.V], w.dtype)
    ref = O.cross_entropy(z, meta.targets)
    check_loss(float(loss), ref["loss"])
    vpce.vpce_backward(views, y, ws, vs)
    got = O.widen(from_device(big, w.dtype), w.dtype)
    check_dlogits(got, O.dlogits(z, meta.targets), w.dtype, 1.0 / ref["n_valid"])


@pytest.mark.parametrize("reduction,grad", [("sum", 0.5), ("mean", 2.5), ("mean", 0.0)])
def test_reductions_and_grad(reduction, grad):
    w = W["s16384_v152064"].replace(s=32)
    check_full(run_full(w, reduction=reduction, grad=grad))


def test_single_row_and_empty_batch():
    w = W["s8192_v128256"].replace(s=1)
    check_full(run_full(w))
    # s = 0: loss is NaN (mean) / 0 (sum), backward is a no-op
    dev = [torch.empty((0, 10), dtype=torch.float32, device="cuda") for _ in range(2)]
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    loss, ws = vpce.vpce_forward(dev, y, [0, 10, 20])
    assert math.isnan(float(loss))
    loss, ws = vpce.vpce_forward(dev, y, [0, 10, 20], reduction="sum")
    assert float(loss) == 0.0
    vpce.vpce_backward(dev, y, ws, [0, 10, 20])
    torch.cuda.synchronize()


def test_all_rows_ignored():
    w = W["s4096_v50304"].replace(s=16)
    res = run_full(w, targets=np.full(16, -100))
    assert math.isnan(res["loss"])
    check_full(res)


def test_out_of_range_target_sets_flag_and_nan():
    w = W["tiny_s64_v1000"]
    y = synth.row_meta(w).targets.copy()
    y[5] = 1000
    y[9] = -3
    res = run_full(w, targets=y)
    assert res["flag"] & vpce.VPCE_FLAG_BAD_TARGET
    assert math.isnan(res["loss"]) and math.isnan(res["row_loss"][5]) and math.isnan(res["row_loss"][9])
    check_full(res)
    # a clean forward afterwards clears the flag in the same workspace
    res2 = run_full(w)
    assert res2["flag"] == 0


def test_max_shift_on_gpu_fp32():
    # fp32 logits on a 1/1024 grid are exactly shiftable by 1000
    rng = np.random.default_rng(3)
    s, V, t = 16, 4096, 4
    z = (rng.integers(-8192, 8192, size=(s, V)) / 1024.0).astype(np.float32)
    y = rng.integers(0, V, size=s)
    vs = synth.even_vocab_start(V, t)
    losses = []
    for c in (0.0, 1000.0):
        host = [np.ascontiguousarray(z[:, vs[i]:vs[i + 1]] + np.float32(c)) for i in range(t)]
        dev = to_device(host, "fp32")
        rl = torch.empty(s, dtype=torch.float32, device="cuda")
        loss, ws = vpce.vpce_forward(dev, torch.from_numpy(y).cuda(), vs, row_loss_out=rl)
        losses.append(rl.cpu().numpy().astype(np.float64))
    ref = O.cross_entropy(z.astype(np.float64), y, reduction="none")["row_loss"]
    for l in losses:
        np.testing.assert_allclose(l, ref, rtol=1e-5)


def test_uniform_logits_closed_form_on_gpu():
    s, V, t = 8, 128256, 8
    vs = synth.even_vocab_start(V, t)
    host = [np.full((s, vs[i + 1] - vs[i]), 0x4040, dtype=np.uint16) for i in range(t)]  # bf16 3.0
    dev = to_device(host, "bf16")
    y = torch.arange(s, dtype=torch.int64, device="cuda") * 1000
    loss, ws = vpce.vpce_forward(dev, y, vs)
    assert float(loss) == pytest.approx(math.log(V), rel=1e-5)
    vpce.vpce_backward(dev, y, ws, vs)
    got = O.assemble([from_device(d, "bf16") for d in dev], vs, "bf16")
    expect = np.full((s, V), 1.0 / V)
    expect[np.arange(s), np.arange(s) * 1000] -= 1.0
    check_dlogits(got, expect / s, "bf16", 1.0 / s)


def test_deterministic_and_t_invariant():
    w = W["s8192_v128256"].replace(s=48)
    a = run_full(w, t=8)
    b = run_full(w, t=8)
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(a["row_loss"], b["row_loss"])
    for x, y in zip(a["back"], b["back"]):
        np.testing.assert_array_equal(x, y)
    c = run_full(w, t=2)
    assert abs(c["loss"] - a["loss"]) <= 1e-6 * abs(a["loss"])
