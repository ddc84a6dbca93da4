"""GPU parity of vpce_forward_backward (loss and in-place dlogits in one call)
against the fp64 oracle, element by element: every workload at every shard
count that divides V, reductions, ignored and bad targets, the fallback for
rows that are not 16-byte aligned, and agreement with the two-call path."""
import math

import numpy as np
import pytest
import torch

from vocab_sharded_lm_gb300 import synth, vpce

from _parity import check_full, run_full

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


@pytest.mark.parametrize("name", list(W))
@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_fused_every_workload_every_t(name, t):
    w = W[name]
    if w.V % t:
        pytest.skip("t does not divide V")
    s = min(w.s, 40 if w.V > 100000 else 64)
    check_full(run_full(w, t=t, s=s, path="fused"))


def test_fused_more_rows_than_blocks():
    # several rows per row group, ignored rows interleaved
    check_full(run_full(W["s4096_v50304"].replace(s=700), path="fused"))


@pytest.mark.parametrize("wl", ["s16384_v152064", "s8192_v128256"])
@pytest.mark.parametrize("reduction,grad", [("sum", 0.5), ("mean", 2.5), ("mean", 0.0), ("sum", -1.5)])
def test_fused_reductions(reduction, grad, wl):
    # fp32 and bf16 rows; a gradient of 0 or below cannot be folded into the
    # exponent and takes the explicit product
    check_full(run_full(W[wl].replace(s=48), reduction=reduction, grad=grad, path="fused"))


@pytest.mark.parametrize("widths", [[8, 8, 16], [16, 1024, 8000, 24], [4] * 64])
def test_fused_narrow_aligned_shards(widths):
    # 16-byte multiples, some narrower than a warp's share of a row
    vs = [0]
    for x in widths:
        vs.append(vs[-1] + x)
    w = synth.Workload("narrow", 12, 40, vs[-1], len(widths), "fp32", 2.0, "uniform", ignore_frac=0.1)
    check_full(run_full(w, vocab_start=vs, path="fused"))


@pytest.mark.parametrize("kw", [dict(misalign=1), dict(ld=4001 + 5)])
def test_fused_unaligned_rows_fall_back(kw):
    w = synth.Workload("fallback", 13, 24, 3 * 4001, 3, "bf16", 2.0, "uniform", ignore_frac=0.1)
    check_full(run_full(w, path="fused", **kw))


def test_fused_bad_and_all_ignored_targets():
    w = W["tiny_s64_v1000"]
    y = synth.row_meta(w).targets.copy()
    y[3] = 5000
    res = run_full(w, targets=y, path="fused")
    assert res["flag"] & vpce.VPCE_FLAG_BAD_TARGET and math.isnan(res["loss"])
    check_full(res)
    res = run_full(W["s4096_v50304"].replace(s=20), targets=np.full(20, -100), path="fused")
    assert math.isnan(res["loss"])
    check_full(res)


def test_fused_empty_batch():
    dev = [torch.empty((0, 16), dtype=torch.float32, device="cuda") for _ in range(2)]
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    loss, _ = vpce.vpce_forward_backward(dev, y, [0, 16, 32])
    assert math.isnan(float(loss))
    loss, _ = vpce.vpce_forward_backward(dev, y, [0, 16, 32], reduction="sum")
    assert float(loss) == 0.0


def test_fused_matches_split_and_is_deterministic():
    w = W["s8192_v128256"].replace(s=96)
    a = run_full(w, path="fused")
    b = run_full(w, path="fused")
    c = run_full(w, path="split")
    assert a["loss"] == b["loss"]
    for x, y in zip(a["back"], b["back"]):
        np.testing.assert_array_equal(x, y)
    assert abs(a["loss"] - c["loss"]) <= 1e-6 * abs(c["loss"])
    np.testing.assert_allclose(a["row_loss"], c["row_loss"], rtol=2e-6)


def test_fused_long_rows():
    # 2 MB fp32 rows: every stats warp walks several chunks per shard segment
    w = synth.Workload("longrows", 14, 6, 500000, 4, "fp32", 2.0, "uniform")
    check_full(run_full(w, path="fused"))


@pytest.mark.parametrize("name", list(W))
def test_fused_plan(name):
    w = W[name]
    vs = synth.even_vocab_start(w.V, w.t)
    plan = vpce.vpce_fused_plan(vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32, vs, w.s)
    assert plan["kernel"] == "stream" and 0 < plan["grid"] <= w.s
    # rows over 224 KB are shared by a pair of CTAs (a cluster of 2)
    row_bytes = w.V * (2 if w.dtype == "bf16" else 4)
    assert plan["cluster"] == (2 if row_bytes > 224 * 1024 else 1)
    assert plan["grid"] % plan["cluster"] == 0
    odd = [0, 3, 10]  # a 3-column bf16 shard is not a 16-byte multiple
    assert vpce.vpce_fused_plan(vpce.VPCE_BF16, odd, 4)["kernel"] == "split"


def test_fused_paired_rows_match_split_and_are_deterministic():
    # 512 KB rows: two CTAs of a cluster share each row
    w = W["s32768_v256000"].replace(s=100)
    assert vpce.vpce_fused_plan(vpce.VPCE_BF16, synth.even_vocab_start(w.V, w.t), w.s)["cluster"] == 2
    a = run_full(w, path="fused")
    b = run_full(w, path="fused")
    c = run_full(w, path="split")
    check_full(a)
    assert a["loss"] == b["loss"]
    for x, y in zip(a["back"], b["back"]):
        np.testing.assert_array_equal(x, y)
    assert abs(a["loss"] - c["loss"]) <= 1e-6 * abs(c["loss"])
    np.testing.assert_allclose(a["row_loss"], c["row_loss"], rtol=2e-6)


@pytest.mark.parametrize("vs", [[0, 200000], [0, 8, 180000, 180016, 200000], [0, 190000, 190008, 200000]])
def test_fused_paired_rows_uneven_shards(vs):
    # 400 KB bf16 rows: one shard split over 16 warps; uneven shards split at
    # the boundary nearest half the row (the halves differ in size)
    w = synth.Workload("paired", 15, 36, vs[-1], len(vs) - 1, "bf16", 2.0, "uniform", ignore_frac=0.1)
    assert vpce.vpce_fused_plan(vpce.VPCE_BF16, vs, w.s)["cluster"] == 2
    check_full(run_full(w, vocab_start=vs, path="fused"))


@pytest.mark.parametrize("name", ["s8192_v128256", "s16384_v152064", "s32768_v256000"])
@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_fused_several_rows_per_cta(name, t):
    # the persistent grid at its full width with three or four rows per CTA
    # (or CTA pair), so that the credit flow carries the stats pass across
    # row boundaries at the workload's own row length; every element is
    # checked against the oracle
    w = W[name]
    if w.V % t:
        pytest.skip("t does not divide V")
    vs = synth.even_vocab_start(w.V, t)
    dt = vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32
    plan = vpce.vpce_fused_plan(dt, vs, w.s)
    units = plan["grid"] // plan["cluster"]
    s = 3 * units + 7
    assert vpce.vpce_fused_plan(dt, vs, s)["grid"] == plan["grid"]
    check_full(run_full(w, t=t, s=s, path="fused"))


@pytest.mark.parametrize("name,t", [("s8192_v128256", 8), ("s8192_v128256", 1), ("s16384_v152064", 8),
                                    ("s32768_v256000", 16)])
def test_fused_pair_targets_at_part_edges(name, t):
    # CTA pairs: the target logit crosses to the other CTA of the pair only
    # when that CTA's half of the row holds it, and the receiving row barrier
    # then waits for 4 more bytes.  Targets on both sides of the split, at
    # shard edges, at the row ends, bad and ignored, in changing order over
    # three or four rows per pair (so every mailbox slot is reused)
    w = W[name]
    vs = synth.even_vocab_start(w.V, t)
    dt = vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32
    eb = 2 if w.dtype == "bf16" else 4
    plan = vpce.vpce_fused_plan(dt, vs, w.s)
    assert plan["cluster"] == 2
    if t >= 2:  # the shard boundary nearest half the row
        mid = vs[min(range(1, t), key=lambda i: abs(2 * vs[i] - vs[t]))]
    else:  # half the row's bytes, rounded down to 16 bytes
        mid = ((w.V * eb // 2) & ~15) // eb
    edges = sorted({0, 1, mid - 1, mid, mid + 1, w.V - 2, w.V - 1, vs[1] - 1, min(vs[1], w.V - 1)})
    pattern = edges + [w.V, w.ignore_index] + edges[::-1] + [-5]
    units = plan["grid"] // plan["cluster"]
    s = 3 * units + 11
    y = np.random.default_rng(5).permutation(np.resize(np.array(pattern, dtype=np.int64), s))
    res = run_full(w, t=t, s=s, targets=y, path="fused")
    assert res["flag"] & vpce.VPCE_FLAG_BAD_TARGET and not res["flag"] & vpce.VPCE_FLAG_WAIT_TIMEOUT
    check_full(res)
