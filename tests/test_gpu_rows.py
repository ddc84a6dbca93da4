"""GPU parity of reduction 'none' and of the per-row backward
(vpce_backward_rows, vpce_forward_backward_rows) against the fp64 oracle,
element by element: per-row upstream gradients of both signs, zeros and NaN,
ignored rows, both paths, the fallback for unaligned rows, and bitwise
agreement with the scalar entry points when every row gets the same scale."""
import numpy as np
import pytest
import torch

from vocab_sharded_lm_gb300 import synth, vpce

from _parity import check_full, run_full, to_device, from_device

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _grad_rows(s, seed, nan_rows=()):
    g = np.random.default_rng(seed).normal(0.0, 1.0, size=s).astype(np.float32)
    g[::7] = 0.0
    g[1::5] *= -3.0
    for r in nan_rows:
        g[r] = np.nan
    return g


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("name,s", [("s4096_v50304", 64), ("s16384_v152064", 24), ("s8192_v128256", 40),
                                    ("tiny_s64_v1000", 64)])
def test_none_with_per_row_gradients(path, name, s):
    w = W[name].replace(s=s)
    g = _grad_rows(s, 11)
    check_full(run_full(w, reduction="none", grad_rows=g, path=path))


@pytest.mark.parametrize("path", ["split", "fused"])
def test_nan_gradient_rows(path):
    # a NaN upstream gradient poisons its own row only; on an ignored row it is never read
    w = W["s4096_v50304"].replace(s=48)
    meta = synth.row_meta(w)
    ign = np.nonzero(meta.targets == w.ignore_index)[0]
    valid = np.nonzero(meta.targets != w.ignore_index)[0]
    nan_rows = [int(valid[3])] + ([int(ign[0])] if ign.size else [])
    res = run_full(w, reduction="none", grad_rows=_grad_rows(w.s, 5, nan_rows), path=path)
    check_full(res)


@pytest.mark.parametrize("path", ["split", "fused"])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_reduced_forward_with_per_row_gradients(path, reduction):
    # the per-row backward does not depend on the forward's reduction
    w = W["s16384_v152064"].replace(s=16)
    check_full(run_full(w, reduction=reduction, grad_rows=_grad_rows(w.s, 3), path=path))


@pytest.mark.parametrize("path", ["split", "fused"])
def test_none_with_scalar_gradient(path):
    # a scalar g after 'none' applies to every row, as 'sum'
    check_full(run_full(W["s4096_v50304"].replace(s=32), reduction="none", grad=0.5, path=path))


def test_per_row_fallback_for_unaligned_rows():
    w = synth.Workload("fallback", 13, 24, 3 * 4001, 3, "bf16", 2.0, "uniform", ignore_frac=0.1)
    check_full(run_full(w, reduction="none", grad_rows=_grad_rows(w.s, 9), path="fused", misalign=1))


@pytest.mark.parametrize("path", ["split", "fused"])
def test_uniform_rows_match_scalar_mean_bitwise(path):
    """grad_rows = g / n_valid (rounded as the device rounds it) on every row
    gives the same bits as the scalar 'mean' backward."""
    w = W["s8192_v128256"].replace(s=24)
    vs = synth.even_vocab_start(w.V, w.t)
    meta = synth.row_meta(w)
    host = synth.shards_host(w, meta, vs)
    y = torch.from_numpy(meta.targets).cuda()
    n_valid = int(np.sum(meta.targets != w.ignore_index))
    g = np.float32(1.75)
    rows = torch.full((w.s,), float(np.float32(g / np.float32(n_valid))), dtype=torch.float32, device="cuda")
    outs = []
    for grad_rows in (None, rows):
        dev = to_device(host, w.dtype)
        if path == "split":
            _, ws = vpce.vpce_forward(dev, y, vs, ignore_index=w.ignore_index)
            vpce.vpce_backward(dev, y, ws, vs, ignore_index=w.ignore_index, grad_output=float(g),
                               grad_rows=grad_rows)
        else:
            vpce.vpce_forward_backward(dev, y, vs, ignore_index=w.ignore_index, grad_output=float(g),
                                       grad_rows=grad_rows)
        torch.cuda.synchronize()
        outs.append([from_device(d, w.dtype) for d in dev])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("path", ["split", "fused"])
def test_none_empty_batch(path):
    dev = [torch.empty((0, 16), dtype=torch.float32, device="cuda") for _ in range(2)]
    y = torch.empty(0, dtype=torch.int64, device="cuda")
    g = torch.empty(0, dtype=torch.float32, device="cuda")
    if path == "split":
        out, ws = vpce.vpce_forward(dev, y, [0, 16, 32], reduction="none")
        vpce.vpce_backward(dev, y, ws, [0, 16, 32], grad_rows=g)
    else:
        out, _ = vpce.vpce_forward_backward(dev, y, [0, 16, 32], reduction="none", grad_rows=g)
    torch.cuda.synchronize()
    assert out.shape == (0,)
