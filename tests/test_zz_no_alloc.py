"""vpce_forward_static: the forward for callers that cannot allocate device
memory (a plugin inside a framework whose pooling allocator owns the GPU's
memory, a path that cannot take cudaMalloc's implicit synchronisation, or a
deployment that forbids allocation after start-up).  Its scratch is a fixed
array inside the library instead of a caller workspace.  This file is
collected last so that a failure here never hides the other tests; it runs
the same way alone in a fresh process.

Checks, through the C ABI: two calls in a row, each on different inputs,
match the workspace entry point within the parity tests' loss tolerance; a
problem larger than the static scratch is refused before anything runs.
"""
import ctypes

import numpy as np
import pytest
import torch

from vocab_sharded_lm_gb300 import synth, vpce

from _parity import LOSS_RTOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _inputs(w):
    meta = synth.row_meta(w)
    vs = synth.even_vocab_start(w.V, w.t)
    dev = to_device(synth.shards_host(w, meta, vs), w.dtype)
    return dev, torch.from_numpy(meta.targets).cuda(), vs


def _static(dev, y, vs, w, reduction=vpce.VPCE_MEAN):
    loss = torch.full((), -1.0, dtype=torch.float32, device="cuda")
    rl = torch.full((w.s,), -1.0, dtype=torch.float32, device="cuda")
    code = vpce.forward_static_raw([d.data_ptr() for d in dev], vpce.VPCE_BF16 if w.dtype == "bf16" else vpce.VPCE_FP32,
                                   len(dev), w.s, vs, 0, ctypes.c_void_p(y.data_ptr()), w.ignore_index, reduction,
                                   ctypes.c_void_p(loss.data_ptr()), ctypes.c_void_p(rl.data_ptr()),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == vpce.VPCE_OK, vpce.vpce_status_string(code)
    return loss, rl


def _with_workspace(dev, y, vs, w, reduction="mean"):
    rl = torch.empty(w.s, dtype=torch.float32, device="cuda")
    loss, _ = vpce.vpce_forward(dev, y, vs, ignore_index=w.ignore_index, reduction=reduction, row_loss_out=rl)
    return loss, rl


def _close(a, b):
    a = np.asarray(a.cpu(), dtype=np.float64)
    b = np.asarray(b.cpu(), dtype=np.float64)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    ok = ~np.isnan(a)
    assert np.all(np.abs(a[ok] - b[ok]) <= LOSS_RTOL * np.maximum(np.abs(b[ok]), 1.0))


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    w1 = synth.WORKLOADS["s4096_v50304"].replace(s=300)        # bf16, t = 4, ignored rows
    w2 = synth.WORKLOADS["s16384_v152064"].replace(s=200)      # fp32, t = 8, spikes, ignored rows
    d1, y1, vs1 = _inputs(w1)
    d2, y2, vs2 = _inputs(w2)
    ref1 = _with_workspace(d1, y1, vs1, w1)
    ref2 = _with_workspace(d2, y2, vs2, w2, "sum")
    got1 = _static(d1, y1, vs1, w1)
    got2 = _static(d2, y2, vs2, w2, vpce.VPCE_SUM)   # reuses the scratch the first call left behind
    torch.cuda.synchronize()
    for got, ref in ((got1, ref1), (got2, ref2)):
        _close(got[0], ref[0])
        _close(got[1], ref[1])
    # and once more on the first inputs, after the second call
    again = _static(d1, y1, vs1, w1)
    _close(again[0], ref1[0])
    _close(again[1], ref1[1])


def test_too_large_for_the_static_scratch_is_refused():
    big_s = vpce.VPCE_STATIC_SCRATCH_BYTES // 8  # 8 bytes per (shard, row) alone exceed it at t = 1
    code = vpce.forward_static_raw([0x7F0000000000], vpce.VPCE_FP32, 1, big_s, [0, 16], 0,
                                   ctypes.c_void_p(0x7F0000000000), -100, vpce.VPCE_MEAN,
                                   ctypes.c_void_p(0x7F0000000000), None, None)
    assert code == 4  # VPCE_ERR_WORKSPACE, nothing launched
