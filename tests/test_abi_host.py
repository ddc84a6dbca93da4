"""The C ABI without a GPU: the library builds, loads, exports every symbol the
header declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from vocab_sharded_lm_gb300 import _build, vpce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vpce.h")

FAKE = 0x7F0000000000  # a 256-byte aligned "device" address, never dereferenced on the host


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return vpce.load_library()


def _declared_functions(path):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vpce_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions(HEADER)
    assert "vpce_forward" in names and "vpce_backward" in names
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(7):
        s = vpce.vpce_status_string(code)
        assert s.startswith(vpce.STATUS_NAMES[code])


def test_workspace_bytes(lib):
    assert vpce.vpce_workspace_bytes(0, 10) == 0
    assert vpce.vpce_workspace_bytes(65, 10) == 0
    assert vpce.vpce_workspace_bytes(1, -1) == 0
    a = vpce.vpce_workspace_bytes(8, 8192)
    assert a >= 8 * 8192 * 8 + 8192 * 8 and a % 256 == 0
    assert vpce.vpce_workspace_bytes(8, 0) > 0


def _fwd(**kw):
    t = kw.get("t", 2)
    args = dict(shard_ptrs=[FAKE, FAKE + 4096][:t] + [FAKE] * max(0, t - 2), dtype=vpce.VPCE_BF16, t=t, s=4,
                vocab_start=[0, 8, 16] if t == 2 else list(range(0, 8 * (t + 1), 8)), ld=0,
                targets_ptr=ctypes.c_void_p(FAKE), ignore_index=-100, reduction=vpce.VPCE_MEAN,
                loss_ptr=ctypes.c_void_p(FAKE), row_loss_ptr=None, ws_ptr=ctypes.c_void_p(FAKE),
                ws_bytes=1 << 20, stream=None)
    args.update(kw)
    args.pop("t", None)
    return vpce.forward_raw(t=t, **args)


def _bwd(**kw):
    args = dict(shard_ptrs=[FAKE, FAKE + 4096], dtype=vpce.VPCE_FP32, t=2, s=4, vocab_start=[0, 8, 16], ld=0,
                targets_ptr=ctypes.c_void_p(FAKE), ignore_index=-100, grad=1.0, ws_ptr=ctypes.c_void_p(FAKE),
                ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return vpce.backward_raw(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=7), 3),
    (dict(t=0, shard_ptrs=[], vocab_start=[0]), 1),
    (dict(t=65, shard_ptrs=[FAKE] * 65, vocab_start=list(range(0, 66 * 8, 8))), 1),
    (dict(s=-1), 1),
    (dict(shard_ptrs=None), 1),
    (dict(shard_ptrs=[FAKE, 0]), 1),
    (dict(shard_ptrs=[FAKE + 1, FAKE]), 2),       # bf16 needs 2-byte alignment
    (dict(vocab_start=None), 1),
    (dict(vocab_start=[1, 8, 16]), 1),            # must start at 0
    (dict(vocab_start=[0, 8, 8]), 1),             # empty shard
    (dict(vocab_start=[0, 9, 8]), 1),             # decreasing
    (dict(ld=-1), 1),
    (dict(ld=7), 1),                              # narrower than a shard
    (dict(targets_ptr=None), 1),
    (dict(targets_ptr=ctypes.c_void_p(FAKE + 4)), 2),
    (dict(reduction=5), 1),
    (dict(loss_ptr=None), 1),
    (dict(loss_ptr=ctypes.c_void_p(FAKE + 2)), 2),
    (dict(ws_ptr=None), 1),
    (dict(ws_ptr=ctypes.c_void_p(FAKE + 16)), 2),
    (dict(ws_bytes=64), 4),
])
def test_forward_rejects_bad_arguments(lib, kw, code):
    assert _fwd(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), 3),
    (dict(grad=float("nan")), 1),
    (dict(grad=float("inf")), 1),
    (dict(ws_bytes=100), 4),
    (dict(shard_ptrs=[FAKE + 2, FAKE]), 2),       # fp32 needs 4-byte alignment
    (dict(vocab_start=[0, 0, 16]), 1),
])
def test_backward_rejects_bad_arguments(lib, kw, code):
    assert _bwd(**kw) == code


def _bwd_rows(**kw):
    args = dict(shard_ptrs=[FAKE, FAKE + 4096], dtype=vpce.VPCE_FP32, t=2, s=4, vocab_start=[0, 8, 16], ld=0,
                targets_ptr=ctypes.c_void_p(FAKE), ignore_index=-100, grad_rows_ptr=ctypes.c_void_p(FAKE),
                ws_ptr=ctypes.c_void_p(FAKE), ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return vpce.backward_rows_raw(**args)


def _fb_rows(**kw):
    args = dict(shard_ptrs=[FAKE, FAKE + 4096], dtype=vpce.VPCE_BF16, t=2, s=4, vocab_start=[0, 8, 16], ld=0,
                targets_ptr=ctypes.c_void_p(FAKE), ignore_index=-100, reduction=vpce.VPCE_NONE,
                grad_rows_ptr=ctypes.c_void_p(FAKE), loss_ptr=None, row_loss_ptr=ctypes.c_void_p(FAKE),
                ws_ptr=ctypes.c_void_p(FAKE), ws_bytes=1 << 20, stream=None)
    args.update(kw)
    return vpce.forward_backward_rows_raw(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(grad_rows_ptr=None), 1),
    (dict(grad_rows_ptr=ctypes.c_void_p(FAKE + 2)), 2),
    (dict(dtype=5), 3),
    (dict(ws_bytes=8), 4),
])
def test_backward_rows_rejects_bad_arguments(lib, kw, code):
    assert _bwd_rows(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(grad_rows_ptr=None), 1),
    (dict(grad_rows_ptr=ctypes.c_void_p(FAKE + 1)), 2),
    (dict(row_loss_ptr=None), 1),                 # 'none' needs the per-row output
    (dict(row_loss_ptr=ctypes.c_void_p(FAKE + 2)), 2),
    (dict(reduction=3), 1),
    (dict(reduction=vpce.VPCE_MEAN), 1),          # 'mean' needs loss_out
])
def test_forward_backward_rows_rejects_bad_arguments(lib, kw, code):
    assert _fb_rows(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(reduction=vpce.VPCE_NONE), 1),          # row_loss_out missing
    (dict(reduction=vpce.VPCE_NONE, loss_ptr=None, row_loss_ptr=ctypes.c_void_p(FAKE + 1)), 2),
])
def test_forward_none_needs_row_losses(lib, kw, code):
    assert _fwd(**kw) == code


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this checks the host-only path")
    # all arguments valid: the first CUDA call (device query) fails, nothing runs
    assert _fwd() == 5
    assert _bwd() == 5
    assert _bwd_rows() == 5
    assert _fb_rows() == 5
    # 'none' takes loss_out as optional
    assert _fwd(reduction=vpce.VPCE_NONE, loss_ptr=None, row_loss_ptr=ctypes.c_void_p(FAKE)) == 5


def _lmhead(**kw):
    args = dict(hidden_ptr=ctypes.c_void_p(FAKE), ld_hidden=0, weight_ptrs=[FAKE, FAKE + 4096], ld_weight=0, t=2,
                s=4, h=128, vocab_start=[0, 16, 40], targets_ptr=ctypes.c_void_p(FAKE), ignore_index=-100,
                reduction=vpce.VPCE_MEAN, loss_ptr=ctypes.c_void_p(FAKE), row_loss_ptr=None,
                ws_ptr=ctypes.c_void_p(FAKE), ws_bytes=1 << 24, stream=None)
    args.update(kw)
    return vpce.lmhead_forward_raw(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(h=100), 1),                               # not a multiple of 64
    (dict(h=0), 1),
    (dict(t=33, weight_ptrs=[FAKE] * 33, vocab_start=list(range(0, 34 * 8, 8))), 1),
    (dict(hidden_ptr=ctypes.c_void_p(FAKE + 8)), 2),  # TMA needs 16-byte bases
    (dict(weight_ptrs=[FAKE, FAKE + 4100]), 2),
    (dict(ld_hidden=130), 2),                       # 260-byte rows are not 16-byte multiples
    (dict(ld_weight=100), 1),                       # narrower than h
    (dict(vocab_start=[0, 16, 16]), 1),
    (dict(weight_ptrs=[FAKE, 0]), 1),
    (dict(reduction=vpce.VPCE_NONE), 1),            # 'none' needs row losses
    (dict(ws_bytes=1024), 4),
    (dict(ws_ptr=ctypes.c_void_p(FAKE + 64)), 2),
])
def test_lmhead_rejects_bad_arguments(lib, kw, code):
    assert _lmhead(**kw) == code


def _lmhead_fb(lib, **kw):
    args = dict(hidden=ctypes.c_void_p(FAKE), ld_hidden=0, weights=[FAKE, FAKE + 4096], ld_weight=0, t=2, s=4,
                h=128, vocab_start=[0, 16, 40], targets=ctypes.c_void_p(FAKE), ignore_index=-100,
                reduction=vpce.VPCE_MEAN, grad=1.0, grad_rows=None, loss=ctypes.c_void_p(FAKE), row_loss=None,
                grad_hidden=ctypes.c_void_p(FAKE), ld_grad_hidden=0, grad_weights=[FAKE + 8192, FAKE + 16384],
                ld_grad_weight=0, ws=ctypes.c_void_p(FAKE), ws_bytes=1 << 30)
    args.update(kw)
    return lib.vpce_lmhead_forward_backward(
        args["hidden"], args["ld_hidden"], ctypes.cast(vpce._ptr_array(args["weights"]), ctypes.c_void_p),
        args["ld_weight"], args["t"], args["s"], args["h"], vpce._i64_array(args["vocab_start"]), args["targets"],
        args["ignore_index"], args["reduction"], args["grad"], args["grad_rows"], args["loss"], args["row_loss"],
        args["grad_hidden"], args["ld_grad_hidden"],
        ctypes.cast(vpce._ptr_array(args["grad_weights"]), ctypes.c_void_p), args["ld_grad_weight"], args["ws"],
        args["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(h=100), 1),                                # not a multiple of 64
    (dict(grad=float("inf")), 1),
    (dict(reduction=vpce.VPCE_NONE, loss=None, row_loss=ctypes.c_void_p(FAKE)), 1),  # 'none' needs grad_rows
    (dict(grad_weights=[FAKE, 0]), 1),
    (dict(grad_hidden=None), 1),
    (dict(hidden=ctypes.c_void_p(FAKE + 8)), 2),
    (dict(grad_weights=[FAKE + 8, FAKE + 4096]), 2),  # fp32 gradient shards are 16-byte aligned
    (dict(ld_grad_weight=130), 2),                    # ... and so are their rows (TMA tile reductions)
    (dict(ws=ctypes.c_void_p(FAKE + 64)), 2),
    (dict(ws_bytes=1 << 16), 4),                      # less than one 128-row chunk
])
def test_lmhead_forward_backward_rejects_bad_arguments(lib, kw, code):
    assert _lmhead_fb(lib, **kw) == code


def test_lmhead_forward_backward_workspace_size(lib):
    f = lib.vpce_lmhead_forward_backward_workspace_bytes
    r256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    s, V, h = 8192, 128256, 8192
    R = 8192
    ld = (V + 7) // 8 * 8 + 8 * 64  # the padded row's bound: each shard's columns start at a multiple of 8
    want = (256 + 2 * r256(4 * s) + r256(8 * 256 * R) + r256(4 * R) + r256(4 * R * ld)
            + r256(2 * R * ld))
    assert f(s, V, h) == want
    assert f(300, 5000, 512) < f(8192, 5000, 512)   # chunks no larger than the batch (rounded to 128)
    assert f(-1, V, h) == 0 and f(s, 0, h) == 0


def test_embedding_rejects_bad_arguments(lib):
    vs = vpce._i64_array([0, 8, 16])
    two = ctypes.cast(vpce._ptr_array([FAKE, FAKE + 4096]), ctypes.c_void_p)
    f = lib.vpce_embedding_forward
    assert f(two, 7, 2, vs, 16, 0, ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), 0, None, None) == 3
    assert f(two, vpce.VPCE_BF16, 0, vs, 16, 0, ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), 0, None, None) == 1
    assert f(two, vpce.VPCE_BF16, 2, vs, 16, 8, ctypes.c_void_p(FAKE), 4, ctypes.c_void_p(FAKE), 0, None, None) == 1
    assert f(two, vpce.VPCE_BF16, 2, vs, 16, 0, ctypes.c_void_p(FAKE + 4), 4, ctypes.c_void_p(FAKE), 0, None,
             None) == 2
    b = lib.vpce_embedding_backward
    ws = ctypes.c_void_p(FAKE)
    nbytes = vpce.vpce_embedding_backward_workspace_bytes()
    assert b(ctypes.c_void_p(FAKE), vpce.VPCE_BF16, 0, ctypes.c_void_p(FAKE), 4, two, 2, vs, 18, 0, ws, nbytes,
             None) == 1                            # h not a multiple of 4
    assert b(ctypes.c_void_p(FAKE + 8), vpce.VPCE_BF16, 0, ctypes.c_void_p(FAKE), 4, two, 2, vs, 16, 0, ws, nbytes,
             None) == 2
    assert b(ctypes.c_void_p(FAKE), vpce.VPCE_BF16, 0, ctypes.c_void_p(FAKE), 4, two, 2, vs, 16, 0, ws, 16,
             None) == 4
    if not __import__("torch").cuda.is_available():
        assert b(ctypes.c_void_p(FAKE), vpce.VPCE_BF16, 0, ctypes.c_void_p(FAKE), 4, two, 2, vs, 16, 0, ws, nbytes,
                 None) == 5
