"""ctypes binding of ``libvpce.so`` (C ABI in include/vpce.h).

Argument marshalling only: every step of the loss runs in the library's CUDA
kernels.  torch supplies device memory and the current stream.  The names are
the C entry points'.  The library is loaded on first use; if it is missing the
call raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_lib", "libvpce.so")

VPCE_OK = 0
STATUS_NAMES = {
    0: "VPCE_OK",
    1: "VPCE_ERR_INVALID_ARG",
    2: "VPCE_ERR_ALIGNMENT",
    3: "VPCE_ERR_DTYPE",
    4: "VPCE_ERR_WORKSPACE",
    5: "VPCE_ERR_CUDA",
    6: "VPCE_ERR_UNSUPPORTED_DEVICE",
}
VPCE_FP32, VPCE_BF16 = 0, 1
VPCE_MEAN, VPCE_SUM, VPCE_NONE = 0, 1, 2
REDUCTIONS = {"mean": VPCE_MEAN, "sum": VPCE_SUM, "none": VPCE_NONE}
VPCE_MAX_SHARDS = 64
VPCE_FLAG_BAD_TARGET = 1
VPCE_FLAG_WAIT_TIMEOUT = 2
VPCE_STATIC_SCRATCH_BYTES = 8 * 1024 * 1024
VPCE_LMHEAD_MAX_GROUPS = 256

_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I64P = ctypes.POINTER(ctypes.c_int64)


class VPCEError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {vpce_status_string(code)} ({code})")


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libvpce.so (once) and declare its signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is not built: run __graft_entry__.build() (nvcc, sm_103a)")
        lib = ctypes.CDLL(p)
        lib.vpce_workspace_bytes.restype = ctypes.c_size_t
        lib.vpce_workspace_bytes.argtypes = [ctypes.c_int, _I64]
        lib.vpce_forward.restype = ctypes.c_int
        lib.vpce_forward.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                     ctypes.c_int, _P, _P, _P, ctypes.c_size_t, _P]
        lib.vpce_backward.restype = ctypes.c_int
        lib.vpce_backward.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                      ctypes.c_float, _P, ctypes.c_size_t, _P]
        lib.vpce_backward_rows.restype = ctypes.c_int
        lib.vpce_backward_rows.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                           _P, _P, ctypes.c_size_t, _P]
        lib.vpce_forward_backward.restype = ctypes.c_int
        lib.vpce_forward_backward.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                              ctypes.c_int, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P]
        lib.vpce_forward_backward_rows.restype = ctypes.c_int
        lib.vpce_forward_backward_rows.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                                   ctypes.c_int, _P, _P, _P, _P, ctypes.c_size_t, _P]
        lib.vpce_fused_plan.restype = ctypes.c_int
        lib.vpce_fused_plan.argtypes = [ctypes.c_int, ctypes.c_int, _I64P, _I64, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]
        lib.vpce_forward_static.restype = ctypes.c_int
        lib.vpce_forward_static.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64,
                                            ctypes.c_int, _P, _P, _P]
        lib.vpce_partials.restype = ctypes.c_int
        lib.vpce_partials.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64, _I64P, _I64, _P, _I64, _P, _P, _P,
                                      ctypes.c_size_t, _P]
        lib.vpce_combine_partials.restype = ctypes.c_int
        lib.vpce_combine_partials.argtypes = [_P, ctypes.c_int, _P, _I64, _I64, _P, _I64, ctypes.c_int, _P, _P,
                                              ctypes.c_int, _P, ctypes.c_size_t, _P]
        lib.vpce_fold_partials.restype = ctypes.c_int
        lib.vpce_fold_partials.argtypes = [_P, ctypes.c_int, _I64, _P, _P]
        lib.vpce_lmhead_workspace_bytes.restype = ctypes.c_size_t
        lib.vpce_lmhead_workspace_bytes.argtypes = [_I64]
        lib.vpce_lmhead_forward.restype = ctypes.c_int
        lib.vpce_lmhead_forward.argtypes = [_P, _I64, _P, _I64, ctypes.c_int, _I64, _I64, _I64P, _P, _I64,
                                            ctypes.c_int, _P, _P, _P, ctypes.c_size_t, _P]
        lib.vpce_lmhead_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.vpce_lmhead_backward_workspace_bytes.argtypes = [_I64, _I64]
        lib.vpce_lmhead_backward.restype = ctypes.c_int
        lib.vpce_lmhead_backward.argtypes = [_P, _I64, _P, _I64, ctypes.c_int, _I64, _I64, _I64P, _P, _I64,
                                             ctypes.c_float, _P, _P, ctypes.c_size_t, _P, _I64, _P, _I64, _P,
                                             ctypes.c_size_t, _P]
        lib.vpce_lmhead_forward_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.vpce_lmhead_forward_backward_workspace_bytes.argtypes = [_I64, _I64, _I64]
        lib.vpce_lmhead_forward_backward.restype = ctypes.c_int
        lib.vpce_lmhead_forward_backward.argtypes = [_P, _I64, _P, _I64, ctypes.c_int, _I64, _I64, _I64P, _P, _I64,
                                                     ctypes.c_int, ctypes.c_float, _P, _P, _P, _P, _I64, _P, _I64,
                                                     _P, ctypes.c_size_t, _P]
        lib.vpce_embedding_forward.restype = ctypes.c_int
        lib.vpce_embedding_forward.argtypes = [_P, ctypes.c_int, ctypes.c_int, _I64P, _I64, _I64, _P, _I64, _P,
                                               _I64, _P, _P]
        lib.vpce_embedding_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.vpce_embedding_backward_workspace_bytes.argtypes = []
        lib.vpce_embedding_backward.restype = ctypes.c_int
        lib.vpce_embedding_backward.argtypes = [_P, ctypes.c_int, _I64, _P, _I64, _P, ctypes.c_int, _I64P, _I64,
                                                _I64, _P, ctypes.c_size_t, _P]
        lib.vpce_read_error_flag.restype = ctypes.c_int
        lib.vpce_read_error_flag.argtypes = [_P, ctypes.POINTER(ctypes.c_int), _P]
        lib.vpce_status_string.restype = ctypes.c_char_p
        lib.vpce_status_string.argtypes = [ctypes.c_int]
        if path is None:
            _lib = lib
        return lib


def vpce_status_string(code: int) -> str:
    try:
        return load_library().vpce_status_string(int(code)).decode()
    except RuntimeError:
        return STATUS_NAMES.get(int(code), "VPCE_ERR_UNKNOWN")


def vpce_workspace_bytes(t: int, s: int) -> int:
    return int(load_library().vpce_workspace_bytes(int(t), int(s)))


# ----------------------------------------------------------------------------
# raw-pointer forms (the C signatures one to one)
# ----------------------------------------------------------------------------
def _ptr_array(ptrs):
    arr = (ctypes.c_void_p * len(ptrs))(*[int(p) for p in ptrs])
    return arr


def _i64_array(vals):
    return (ctypes.c_int64 * len(vals))(*[int(v) for v in vals])


def forward_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, reduction,
                loss_ptr, row_loss_ptr, ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_forward(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype), int(t),
                                int(s), vs, int(ld), targets_ptr, int(ignore_index), int(reduction),
                                loss_ptr, row_loss_ptr, ws_ptr, int(ws_bytes), stream))


def backward_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, grad,
                 ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_backward(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype), int(t),
                                 int(s), vs, int(ld), targets_ptr, int(ignore_index), float(grad),
                                 ws_ptr, int(ws_bytes), stream))


def backward_rows_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, grad_rows_ptr,
                      ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_backward_rows(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype), int(t),
                                      int(s), vs, int(ld), targets_ptr, int(ignore_index), grad_rows_ptr,
                                      ws_ptr, int(ws_bytes), stream))


# ----------------------------------------------------------------------------
# torch-tensor forms
# ----------------------------------------------------------------------------
def _describe(shards, vocab_start):
    import torch

    if not shards:
        raise ValueError("need at least one shard")
    dt = shards[0].dtype
    if dt == torch.bfloat16:
        dtype = VPCE_BF16
    elif dt == torch.float32:
        dtype = VPCE_FP32
    else:
        raise TypeError(f"unsupported logits dtype {dt}")
    s = shards[0].shape[0]
    widths = []
    for sh in shards:
        if sh.dtype != dt or sh.dim() != 2 or sh.shape[0] != s or not sh.is_cuda:
            raise ValueError("shards must be 2-D CUDA tensors of one dtype and row count")
        if sh.stride(1) != 1:
            raise ValueError("shard columns must be contiguous")
        widths.append(sh.shape[1])
    if vocab_start is None:
        vocab_start = [0]
        for w in widths:
            vocab_start.append(vocab_start[-1] + w)
    vocab_start = [int(v) for v in vocab_start]
    strides = {sh.stride(0) for sh in shards}
    if s <= 1 or all(sh.stride(0) == sh.shape[1] for sh in shards):
        ld = 0
    elif len(strides) == 1:
        ld = strides.pop()
    else:
        raise ValueError("shards must share one row stride or each be dense")
    return dtype, s, vocab_start, ld


def _stream_ptr(stream):
    import torch

    st = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(st.cuda_stream)


def new_workspace(t: int, s: int, device=None):
    import torch

    n = vpce_workspace_bytes(t, s)
    if n == 0:
        raise ValueError("t or s out of range")
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(n, dtype=torch.uint8, device=device)


def _ptr(x):
    return ctypes.c_void_p(x.data_ptr()) if x is not None else None


def _outputs(reduction, loss_out, row_loss_out, s, dev):
    """The reduction code and the loss buffers: 'none' returns the per-row
    vector (allocated if not given); the others a scalar."""
    import torch

    red = REDUCTIONS[reduction]
    if red == VPCE_NONE:
        if row_loss_out is None:
            row_loss_out = torch.empty(s, dtype=torch.float32, device=dev)
        return red, loss_out, row_loss_out, row_loss_out
    if loss_out is None:
        loss_out = torch.empty((), dtype=torch.float32, device=dev)
    return red, loss_out, row_loss_out, loss_out


def _check_grad_rows(grad_rows, s):
    import torch

    if grad_rows.dtype != torch.float32 or not grad_rows.is_cuda or grad_rows.numel() != s \
            or (s > 1 and grad_rows.stride(0) != 1):
        raise ValueError("grad_rows must be a contiguous CUDA float32 tensor with one entry per row")


def vpce_forward(shards, targets, vocab_start=None, *, ignore_index: int = -100, reduction: str = "mean",
                 loss_out=None, row_loss_out=None, workspace=None, stream=None):
    """Loss of vocab-sharded logits.  Returns ``(loss, workspace)``; pass the
    workspace unchanged to :func:`vpce_backward`.  With ``reduction='none'``
    the loss returned is the per-row vector."""
    import torch

    dtype, s, vs, ld = _describe(shards, vocab_start)
    t = len(shards)
    dev = shards[0].device
    if targets.dtype != torch.int64 or not targets.is_cuda or targets.numel() != s:
        raise ValueError("targets must be a CUDA int64 tensor with one entry per row")
    if workspace is None:
        workspace = new_workspace(t, s, dev)
    red, loss_out, row_loss_out, result = _outputs(reduction, loss_out, row_loss_out, s, dev)
    code = forward_raw([sh.data_ptr() for sh in shards], dtype, t, s, vs, ld,
                       ctypes.c_void_p(targets.data_ptr()), ignore_index, red, _ptr(loss_out),
                       _ptr(row_loss_out), ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                       _stream_ptr(stream))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_forward")
    return result, workspace


def vpce_backward(shards, targets, workspace, vocab_start=None, *, ignore_index: int = -100,
                  grad_output: float = 1.0, grad_rows=None, stream=None):
    """Overwrite ``shards`` in place with dlogits of the preceding forward.
    ``grad_rows`` (a float32 vector, one entry per row) selects the per-row
    backward (vpce_backward_rows) instead of the scalar ``grad_output``."""
    dtype, s, vs, ld = _describe(shards, vocab_start)
    ptrs = [sh.data_ptr() for sh in shards]
    if grad_rows is not None:
        _check_grad_rows(grad_rows, s)
        code = backward_rows_raw(ptrs, dtype, len(shards), s, vs, ld, ctypes.c_void_p(targets.data_ptr()),
                                 ignore_index, _ptr(grad_rows), ctypes.c_void_p(workspace.data_ptr()),
                                 workspace.numel(), _stream_ptr(stream))
        where = "vpce_backward_rows"
    else:
        code = backward_raw(ptrs, dtype, len(shards), s, vs, ld, ctypes.c_void_p(targets.data_ptr()),
                            ignore_index, grad_output, ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                            _stream_ptr(stream))
        where = "vpce_backward"
    if code != VPCE_OK:
        raise VPCEError(code, where)
    return shards


def forward_backward_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, reduction, grad,
                         loss_ptr, row_loss_ptr, ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_forward_backward(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype),
                                         int(t), int(s), vs, int(ld), targets_ptr, int(ignore_index),
                                         int(reduction), float(grad), loss_ptr, row_loss_ptr, ws_ptr,
                                         int(ws_bytes), stream))


def forward_backward_rows_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, reduction,
                              grad_rows_ptr, loss_ptr, row_loss_ptr, ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_forward_backward_rows(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype),
                                              int(t), int(s), vs, int(ld), targets_ptr, int(ignore_index),
                                              int(reduction), grad_rows_ptr, loss_ptr, row_loss_ptr, ws_ptr,
                                              int(ws_bytes), stream))


def vpce_forward_backward(shards, targets, vocab_start=None, *, ignore_index: int = -100,
                          reduction: str = "mean", grad_output: float = 1.0, grad_rows=None, loss_out=None,
                          row_loss_out=None, workspace=None, stream=None):
    """Loss and in-place dlogits in one call (the logits cross HBM once each
    way).  Returns ``(loss, workspace)`` (the per-row vector for
    ``reduction='none'``); ``shards`` now hold dlogits.  ``grad_rows`` (one
    float32 per row) replaces the scalar ``grad_output``."""
    import torch

    dtype, s, vs, ld = _describe(shards, vocab_start)
    t = len(shards)
    dev = shards[0].device
    if targets.dtype != torch.int64 or not targets.is_cuda or targets.numel() != s:
        raise ValueError("targets must be a CUDA int64 tensor with one entry per row")
    if workspace is None:
        workspace = new_workspace(t, s, dev)
    red, loss_out, row_loss_out, result = _outputs(reduction, loss_out, row_loss_out, s, dev)
    ptrs = [sh.data_ptr() for sh in shards]
    if grad_rows is not None:
        _check_grad_rows(grad_rows, s)
        code = forward_backward_rows_raw(ptrs, dtype, t, s, vs, ld, ctypes.c_void_p(targets.data_ptr()),
                                         ignore_index, red, _ptr(grad_rows), _ptr(loss_out), _ptr(row_loss_out),
                                         ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                         _stream_ptr(stream))
        where = "vpce_forward_backward_rows"
    else:
        code = forward_backward_raw(ptrs, dtype, t, s, vs, ld, ctypes.c_void_p(targets.data_ptr()), ignore_index,
                                    red, grad_output, _ptr(loss_out), _ptr(row_loss_out),
                                    ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
        where = "vpce_forward_backward"
    if code != VPCE_OK:
        raise VPCEError(code, where)
    return result, workspace


def vpce_fused_plan(dtype: int, vocab_start, s: int) -> dict:
    """The launch vpce_forward_backward would use (kernel: 'split' two-call
    path or 'stream' fused kernel; grid in CTAs)."""
    k, c, g = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    code = load_library().vpce_fused_plan(int(dtype), len(vocab_start) - 1, _i64_array(vocab_start), int(s),
                                          ctypes.byref(k), ctypes.byref(c), ctypes.byref(g))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_fused_plan")
    return {"kernel": ["split", "stream"][k.value], "cluster": c.value, "grid": g.value}


def vpce_read_error_flag(workspace, stream=None) -> int:
    flag = ctypes.c_int(0)
    code = load_library().vpce_read_error_flag(ctypes.c_void_p(workspace.data_ptr()), ctypes.byref(flag),
                                               _stream_ptr(stream))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_read_error_flag")
    return flag.value


# ----------------------------------------------------------------------------
# forward with the library's own static scratch (no workspace argument)
# ----------------------------------------------------------------------------
def forward_static_raw(shard_ptrs, dtype, t, s, vocab_start, ld, targets_ptr, ignore_index, reduction,
                       loss_ptr, row_loss_ptr, stream) -> int:
    """vpce_forward_static one to one.  For callers that cannot allocate
    device memory: the scratch is a fixed array inside the library (see
    include/vpce.h); calls that overlap on the GPU share it and race."""
    lib = load_library()
    ptrs = _ptr_array(shard_ptrs) if shard_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_forward_static(ctypes.cast(ptrs, _P) if ptrs is not None else None, int(dtype), int(t),
                                       int(s), vs, int(ld), targets_ptr, int(ignore_index), int(reduction),
                                       loss_ptr, row_loss_ptr, stream))


def vpce_forward_static(shards, targets, loss_out, vocab_start=None, *, ignore_index: int = -100,
                        reduction: str = "mean", row_loss_out=None, stream=None):
    """Loss of vocab-sharded logits into the caller's ``loss_out`` (and
    ``row_loss_out``), using no workspace from the caller."""
    dtype, s, vs, ld = _describe(shards, vocab_start)
    red = REDUCTIONS[reduction]
    code = forward_static_raw([sh.data_ptr() for sh in shards], dtype, len(shards), s, vs, ld,
                              ctypes.c_void_p(targets.data_ptr()), ignore_index, red, _ptr(loss_out),
                              _ptr(row_loss_out), _stream_ptr(stream))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_forward_static")
    return loss_out



# ----------------------------------------------------------------------------
# LM-head GEMM fused with the forward loss (the logits are never written)
# ----------------------------------------------------------------------------
def vpce_lmhead_workspace_bytes(s: int) -> int:
    return int(load_library().vpce_lmhead_workspace_bytes(int(s)))


def lmhead_forward_raw(hidden_ptr, ld_hidden, weight_ptrs, ld_weight, t, s, h, vocab_start, targets_ptr,
                       ignore_index, reduction, loss_ptr, row_loss_ptr, ws_ptr, ws_bytes, stream) -> int:
    lib = load_library()
    ptrs = _ptr_array(weight_ptrs) if weight_ptrs is not None else None
    vs = _i64_array(vocab_start) if vocab_start is not None else None
    return int(lib.vpce_lmhead_forward(hidden_ptr, int(ld_hidden), ctypes.cast(ptrs, _P) if ptrs is not None else None,
                                       int(ld_weight), int(t), int(s), int(h), vs, targets_ptr, int(ignore_index),
                                       int(reduction), loss_ptr, row_loss_ptr, ws_ptr, int(ws_bytes), stream))


def vpce_lmhead_forward(hidden, weight_shards, targets, vocab_start=None, *, ignore_index: int = -100,
                        reduction: str = "mean", loss_out=None, row_loss_out=None, workspace=None, stream=None):
    """Loss of the logits ``hidden @ W_i^T`` of every vocabulary shard, formed
    and reduced tile by tile on the tensor cores.  ``hidden``: CUDA bf16
    ``[s, h]``; ``weight_shards``: CUDA bf16 ``[w_i, h]`` sharing one row
    stride.  Returns ``(loss, workspace)`` (the per-row vector for 'none')."""
    import torch

    if hidden.dtype != torch.bfloat16 or hidden.dim() != 2 or not hidden.is_cuda or hidden.stride(1) != 1:
        raise ValueError("hidden must be a CUDA bf16 [s, h] tensor with contiguous columns")
    s, h = hidden.shape
    if not weight_shards:
        raise ValueError("need at least one weight shard")
    for w in weight_shards:
        if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_cuda or w.shape[1] != h or w.stride(1) != 1:
            raise ValueError("weight shards must be CUDA bf16 [w_i, h] tensors with contiguous columns")
    strides = {w.stride(0) for w in weight_shards if w.shape[0] > 1}
    if len(strides) > 1:
        raise ValueError("weight shards must share one row stride")
    ld_w = strides.pop() if strides else h
    ld_x = hidden.stride(0) if s > 1 else h
    if vocab_start is None:
        vocab_start = [0]
        for w in weight_shards:
            vocab_start.append(vocab_start[-1] + w.shape[0])
    if targets.dtype != torch.int64 or not targets.is_cuda or targets.numel() != s:
        raise ValueError("targets must be a CUDA int64 tensor with one entry per row")
    dev = hidden.device
    if workspace is None:
        workspace = torch.empty(vpce_lmhead_workspace_bytes(s), dtype=torch.uint8, device=dev)
    red, loss_out, row_loss_out, result = _outputs(reduction, loss_out, row_loss_out, s, dev)
    code = lmhead_forward_raw(ctypes.c_void_p(hidden.data_ptr()), ld_x, [w.data_ptr() for w in weight_shards],
                              ld_w, len(weight_shards), s, h, vocab_start, ctypes.c_void_p(targets.data_ptr()),
                              ignore_index, red, _ptr(loss_out), _ptr(row_loss_out),
                              ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_lmhead_forward")
    return result, workspace


def vpce_lmhead_backward_workspace_bytes(V: int, h: int) -> int:
    return int(load_library().vpce_lmhead_backward_workspace_bytes(int(V), int(h)))


def vpce_lmhead_backward(hidden, weight_shards, targets, fwd_workspace, vocab_start=None, *,
                         ignore_index: int = -100, grad_output: float = 1.0, grad_rows=None, grad_hidden=None,
                         grad_weight_shards=None, workspace=None, stream=None):
    """dX (bf16, overwritten) and dW_i (fp32, accumulated) of the loss of
    the preceding :func:`vpce_lmhead_forward` (same inputs, its workspace).
    Returns ``(grad_hidden, grad_weight_shards)``."""
    import torch

    s, h = hidden.shape
    if vocab_start is None:
        vocab_start = [0]
        for w in weight_shards:
            vocab_start.append(vocab_start[-1] + w.shape[0])
    vocab_start = [int(v) for v in vocab_start]
    strides = {w.stride(0) for w in weight_shards if w.shape[0] > 1}
    ld_w = strides.pop() if len(strides) == 1 else h
    dev = hidden.device
    if grad_hidden is None:
        grad_hidden = torch.empty((s, h), dtype=torch.bfloat16, device=dev)
    if grad_weight_shards is None:
        grad_weight_shards = [torch.zeros((w.shape[0], h), dtype=torch.float32, device=dev) for w in weight_shards]
    gstr = {g.stride(0) for g in grad_weight_shards if g.shape[0] > 1}
    ld_gw = gstr.pop() if len(gstr) == 1 else h
    if grad_rows is not None:
        _check_grad_rows(grad_rows, s)
    if workspace is None:
        workspace = torch.empty(vpce_lmhead_backward_workspace_bytes(vocab_start[-1], h), dtype=torch.uint8,
                                device=dev)
    code = int(load_library().vpce_lmhead_backward(
        ctypes.c_void_p(hidden.data_ptr()), int(hidden.stride(0) if s > 1 else h),
        ctypes.cast(_ptr_array([w.data_ptr() for w in weight_shards]), _P), int(ld_w), len(weight_shards), int(s),
        int(h), _i64_array(vocab_start), ctypes.c_void_p(targets.data_ptr()), int(ignore_index), float(grad_output),
        _ptr(grad_rows), ctypes.c_void_p(fwd_workspace.data_ptr()), fwd_workspace.numel(),
        ctypes.c_void_p(grad_hidden.data_ptr()), int(grad_hidden.stride(0) if s > 1 else h),
        ctypes.cast(_ptr_array([g.data_ptr() for g in grad_weight_shards]), _P), int(ld_gw),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream)))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_lmhead_backward")
    return grad_hidden, grad_weight_shards


# ----------------------------------------------------------------------------
# vocabulary-parallel input embedding
# ----------------------------------------------------------------------------
def _table_desc(shards, vocab_start):
    import torch

    if not shards:
        raise ValueError("need at least one shard")
    dt = shards[0].dtype
    h = shards[0].shape[1]
    for e in shards:
        if e.dtype != dt or e.dim() != 2 or e.shape[1] != h or not e.is_cuda or e.stride(1) != 1:
            raise ValueError("table shards must be 2-D CUDA tensors [w_i, h] of one dtype, contiguous columns")
    strides = {e.stride(0) for e in shards if e.shape[0] > 1}
    if len(strides) > 1:
        raise ValueError("table shards must share one row stride")
    ld = strides.pop() if strides else h
    if vocab_start is None:
        vocab_start = [0]
        for e in shards:
            vocab_start.append(vocab_start[-1] + e.shape[0])
    code = {torch.bfloat16: VPCE_BF16, torch.float32: VPCE_FP32}.get(dt)
    return code, h, ld, [int(v) for v in vocab_start]


def vpce_lmhead_forward_backward_workspace_bytes(s: int, V: int, h: int) -> int:
    return int(load_library().vpce_lmhead_forward_backward_workspace_bytes(int(s), int(V), int(h)))


def vpce_lmhead_forward_backward(hidden, weight_shards, targets, vocab_start=None, *, ignore_index: int = -100,
                                 reduction: str = "mean", grad_output: float = 1.0, grad_rows=None, loss_out=None,
                                 row_loss_out=None, grad_hidden=None, grad_weight_shards=None, workspace=None,
                                 stream=None):
    """:func:`vpce_lmhead_forward` and :func:`vpce_lmhead_backward` in one
    call (the upstream gradient known up front): each row chunk's logits are
    formed once and kept in the workspace for its gradient.  Returns
    ``(loss, grad_hidden, grad_weight_shards)`` (the per-row vector as the
    loss for 'none'); dX is overwritten, dW accumulated."""
    import torch

    if hidden.dtype != torch.bfloat16 or hidden.dim() != 2 or not hidden.is_cuda or hidden.stride(1) != 1:
        raise ValueError("hidden must be a CUDA bf16 [s, h] tensor with contiguous columns")
    s, h = hidden.shape
    if not weight_shards:
        raise ValueError("need at least one weight shard")
    for w in weight_shards:
        if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_cuda or w.shape[1] != h or w.stride(1) != 1:
            raise ValueError("weight shards must be CUDA bf16 [w_i, h] tensors with contiguous columns")
    strides = {w.stride(0) for w in weight_shards if w.shape[0] > 1}
    if len(strides) > 1:
        raise ValueError("weight shards must share one row stride")
    ld_w = strides.pop() if strides else h
    ld_x = hidden.stride(0) if s > 1 else h
    if vocab_start is None:
        vocab_start = [0]
        for w in weight_shards:
            vocab_start.append(vocab_start[-1] + w.shape[0])
    vocab_start = [int(v) for v in vocab_start]
    if targets.dtype != torch.int64 or not targets.is_cuda or targets.numel() != s:
        raise ValueError("targets must be a CUDA int64 tensor with one entry per row")
    dev = hidden.device
    if grad_hidden is None:
        grad_hidden = torch.empty((s, h), dtype=torch.bfloat16, device=dev)
    if grad_weight_shards is None:
        grad_weight_shards = [torch.zeros((w.shape[0], h), dtype=torch.float32, device=dev) for w in weight_shards]
    gstr = {g.stride(0) for g in grad_weight_shards if g.shape[0] > 1}
    ld_gw = gstr.pop() if len(gstr) == 1 else h
    if grad_rows is not None:
        _check_grad_rows(grad_rows, s)
    if workspace is None:
        workspace = torch.empty(vpce_lmhead_forward_backward_workspace_bytes(s, vocab_start[-1], h),
                                dtype=torch.uint8, device=dev)
    red, loss_out, row_loss_out, result = _outputs(reduction, loss_out, row_loss_out, s, dev)
    code = int(load_library().vpce_lmhead_forward_backward(
        ctypes.c_void_p(hidden.data_ptr()), int(ld_x), ctypes.cast(_ptr_array([w.data_ptr() for w in weight_shards]), _P),
        int(ld_w), len(weight_shards), int(s), int(h), _i64_array(vocab_start), ctypes.c_void_p(targets.data_ptr()),
        int(ignore_index), red, float(grad_output), _ptr(grad_rows), _ptr(loss_out), _ptr(row_loss_out),
        ctypes.c_void_p(grad_hidden.data_ptr()), int(grad_hidden.stride(0) if s > 1 else h),
        ctypes.cast(_ptr_array([g.data_ptr() for g in grad_weight_shards]), _P), int(ld_gw),
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel(), _stream_ptr(stream)))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_lmhead_forward_backward")
    return result, grad_hidden, grad_weight_shards


def vpce_embedding_forward(table_shards, ids, vocab_start=None, *, out=None, flag=None, stream=None):
    """Rows ``table[ids]`` of a vocabulary-split table (zero rows for ids
    outside [0, V)).  ``flag`` (CUDA int32 scalar) receives bit 0 if any id
    was outside."""
    import torch

    dtype, h, ld, vs = _table_desc(table_shards, vocab_start)
    if dtype is None:
        raise TypeError("table dtype must be bf16 or fp32")
    if ids.dtype != torch.int64 or not ids.is_cuda or ids.dim() != 1:
        raise ValueError("ids must be a 1-D CUDA int64 tensor")
    s = ids.numel()
    if out is None:
        out = torch.empty((s, h), dtype=table_shards[0].dtype, device=ids.device)
    ld_out = out.stride(0) if s > 1 else h
    lib = load_library()
    code = int(lib.vpce_embedding_forward(ctypes.cast(_ptr_array([e.data_ptr() for e in table_shards]), _P),
                                          int(dtype), len(table_shards), _i64_array(vs), int(h), int(ld),
                                          ctypes.c_void_p(ids.data_ptr()), int(s), _ptr(out), int(ld_out),
                                          _ptr(flag), _stream_ptr(stream)))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_embedding_forward")
    return out


def vpce_embedding_backward_workspace_bytes() -> int:
    return int(load_library().vpce_embedding_backward_workspace_bytes())


def vpce_embedding_backward(grad_out, ids, grad_shards, vocab_start=None, *, workspace=None, stream=None):
    """Accumulate the lookup's adjoint into the fp32 gradient-table shards
    (in place): each gradient row is added into its id's row."""
    import torch

    gdt, h, ld, vs = _table_desc(grad_shards, vocab_start)
    if gdt != VPCE_FP32:
        raise TypeError("gradient table shards must be fp32")
    if grad_out.dim() != 2 or grad_out.shape[1] != h or not grad_out.is_cuda or grad_out.stride(1) != 1:
        raise ValueError("grad_out must be a CUDA [s, h] tensor with contiguous columns")
    code_dt = {torch.bfloat16: VPCE_BF16, torch.float32: VPCE_FP32}.get(grad_out.dtype)
    if code_dt is None:
        raise TypeError("grad_out dtype must be bf16 or fp32")
    s = grad_out.shape[0]
    if ids.dtype != torch.int64 or not ids.is_cuda or ids.numel() != s:
        raise ValueError("ids must be a CUDA int64 tensor with one entry per row")
    if workspace is None:
        workspace = torch.empty(vpce_embedding_backward_workspace_bytes(), dtype=torch.uint8, device=ids.device)
    lib = load_library()
    code = int(lib.vpce_embedding_backward(_ptr(grad_out), int(code_dt), int(grad_out.stride(0) if s > 1 else h),
                                           ctypes.c_void_p(ids.data_ptr()), int(s),
                                           ctypes.cast(_ptr_array([g.data_ptr() for g in grad_shards]), _P),
                                           len(grad_shards), _i64_array(vs), int(h), int(ld),
                                           ctypes.c_void_p(workspace.data_ptr()), workspace.numel(),
                                           _stream_ptr(stream)))
    if code != VPCE_OK:
        raise VPCEError(code, "vpce_embedding_backward")
    return grad_shards
