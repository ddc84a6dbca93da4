"""Helpers of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare it with the fp64 oracle element by element.

Tolerances (written here, used by every parity test):
* loss and per-row loss: relative error <= 1e-5;
* dlogits (mean loss): max abs error <= 4e-3 for bf16 outputs and <= 1e-6 for
  fp32; and, since |d| <= scale is small (scale = g / n_valid for 'mean', g
  for 'sum' and for 'none' with one scalar, g_r per row for 'none' with
  per-row gradients), also the unscaled error max |(d_gpu - d_ref) / scale|
  <= 8e-3 (bf16: two bf16 ulps at values up to 1) and <= 1e-5 (fp32: fp32
  exp2 arguments of magnitude ~40 carry a relative error of a few 1e-6);
  rows whose scale is 0 (or NaN, on an ignored row) must match exactly.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

LOSS_RTOL = 1e-5
D_ATOL = {"bf16": 4e-3, "fp32": 1e-6}
D_UNSCALED = {"bf16": 8e-3, "fp32": 1e-5}


def to_device(host_shards, dtype, device="cuda", misalign: int = 0):
    """Copy host shard arrays to the GPU.  ``misalign`` > 0 places each shard
    that many elements past a 16-byte boundary."""
    out = []
    for h in host_shards:
        if dtype == "bf16":
            tt = torch.from_numpy(np.ascontiguousarray(h).view(np.int16)).view(torch.bfloat16)
        else:
            tt = torch.from_numpy(np.ascontiguousarray(h, dtype=np.float32))
        if misalign:
            flat = torch.empty(tt.numel() + misalign, dtype=tt.dtype, device=device)
            view = flat[misalign:].view(tt.shape)
            view.copy_(tt.to(device))
            out.append(view)
        else:
            out.append(tt.to(device))
    return out


def from_device(t: torch.Tensor, dtype: str) -> np.ndarray:
    """Device shard -> host array in the oracle's stored form."""
    if dtype == "bf16":
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.detach().contiguous().cpu().numpy()


def as_f64(host, dtype):
    return O.widen(host, dtype)


def bits(host, dtype):
    return host.view(np.uint16) if dtype == "bf16" else host.view(np.uint32)


def check_loss(got: float, ref: float):
    if np.isnan(ref):
        assert np.isnan(got), (got, ref)
        return
    assert abs(got - ref) <= LOSS_RTOL * max(abs(ref), 1e-30), (got, ref)


def check_row_losses(got: np.ndarray, ref: np.ndarray, valid: np.ndarray):
    g = got[valid].astype(np.float64)
    r = ref[valid]
    err = np.abs(g - r) / np.maximum(np.abs(r), 1.0)
    assert err.max(initial=0.0) <= LOSS_RTOL, err.max()
    assert np.all(got[~valid] == 0.0) or np.all(np.isnan(got[~valid]) | (got[~valid] == 0.0))


def check_dlogits(got: np.ndarray, ref: np.ndarray, dtype: str, scale, abs_check: bool = True):
    """got, ref: float64 arrays of the same shape [rows, columns]; ``scale``
    is the factor the gradient carries (g / n_valid for 'mean', g for 'sum'),
    a scalar or one value per row.  The absolute bound is the one stated for
    the mean loss; the unscaled bound divides the error by |scale| and holds
    for every reduction."""
    diff = np.abs(got - ref)
    assert np.all(np.isfinite(got) == np.isfinite(ref))
    fin = np.isfinite(ref)
    if not fin.any():
        return
    if abs_check:
        assert diff[fin].max() <= D_ATOL[dtype], diff[fin].max()
    sc = np.abs(np.asarray(scale, dtype=np.float64))
    sc = np.broadcast_to(sc.reshape(-1, 1) if sc.ndim else sc, got.shape)
    # a row scaled by 0 is exactly 0; a finite row under a NaN scale (an
    # ignored row) is exactly the reference
    exact = fin & ((sc == 0) | ~np.isfinite(sc))
    assert np.all(diff[exact] == 0.0)
    nz = fin & ~exact
    if nz.any():
        u = (diff[nz] / sc[nz]).max()
        assert u <= D_UNSCALED[dtype], u


def grad_scale(reduction: str, grad: float, n_valid: int) -> float:
    if reduction in ("sum", "none"):
        return grad
    return grad / n_valid if n_valid > 0 else 0.0


def run_full(w: synth.Workload, *, t: int | None = None, s: int | None = None, vocab_start=None, ld=None,
             reduction: str = "mean", grad: float = 1.0, misalign: int = 0, targets=None, path: str = "split",
             grad_rows=None):
    """Whole-batch parity: oracle on every row and every element.  ``path``:
    'split' (vpce_forward then vpce_backward) or 'fused' (vpce_forward_backward).
    ``grad_rows`` (float32 array, one per row) takes the per-row backward
    entry points instead of the scalar ``grad``."""
    t = w.t if t is None else t
    s = w.s if s is None else s
    w = w.replace(t=t, s=s)
    vs = synth.even_vocab_start(w.V, t) if vocab_start is None else list(vocab_start)
    meta = synth.row_meta(w)
    if targets is not None:
        meta = synth.RowMeta(np.asarray(targets, dtype=np.int64), meta.boost_col, meta.boost_val)
    host = synth.shards_host(w, meta, vs, ld)
    z = O.assemble(host, vs, w.dtype)
    ref = O.cross_entropy(z, meta.targets, w.ignore_index, reduction=reduction)
    if grad_rows is not None:
        grad_rows = np.asarray(grad_rows, dtype=np.float32)
        dref = O.dlogits(z, meta.targets, w.ignore_index, grad=grad_rows.astype(np.float64), reduction="none")
    else:
        dref = O.dlogits(z, meta.targets, w.ignore_index, grad=grad, reduction=reduction)

    dev = to_device(host, w.dtype, misalign=misalign)
    views = [d[:, :vs[i + 1] - vs[i]] for i, d in enumerate(dev)]
    y = torch.from_numpy(meta.targets).cuda()
    row_loss = torch.full((s,), -7.0, dtype=torch.float32, device="cuda")
    loss_t = torch.full((), -7.0, dtype=torch.float32, device="cuda")
    gr = torch.from_numpy(grad_rows).cuda() if grad_rows is not None else None
    if path == "split":
        out, ws = vpce.vpce_forward(views, y, vs, ignore_index=w.ignore_index, reduction=reduction,
                                    loss_out=loss_t, row_loss_out=row_loss)
        flag = vpce.vpce_read_error_flag(ws)
        loss_v = float(loss_t.item())
        rl = row_loss.cpu().numpy()
        vpce.vpce_backward(views, y, ws, vs, ignore_index=w.ignore_index, grad_output=grad, grad_rows=gr)
    else:
        out, ws = vpce.vpce_forward_backward(views, y, vs, ignore_index=w.ignore_index, reduction=reduction,
                                             grad_output=grad, grad_rows=gr, loss_out=loss_t,
                                             row_loss_out=row_loss)
        flag = vpce.vpce_read_error_flag(ws)
        loss_v = float(loss_t.item())
        rl = row_loss.cpu().numpy()
    assert out is (row_loss if reduction == "none" else loss_t)
    torch.cuda.synchronize()
    back = [from_device(d, w.dtype) for d in dev]
    return dict(w=w, vs=vs, meta=meta, host=host, ref=ref, dref=dref, loss=loss_v, row_loss=rl, flag=flag,
                back=back, grad=grad, reduction=reduction, grad_rows=grad_rows)


def check_full(res, *, check_padding=True):
    w, vs, ref = res["w"], res["vs"], res["ref"]
    # 'none' writes the plain sum to loss_out when one is given
    check_loss(res["loss"], ref["loss"] if np.ndim(ref["loss"]) == 0 else float(ref["row_loss"].sum()))
    check_row_losses(res["row_loss"], ref["row_loss"], ref["valid"])
    assert res["flag"] == ref["error_flag"]
    got = O.assemble(res["back"], vs, w.dtype)
    if res.get("grad_rows") is not None:
        scale, abs_check = res["grad_rows"].astype(np.float64), False
    else:
        scale = grad_scale(res["reduction"], res["grad"], ref["n_valid"])
        abs_check = res["reduction"] == "mean"
    check_dlogits(got, res["dref"], w.dtype, scale, abs_check=abs_check)
    ign = res["meta"].targets == w.ignore_index
    assert np.all(got[ign] == 0.0)
    if check_padding:
        for i, (h, b) in enumerate(zip(res["host"], res["back"])):
            width = vs[i + 1] - vs[i]
            if b.shape[1] > width:
                np.testing.assert_array_equal(bits(b[:, width:], w.dtype), bits(h[:, width:], w.dtype))
