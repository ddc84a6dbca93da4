"""GPU parity of vpce_lmhead_forward (LM-head GEMM on the tensor cores fused
with the sharded loss) against the fp64 oracle: z = X W^T, then the
cross-entropy of z, every row of small cases with ragged M and N tiles,
uneven and one-column shards, padded row strides, ignored and bad targets,
the reductions, and sampled rows of the full-size head.

Tolerances.  The tensor cores multiply bf16 exactly and accumulate in fp32,
h / 16 accumulator updates per logit (16 products per tcgen05.mma step).  A
logit's error is then at most gamma * S_rk, gamma = (h / 16) * 2^-24 and S_rk
= sum_k |x_rk w_jk| (the classic bound for that many rounded additions), and
a row's loss lse - z_y moves by at most twice the largest logit error.  The
test bounds each row by 2 * gamma * max_j S_rj.  The batch loss carries the
loss tolerance of the sharded path, 1e-5 relative."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _host(m, vs, rows=None):
    rows = np.arange(m.s) if rows is None else np.asarray(rows)
    xh = synth.dense_host(m.seed, synth.STREAM_HIDDEN, rows, m.h, m.sigma_x)
    wh = [synth.dense_host(m.seed, synth.STREAM_WEIGHT, np.arange(vs[i], vs[i + 1]), m.h, m.sigma_w)
          for i in range(len(vs) - 1)]
    return xh, wh


def _row_bound(xh, wh, h):
    """2 * gamma * max_j sum_k |x_rk w_jk| per row."""
    X = np.abs(O.widen(xh, "bf16"))
    S = np.max(np.concatenate([X @ np.abs(O.widen(w, "bf16")).T for w in wh], axis=1), axis=1)
    return 2.0 * (h / 16) * 2.0 ** -24 * S


def _check(m, vs=None, *, targets=None, reduction="mean", pad_x=0, pad_w=0):
    vs = synth.even_vocab_start(m.V, m.t) if vs is None else list(vs)
    meta = synth.lmhead_meta(m)
    y_host = meta.targets if targets is None else np.asarray(targets, dtype=np.int64)
    x, ws = synth.lmhead_device(m, vs)
    if pad_x:
        xp = torch.zeros((m.s, m.h + pad_x), dtype=torch.bfloat16, device="cuda")
        xp[:, :m.h] = x
        x = xp[:, :m.h]
    if pad_w:
        wp = []
        for w in ws:
            b = torch.zeros((w.shape[0], m.h + pad_w), dtype=torch.bfloat16, device="cuda")
            b[:, :m.h] = w
            wp.append(b[:, :m.h])
        ws = wp
    y = torch.from_numpy(y_host).cuda()
    rl = torch.full((m.s,), -7.0, dtype=torch.float32, device="cuda")
    loss_t = torch.full((), -7.0, dtype=torch.float32, device="cuda")
    out, wk = vpce.vpce_lmhead_forward(x, ws, y, vs, ignore_index=m.ignore_index, reduction=reduction,
                                       loss_out=loss_t, row_loss_out=rl)
    flag = vpce.vpce_read_error_flag(wk)
    got_rows = rl.cpu().numpy().astype(np.float64)
    got_loss = float(loss_t.item())

    xh, wh = _host(m, vs)
    z = O.lmhead_logits(xh, wh, vs)
    ref = O.cross_entropy(z, y_host, m.ignore_index, reduction=reduction)
    valid = ref["valid"]
    bound = _row_bound(xh, wh, m.h)
    err = np.abs(got_rows - ref["row_loss"])
    assert np.all(err[valid] <= bound[valid]), (err[valid].max(), bound[valid].min())
    assert np.all(got_rows[y_host == m.ignore_index] == 0.0)
    bad = (~valid) & (y_host != m.ignore_index)
    assert np.all(np.isnan(got_rows[bad]))
    assert flag == ref["error_flag"]
    exp_loss = ref["loss"] if np.ndim(ref["loss"]) == 0 else float(ref["row_loss"].sum())
    if np.isnan(exp_loss):
        assert np.isnan(got_loss)
    else:
        assert abs(got_loss - exp_loss) <= LOSS_RTOL * abs(exp_loss), (got_loss, exp_loss)
    return got_rows, got_loss


@pytest.mark.parametrize("m,vs", [
    (synth.LMHEADS["lmhead_s300_h512_v5000"], None),          # ragged M and N tiles, 3 shards, ignored rows
    (synth.LmHead("one_tile", 8, 128, 64, 256, 1), None),      # one tile, one K step
    (synth.LmHead("one_row", 9, 1, 128, 17, 1), None),         # one row, 17 columns
    (synth.LmHead("uneven", 10, 513, 192, 3000, 5), [0, 1, 300, 301, 2000, 3000]),  # one-column shards
    (synth.LmHead("deep", 11, 256, 8192, 2000, 2), None),      # the pages' hidden size
    (synth.LmHead("many_waves", 12, 1200, 128, 700, 7, ignore_frac=0.1), None),  # more M tiles than one wave
])
def test_lmhead_parity(m, vs):
    _check(m, vs)


def test_lmhead_padded_row_strides():
    _check(synth.LmHead("padded", 13, 200, 256, 1500, 3), pad_x=64, pad_w=128)


@pytest.mark.parametrize("reduction", ["sum", "none"])
def test_lmhead_reductions(reduction):
    _check(synth.LmHead("red", 14, 160, 128, 900, 2, ignore_frac=0.1), reduction=reduction)


def test_lmhead_bad_and_ignored_targets():
    m = synth.LmHead("bad", 15, 140, 64, 600, 3)
    y = synth.lmhead_meta(m).targets.copy()
    y[[0, 77]] = -100
    y[5] = 600          # one past the vocabulary
    y[6] = -3
    rows, loss = _check(m, targets=y)
    assert np.isnan(loss)


def test_lmhead_deterministic():
    m = synth.LmHead("det", 16, 300, 256, 3000, 4)
    a = _check(m)
    b = _check(m)
    np.testing.assert_array_equal(a[0], b[0])
    assert a[1] == b[1]


def test_lmhead_full_size_sampled_rows():
    """The pages' head (s = 8192, h = 8192, V = 128256, t = 8) in the launch
    configuration bench.py times, checked on sampled rows.  The 1.05e9
    weights come from the generator's device twin: a random sample of them is
    first checked against the host generator, then the sampled rows' logits
    are formed in fp64 from the read-back weights."""
    m = synth.LMHEADS["lmhead_s8192_h8192_v128256"]
    vs = synth.even_vocab_start(m.V, m.t)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs)
    y = torch.from_numpy(meta.targets).cuda()
    rl = torch.empty(m.s, dtype=torch.float32, device="cuda")
    loss, wk = vpce.vpce_lmhead_forward(x, ws, y, vs, row_loss_out=rl)
    assert vpce.vpce_read_error_flag(wk) == 0
    got = rl.cpu().numpy().astype(np.float64)
    assert abs(float(loss) - got.mean()) <= 1e-6 * abs(got.mean())

    rng = np.random.default_rng(7)
    w_host = [w.view(torch.int16).cpu().numpy().view(np.uint16) for w in ws]
    for i in range(m.t):
        pick = rng.integers(0, vs[i + 1] - vs[i], size=64)
        ref = synth.dense_host(m.seed, synth.STREAM_WEIGHT, vs[i] + pick, m.h, m.sigma_w)
        # the device generator's float64 log/cos may differ from the host's in
        # the last bit, which moves a stored value by at most one bf16 ulp
        diff = np.abs(w_host[i][pick].astype(np.int64) - ref.astype(np.int64))
        assert diff.max() <= 1 and np.count_nonzero(diff) <= 2
    rows = np.concatenate([[0, m.s - 1], rng.integers(1, m.s - 1, size=6)])
    xh = synth.dense_host(m.seed, synth.STREAM_HIDDEN, rows, m.h, m.sigma_x)
    z = O.lmhead_logits(xh, w_host, vs)
    ref = O.cross_entropy(z, meta.targets[rows], m.ignore_index, n_valid=int(np.sum(meta.targets != m.ignore_index)))
    bound = _row_bound(xh, w_host, m.h)
    err = np.abs(got[rows] - ref["row_loss"])
    assert np.all(err <= bound), (err, bound)


# ---------------------------------------------------------------- backward
def _bwd_bound(dz, mat, ref, K):
    """dZ rounded to bf16 (8 significant bits: unit roundoff 2^-8), the
    recomputed logits' error carried through exp (under 2^-11 for h <= 8192,
    from the bound above), fp32 accumulation over K terms in 16-term MMA
    steps, and, for bf16 outputs, the final rounding (2^-8 of the result)."""
    eps = 2.0 ** -8 + 2.0 ** -11 + (K / 16) * 2.0 ** -24
    a = eps * (np.abs(dz) @ np.abs(mat))
    return a + 2.0 ** -8 * (np.abs(ref) + a) + 1e-30


def _padded_ld(V):
    # each shard's columns padded to a multiple of 8, at most 64 shards
    return (V + 7) // 8 * 8 + 8 * 64


def _bwd_workspace(V, h, rows):
    """Backward workspace sized for chunks of `rows` rows (forces several
    chunks): the chunk's bf16 dZ, rows padded per shard."""
    r256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    return torch.empty(r256(rows * _padded_ld(V) * 2), dtype=torch.uint8, device="cuda")


def _train_workspace(s, V, h, rows):
    """vpce_lmhead_forward_backward workspace for chunks of `rows` rows:
    header, logsumexp and row losses of the batch, then per chunk the column
    groups' partials, target logits, fp32 logits and bf16 dZ (rows padded per
    shard)."""
    r256 = lambda n: (n + 255) // 256 * 256  # noqa: E731
    ld = _padded_ld(V)
    size = (256 + 2 * r256(4 * s) + r256(8 * 256 * rows) + r256(4 * rows) + r256(4 * rows * ld)
            + r256(2 * rows * ld))
    return torch.empty(size, dtype=torch.uint8, device="cuda")


def _check_backward(m, vs=None, *, reduction="mean", grad=1.0, grad_rows=None, chunk_rows=None, fused=False):
    """dX and dW against the oracle; with fused, through
    vpce_lmhead_forward_backward, whose row losses and loss are checked as
    the forward's are."""
    vs = synth.even_vocab_start(m.V, m.t) if vs is None else list(vs)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs)
    y = torch.from_numpy(meta.targets).cuda()
    rl = torch.full((m.s,), -7.0, dtype=torch.float32, device="cuda")
    gw0 = [torch.full((w.shape[0], m.h), 0.5, dtype=torch.float32, device="cuda") for w in ws]
    gr = torch.from_numpy(np.asarray(grad_rows, dtype=np.float32)).cuda() if grad_rows is not None else None
    if fused:
        loss_t = torch.full((), -7.0, dtype=torch.float32, device="cuda")
        twk = _train_workspace(m.s, m.V, m.h, chunk_rows) if chunk_rows else None
        _, dx, dw = vpce.vpce_lmhead_forward_backward(x, ws, y, vs, ignore_index=m.ignore_index, reduction=reduction,
                                                      grad_output=grad, grad_rows=gr, loss_out=loss_t,
                                                      row_loss_out=rl, grad_weight_shards=gw0, workspace=twk)
    else:
        _, fwk = vpce.vpce_lmhead_forward(x, ws, y, vs, ignore_index=m.ignore_index, reduction=reduction,
                                          row_loss_out=rl)
        bwk = _bwd_workspace(m.V, m.h, chunk_rows) if chunk_rows else None
        dx, dw = vpce.vpce_lmhead_backward(x, ws, y, fwk, vs, ignore_index=m.ignore_index, grad_output=grad,
                                           grad_rows=gr, grad_weight_shards=gw0, workspace=bwk)
    torch.cuda.synchronize()
    xh, wh = _host(m, vs)
    if fused:
        z = O.lmhead_logits(xh, wh, vs)
        ref = O.cross_entropy(z, meta.targets, m.ignore_index, reduction=reduction)
        got_rows = rl.cpu().numpy().astype(np.float64)
        valid = ref["valid"]
        bound = _row_bound(xh, wh, m.h)
        assert np.all(np.abs(got_rows - ref["row_loss"])[valid] <= bound[valid])
        assert np.all(got_rows[meta.targets == m.ignore_index] == 0.0)
        exp_loss = ref["loss"] if np.ndim(ref["loss"]) == 0 else float(ref["row_loss"].sum())
        got_loss = float(loss_t.item())
        assert abs(got_loss - exp_loss) <= LOSS_RTOL * abs(exp_loss), (got_loss, exp_loss)
    if grad_rows is not None:
        ref_x, ref_w, dz = O.lmhead_backward(xh, wh, vs, meta.targets, m.ignore_index,
                                             grad=np.asarray(grad_rows, dtype=np.float64), reduction="none")
    else:
        ref_x, ref_w, dz = O.lmhead_backward(xh, wh, vs, meta.targets, m.ignore_index, grad=grad,
                                             reduction=reduction)
    got_x = O.widen(dx.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    W = np.concatenate([O.widen(w, "bf16") for w in wh])
    bx = _bwd_bound(dz, W, ref_x, m.V)
    assert np.all(np.abs(got_x - ref_x) <= bx), np.max(np.abs(got_x - ref_x) / bx)
    X = O.widen(xh, "bf16")
    for i in range(len(vs) - 1):
        got_w = dw[i].cpu().numpy().astype(np.float64) - 0.5
        dzi = dz[:, vs[i]:vs[i + 1]]
        # plus one fp32 rounding of the accumulation onto 0.5 per row chunk
        rows = chunk_rows or 8192
        chunks = (m.s + rows - 1) // rows
        bw = _bwd_bound(dzi.T, X, np.zeros_like(ref_w[i]), min(m.s, rows)) + chunks * 2.0 ** -24 * (0.5 + np.abs(ref_w[i]))
        assert np.all(np.abs(got_w - ref_w[i]) <= bw), (i, np.max(np.abs(got_w - ref_w[i]) / bw))


@pytest.mark.parametrize("m,vs", [
    (synth.LMHEADS["lmhead_s300_h512_v5000"], None),                    # ragged tiles, ignored rows
    (synth.LmHead("bwd_chunks", 17, 1200, 128, 700, 7, ignore_frac=0.1), None),  # several M tiles, one chunk
    (synth.LmHead("bwd_uneven", 18, 130, 64, 600, 3), [0, 1, 300, 600]),  # one-column shard
])
def test_lmhead_backward_parity(m, vs):
    _check_backward(m, vs)


def test_lmhead_backward_sum_and_per_row_gradients():
    m = synth.LmHead("bwd_red", 19, 200, 128, 900, 2, ignore_frac=0.1)
    _check_backward(m, reduction="sum", grad=0.75)
    g = np.random.default_rng(2).normal(size=m.s).astype(np.float32)
    g[::9] = 0.0
    _check_backward(m, reduction="none", grad_rows=g)


def test_lmhead_backward_small_workspace_chunks():
    # a workspace for 128-row chunks: 1200 rows run as 10 chunks, dW accumulated across them
    _check_backward(synth.LmHead("bwd_small_ws", 22, 1200, 128, 700, 7, ignore_frac=0.1), chunk_rows=128)


# ------------------------------------------------ forward and backward in one call
@pytest.mark.parametrize("m,vs", [
    (synth.LMHEADS["lmhead_s300_h512_v5000"], None),                    # ragged tiles, ignored rows
    (synth.LmHead("fb_chunks", 23, 1200, 128, 700, 7, ignore_frac=0.1), None),   # several M tiles
    (synth.LmHead("fb_uneven", 24, 130, 64, 601, 3), [0, 1, 300, 601]),  # one-column shard, odd V
    (synth.LmHead("fb_deep", 25, 256, 8192, 2000, 2), None),             # the pages' hidden size
])
def test_lmhead_forward_backward_parity(m, vs):
    _check_backward(m, vs, fused=True)


def test_lmhead_forward_backward_sum_and_per_row_gradients():
    m = synth.LmHead("fb_red", 26, 200, 128, 900, 2, ignore_frac=0.1)
    _check_backward(m, reduction="sum", grad=0.75, fused=True)
    g = np.random.default_rng(3).normal(size=m.s).astype(np.float32)
    g[::7] = 0.0
    _check_backward(m, reduction="none", grad_rows=g, fused=True)


def test_lmhead_forward_backward_small_workspace_chunks():
    # 128-row chunks: 1200 rows as 10 chunks; the loss is the whole batch's
    _check_backward(synth.LmHead("fb_small_ws", 27, 1200, 128, 700, 7, ignore_frac=0.1), chunk_rows=128,
                    fused=True)


def test_lmhead_forward_backward_matches_two_calls():
    """The one-call step against vpce_lmhead_forward + vpce_lmhead_backward on
    the same inputs: row losses within the forward's bound, gradients within
    a few bf16 steps (the logsumexp's column grouping may differ)."""
    m = synth.LmHead("fb_vs_two", 28, 500, 256, 3000, 4, ignore_frac=0.05)
    vs = synth.even_vocab_start(m.V, m.t)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs)
    y = torch.from_numpy(meta.targets).cuda()
    rl1 = torch.empty(m.s, dtype=torch.float32, device="cuda")
    rl2 = torch.empty(m.s, dtype=torch.float32, device="cuda")
    l1, dx1, dw1 = vpce.vpce_lmhead_forward_backward(x, ws, y, vs, ignore_index=m.ignore_index, row_loss_out=rl1)
    l2, fwk = vpce.vpce_lmhead_forward(x, ws, y, vs, ignore_index=m.ignore_index, row_loss_out=rl2)
    dx2, dw2 = vpce.vpce_lmhead_backward(x, ws, y, fwk, vs, ignore_index=m.ignore_index)
    torch.cuda.synchronize()
    assert torch.allclose(rl1, rl2, rtol=0, atol=1e-5)
    assert abs(float(l1) - float(l2)) <= 1e-6 * abs(float(l2))
    # an element of dZ may round to the neighbouring bf16 value: 2^-8 of a
    # term, so a few bf16 steps of the largest result at most
    assert torch.allclose(dx1.float(), dx2.float(), rtol=2 ** -7, atol=2 ** -7 * float(dx2.float().abs().max()))
    for a, b in zip(dw1, dw2):
        assert torch.allclose(a, b, rtol=2 ** -7, atol=2 ** -7 * float(b.abs().max()))


def test_lmhead_backward_ragged_hidden_and_many_shards():
    # h = 320: the second N tile of dX and dW holds 64 valid columns; V and the
    # rows are ragged; ten shards of unequal width
    m = synth.LmHead("bwd_ragged_h", 29, 333, 320, 1337, 10, ignore_frac=0.05)
    _check_backward(m)
    _check_backward(m, fused=True)


def _strided_outputs(m, ws, pad_x, pad_w, off_x=0):
    """dX and dW outputs as views of larger buffers: row strides h + pad, and
    dX starting off_x elements past a 16-byte boundary (element stores)."""
    base = torch.zeros(m.s * (m.h + pad_x) + off_x, dtype=torch.bfloat16, device="cuda")
    gx = base[off_x:].view(m.s, m.h + pad_x)[:, :m.h]
    gw = []
    for w in ws:
        b = torch.full((w.shape[0], m.h + pad_w), 0.5, dtype=torch.float32, device="cuda")
        gw.append(b[:, :m.h])
    return gx, gw


@pytest.mark.parametrize("off_x", [0, 1])
def test_lmhead_backward_strided_outputs(off_x):
    m = synth.LmHead("bwd_strided", 30, 200, 192, 900, 3, ignore_frac=0.1)
    vs = synth.even_vocab_start(m.V, m.t)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs)
    y = torch.from_numpy(meta.targets).cuda()
    gx, gw = _strided_outputs(m, ws, pad_x=24, pad_w=12, off_x=off_x)
    _, fwk = vpce.vpce_lmhead_forward(x, ws, y, vs, ignore_index=m.ignore_index)
    vpce.vpce_lmhead_backward(x, ws, y, fwk, vs, ignore_index=m.ignore_index, grad_hidden=gx,
                              grad_weight_shards=gw)
    torch.cuda.synchronize()
    xh, wh = _host(m, vs)
    ref_x, ref_w, dz = O.lmhead_backward(xh, wh, vs, meta.targets, m.ignore_index)
    got_x = O.widen(gx.contiguous().view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    W = np.concatenate([O.widen(w, "bf16") for w in wh])
    bx = _bwd_bound(dz, W, ref_x, m.V)
    assert np.all(np.abs(got_x - ref_x) <= bx)
    X = O.widen(xh, "bf16")
    for i in range(m.t):
        got_w = gw[i].cpu().numpy().astype(np.float64) - 0.5
        bw = _bwd_bound(dz[:, vs[i]:vs[i + 1]].T, X, np.zeros_like(ref_w[i]), m.s) + 2.0 ** -24 * (0.5 + np.abs(ref_w[i]))
        assert np.all(np.abs(got_w - ref_w[i]) <= bw)
    # the padding columns are neither read nor written
    assert torch.all(gw[0].as_strided((gw[0].shape[0], 12), (m.h + 12, 1), m.h) == 0.5)


def test_lmhead_train_full_size_sampled_rows():
    """The one-call training step on the pages' head (s = 8192, h = 8192,
    V = 128256, t = 8) in the configuration bench.py times: sampled rows of
    the loss and of dX against the oracle, formed in fp64 from the hidden
    states and head read back from the device; every row of dW is summed
    over the vocabulary, which is zero for exact arithmetic (each valid row of
    dZ sums to zero), to within the rounding of dZ."""
    m = synth.LMHEADS["lmhead_s8192_h8192_v128256"]
    vs = synth.even_vocab_start(m.V, m.t)
    meta = synth.lmhead_meta(m)
    x, ws = synth.lmhead_device(m, vs)
    y = torch.from_numpy(meta.targets).cuda()
    rl = torch.empty(m.s, dtype=torch.float32, device="cuda")
    loss, dx, dw = vpce.vpce_lmhead_forward_backward(x, ws, y, vs, ignore_index=m.ignore_index, row_loss_out=rl)
    torch.cuda.synchronize()
    n_valid = int(np.sum(meta.targets != m.ignore_index))
    got_rl = rl.cpu().numpy().astype(np.float64)
    assert abs(float(loss) - got_rl.sum() / n_valid) <= 1e-6 * abs(float(loss))
    rng = np.random.default_rng(11)
    rows = np.concatenate([[0, m.s - 1], rng.integers(1, m.s - 1, size=4)])
    xr = x[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    w_host = [w.view(torch.int16).cpu().numpy().view(np.uint16) for w in ws]
    z = O.lmhead_logits(xr, w_host, vs)
    ref = O.cross_entropy(z, meta.targets[rows], m.ignore_index, n_valid=n_valid)
    assert np.all(np.abs(got_rl[rows] - ref["row_loss"]) <= _row_bound(xr, w_host, m.h))
    dz = O.dlogits(z, meta.targets[rows], m.ignore_index, n_valid=n_valid)
    ref_x = np.zeros((len(rows), m.h))
    bound = np.zeros((len(rows), m.h))
    eps = 2.0 ** -8 + 2.0 ** -11 + (m.V / 16) * 2.0 ** -24
    for i in range(m.t):
        Wi = O.widen(w_host[i], "bf16")
        dzi = dz[:, vs[i]:vs[i + 1]]
        ref_x += dzi @ Wi
        bound += eps * (np.abs(dzi) @ np.abs(Wi))
    bound += 2.0 ** -8 * (np.abs(ref_x) + bound)
    got_x = O.widen(dx[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    assert np.all(np.abs(got_x - ref_x) <= bound), np.max(np.abs(got_x - ref_x) / bound)
    # sum over the vocabulary of dW_i[v, :] = sum_r (sum_v dZ[r, v]) X[r, :]: zero for
    # exact arithmetic.  A valid row of dZ has sum_v |dZ[r, v]| <= 2 / n_valid, so its
    # bf16 rounding (2^-9 relative) moves the row sum by at most 2^-8 / n_valid; the
    # fp32 accumulation of dW over the 8192 rows (512 MMA steps of 16) adds at most
    # 512 * 2^-24 of the same sum, 2^-14 / n_valid
    col = sum(d.double().sum(dim=0) for d in dw).cpu().numpy()
    xs = np.abs(x.float().cpu().numpy().astype(np.float64)).sum(axis=0)
    assert np.all(np.abs(col) <= (2.0 ** -8 + 2.0 ** -14) / n_valid * xs + 1e-12)
