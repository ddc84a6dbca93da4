"""Pins for the fp64 oracle: closed forms, invariants, brute force and the
library routine the pages compared against.  No GPU; each test is chosen so
that a plausible slip in the oracle (a dropped max shift, a wrong sign, an
off-by-one target column, a missing 1/n_valid, a wrong rescale in the
combine, a bad bf16 widening) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O

RNG = np.random.default_rng(12345)


def _rand_case(s, V, scale=3.0, ignore=(), bad=()):
    z = RNG.normal(0.0, scale, size=(s, V))
    y = RNG.integers(0, V, size=s).astype(np.int64)
    for r in ignore:
        y[r] = -100
    for r in bad:
        y[r] = V + 3
    return z, y


# ---------------------------------------------------------------- closed forms
@pytest.mark.parametrize("V", [1, 2, 7, 1000, 128256])
@pytest.mark.parametrize("c", [0.0, -3.5, 17.25])
def test_uniform_logits_give_log_V(V, c):
    s = 5
    z = np.full((s, V), c)
    y = np.arange(s) % V
    out = O.cross_entropy(z, y)
    np.testing.assert_allclose(out["row_loss"], math.log(V), rtol=0, atol=1e-12)
    assert out["loss"] == pytest.approx(math.log(V), abs=1e-12)
    d = O.dlogits(z, y)
    expect = np.full((s, V), 1.0 / V)
    expect[np.arange(s), y] -= 1.0
    np.testing.assert_allclose(d, expect / s, rtol=0, atol=1e-15)


@pytest.mark.parametrize("V,L", [(2, 1.0), (10, 3.0), (50304, 8.0), (128256, -2.0)])
def test_single_spike_closed_form(V, L):
    # z_y = L and every other logit 0: loss = ln(1 + (V-1) e^-L)
    z = np.zeros((2, V))
    y = np.array([V - 1, 0])
    z[0, V - 1] = L
    z[1, 0] = L
    out = O.cross_entropy(z, y, reduction="none")
    expect = math.log1p((V - 1) * math.exp(-L))
    np.testing.assert_allclose(out["row_loss"], [expect, expect], rtol=1e-14)
    # the spike off the target: loss = ln(e^L + V - 1) - 0
    z2 = np.zeros((1, V))
    z2[0, 0] = L
    out2 = O.cross_entropy(z2, np.array([V - 1]), reduction="none")
    assert out2["row_loss"][0] == pytest.approx(math.log(math.exp(L) + V - 1), rel=1e-14)
    # softmax closed form in the gradient of the first row (g = 1, n_valid = 1)
    d = O.dlogits(z[:1], y[:1])
    pt = math.exp(L) / (math.exp(L) + V - 1)
    assert d[0, V - 1] == pytest.approx(pt - 1.0, rel=1e-12, abs=1e-15)
    if V > 1:
        assert d[0, 0] == pytest.approx(1.0 / (math.exp(L) + V - 1), rel=1e-12)


def test_max_shift_identity():
    # values on a 1/1024 grid so that z + 1000 is exact in fp64
    z = RNG.integers(-8192, 8192, size=(6, 3001)).astype(np.float64) / 1024.0
    y = RNG.integers(0, 3001, size=6)
    a = O.cross_entropy(z, y, reduction="none")["row_loss"]
    b = O.cross_entropy(z + 1000.0, y, reduction="none")["row_loss"]
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=0)
    np.testing.assert_allclose(O.dlogits(z, y), O.dlogits(z + 1000.0, y), rtol=0, atol=1e-15)
    # shifts large enough to overflow a naive exp must still work
    big = O.cross_entropy(z + 800.0, y, reduction="none")["row_loss"]
    assert np.all(np.isfinite(big))
    np.testing.assert_allclose(a, big, rtol=1e-13)


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("V", [1, 2, 3, 5, 8])
def test_brute_force_tiny_vocab(V):
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    z = RNG.normal(0, 4.0, size=(4, V))
    for r in range(4):
        losses = []
        for y in range(V):
            out = O.cross_entropy(z[r:r + 1], np.array([y]), reduction="none")
            losses.append(out["row_loss"][0])
            # direct, unshifted log-sum-exp in 50-digit arithmetic
            ref = mp.log(mp.fsum(mp.exp(mp.mpf(float(v))) for v in z[r])) - mp.mpf(float(z[r, y]))
            assert abs(out["row_loss"][0] - float(ref)) <= 1e-14 * max(1.0, abs(float(ref)))
        # probabilities over all possible targets sum to one
        assert math.fsum(math.exp(-l) for l in losses) == pytest.approx(1.0, abs=1e-14)


# ---------------------------------------------------------------- library routine
@pytest.mark.parametrize("s,V,ignore", [(64, 1000, ()), (33, 517, (0, 5, 32)), (16, 50304, (3,))])
@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_matches_torch_cross_entropy_fp64(s, V, ignore, reduction):
    z, y = _rand_case(s, V, ignore=ignore)
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    yt = torch.tensor(y)
    ref = torch.nn.functional.cross_entropy(zt, yt, ignore_index=-100, reduction=reduction)
    out = O.cross_entropy(z, y, reduction=reduction)
    np.testing.assert_allclose(np.asarray(out["loss"]), ref.detach().numpy(), rtol=1e-12, atol=1e-13)
    if reduction != "none":
        g = 0.75
        (ref * g).backward()
        d = O.dlogits(z, y, grad=g, reduction=reduction)
    else:
        # one upstream gradient per row, of both signs, some zero
        g = RNG.normal(0.0, 1.0, size=s)
        g[::5] = 0.0
        ref.backward(torch.tensor(g))
        d = O.dlogits(z, y, grad=g, reduction="none")
    np.testing.assert_allclose(d, zt.grad.numpy(), rtol=1e-12, atol=1e-15)


def test_matches_torch_with_large_logits():
    z, y = _rand_case(8, 2000, scale=30.0)
    z[:, 7] += 500.0
    ref = torch.nn.functional.cross_entropy(torch.tensor(z), torch.tensor(y))
    assert O.cross_entropy(z, y)["loss"] == pytest.approx(float(ref), rel=1e-13)


# ---------------------------------------------------------------- gradient
def test_gradient_by_central_differences():
    s, V = 3, 6
    z, y = _rand_case(s, V, scale=1.5, ignore=(1,))
    d = O.dlogits(z, y, grad=1.0)
    h = 1e-6
    fd = np.zeros_like(z)
    for r in range(s):
        for k in range(V):
            zp = z.copy()
            zm = z.copy()
            zp[r, k] += h
            zm[r, k] -= h
            fd[r, k] = (O.cross_entropy(zp, y)["loss"] - O.cross_entropy(zm, y)["loss"]) / (2 * h)
    np.testing.assert_allclose(d, fd, rtol=0, atol=1e-8)


def test_per_row_gradient_by_central_differences():
    """'none': d/dz of sum_r g_r * CE_r, differentiated numerically."""
    s, V = 4, 5
    z, y = _rand_case(s, V, scale=1.5, ignore=(2,))
    g = np.array([0.5, -1.25, 7.0, 2.0])
    d = O.dlogits(z, y, grad=g, reduction="none")
    h = 1e-6
    fd = np.zeros_like(z)
    for r in range(s):
        for k in range(V):
            zp = z.copy()
            zm = z.copy()
            zp[r, k] += h
            zm[r, k] -= h
            lp = O.cross_entropy(zp, y, reduction="none")["loss"]
            lm = O.cross_entropy(zm, y, reduction="none")["loss"]
            fd[r, k] = float(np.dot(g, lp - lm)) / (2 * h)
    np.testing.assert_allclose(d, fd, rtol=0, atol=5e-8)
    assert np.all(d[2] == 0.0)


def test_gradient_rows_sum_to_zero_and_ignored_rows_zero():
    z, y = _rand_case(40, 3000, ignore=(2, 9, 39))
    d = O.dlogits(z, y, grad=2.0)
    n = 37
    np.testing.assert_allclose(d.sum(axis=1), 0.0, atol=1e-12 * 3000 / n)
    assert np.all(d[[2, 9, 39]] == 0.0)
    # the only negative entry of a valid row sits on its target
    for r in range(40):
        if y[r] >= 0:
            assert np.argmin(d[r]) == y[r]
            assert np.sum(d[r] < 0) == 1


# ---------------------------------------------------------------- special cases
def test_all_rows_ignored_gives_nan_and_zero_gradient():
    z = RNG.normal(size=(5, 11))
    y = np.full(5, -100)
    out = O.cross_entropy(z, y)
    assert math.isnan(out["loss"]) and out["n_valid"] == 0
    assert np.all(O.dlogits(z, y) == 0.0)
    ref = torch.nn.functional.cross_entropy(torch.tensor(z), torch.tensor(y))
    assert math.isnan(float(ref))


def test_empty_batch():
    z = np.zeros((0, 9))
    y = np.zeros(0, dtype=np.int64)
    out = O.cross_entropy(z, y)
    assert math.isnan(out["loss"]) and out["n_valid"] == 0
    assert O.dlogits(z, y).shape == (0, 9)


def test_out_of_range_target_flags_and_poisons_row():
    z, y = _rand_case(6, 50, bad=(4,))
    out = O.cross_entropy(z, y)
    assert out["error_flag"] == 1
    assert math.isnan(out["loss"])
    assert math.isnan(out["row_loss"][4]) and np.isfinite(out["row_loss"][:4]).all()
    d = O.dlogits(z, y)
    assert np.isnan(d[4]).all() and np.isfinite(d[:4]).all()
    y2 = y.copy()
    y2[4] = -1  # negative but not ignore_index
    assert O.cross_entropy(z, y2)["error_flag"] == 1


def test_sampled_rows_use_batch_n_valid():
    z, y = _rand_case(30, 400, ignore=(1, 2))
    full = O.dlogits(z, y)
    rows = np.array([0, 7, 29])
    part = O.dlogits(z[rows], y[rows], n_valid=28)
    np.testing.assert_allclose(part, full[rows], rtol=0, atol=0)


# ---------------------------------------------------------------- bf16 widening
# ---------------------------------------------------------------- LM head
def _bf16(a):
    return torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_lmhead_one_hot_rows_select_weight_columns():
    """X rows that are unit vectors e_k pick column k of the head exactly."""
    rng = np.random.default_rng(3)
    h, V, s = 64, 37, 5
    W = _bf16(rng.normal(size=(V, h)))
    ks = np.array([0, 5, 63, 17, 5])
    x = np.zeros((s, h), dtype=np.float32)
    x[np.arange(s), ks] = 1.0
    vs = [0, 10, 37]
    z = O.lmhead_logits(_bf16(x), [W[:10], W[10:]], vs)
    np.testing.assert_array_equal(z, O.widen(W, "bf16")[:, ks].T)


def test_lmhead_matches_torch_linear_and_cross_entropy():
    rng = np.random.default_rng(4)
    s, h, V = 40, 128, 300
    x = _bf16(rng.normal(size=(s, h)))
    W = _bf16(rng.normal(0.0, 3.0 / np.sqrt(h), size=(V, h)))
    y = rng.integers(0, V, size=s)
    y[[3, 11]] = -100
    vs = [0, 100, 256, 300]
    z = O.lmhead_logits(x, [W[vs[i]:vs[i + 1]] for i in range(3)], vs)
    xt = torch.tensor(O.widen(x, "bf16"))
    wt = torch.tensor(O.widen(W, "bf16"))
    zt = torch.nn.functional.linear(xt, wt)
    np.testing.assert_allclose(z, zt.numpy(), rtol=1e-13, atol=1e-13)
    ref = torch.nn.functional.cross_entropy(zt, torch.tensor(y), ignore_index=-100)
    assert O.cross_entropy(z, y)["loss"] == pytest.approx(float(ref), rel=1e-12)
    # the split does not change the logits
    z1 = O.lmhead_logits(x, [W], [0, V])
    np.testing.assert_allclose(z, z1, rtol=1e-14, atol=1e-14)


def test_lmhead_backward_matches_torch_autograd():
    rng = np.random.default_rng(8)
    s, h, V = 30, 64, 200
    x = _bf16(rng.normal(size=(s, h)))
    W = _bf16(rng.normal(0.0, 3.0 / np.sqrt(h), size=(V, h)))
    y = rng.integers(0, V, size=s)
    y[[2, 9]] = -100
    vs = [0, 64, 65, 200]
    shards = [W[vs[i]:vs[i + 1]] for i in range(3)]
    for red, g in (("mean", 1.5), ("sum", 0.5)):
        xt = torch.tensor(O.widen(x, "bf16"), requires_grad=True)
        wt = torch.tensor(O.widen(W, "bf16"), requires_grad=True)
        loss = torch.nn.functional.cross_entropy(torch.nn.functional.linear(xt, wt), torch.tensor(y),
                                                 ignore_index=-100, reduction=red)
        (loss * g).backward()
        dX, dW, _ = O.lmhead_backward(x, shards, vs, y, grad=g, reduction=red)
        np.testing.assert_allclose(dX, xt.grad.numpy(), rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(np.concatenate(dW), wt.grad.numpy(), rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- embedding
def test_embedding_forward_matches_torch_embedding():
    rng = np.random.default_rng(5)
    V, h, s = 300, 24, 50
    E = _bf16(rng.normal(size=(V, h)))
    vs = [0, 7, 150, 300]
    ids = rng.integers(0, V, size=s)
    ids[:4] = [0, 6, 7, 299]           # shard edges
    out, bad = O.embedding_forward([E[vs[i]:vs[i + 1]] for i in range(3)], vs, ids)
    ref = torch.nn.functional.embedding(torch.tensor(ids), torch.tensor(O.widen(E, "bf16")))
    np.testing.assert_array_equal(out, ref.numpy())
    assert not bad


def test_embedding_forward_out_of_range_ids_give_zero_rows():
    E = _bf16(np.arange(40, dtype=np.float32).reshape(10, 4) + 1.0)
    out, bad = O.embedding_forward([E[:3], E[3:]], [0, 3, 10], np.array([2, -1, 10, 3, 1000]))
    assert bad
    np.testing.assert_array_equal(out[[1, 2, 4]], 0.0)
    np.testing.assert_array_equal(out[0], O.widen(E, "bf16")[2])
    np.testing.assert_array_equal(out[3], O.widen(E, "bf16")[3])


def test_embedding_backward_matches_torch_autograd():
    rng = np.random.default_rng(6)
    V, h, s = 40, 8, 200               # many repeated ids
    vs = [0, 13, 14, 40]
    ids = rng.integers(0, V, size=s)
    g = rng.normal(size=(s, h))
    E = torch.zeros((V, h), dtype=torch.float64, requires_grad=True)
    torch.nn.functional.embedding(torch.tensor(ids), E).backward(torch.tensor(g))
    got = O.embedding_backward(g, ids, vs, h)
    np.testing.assert_allclose(np.concatenate(got), E.grad.numpy(), rtol=1e-13, atol=1e-13)


def test_embedding_backward_drops_out_of_range_ids():
    g = np.ones((3, 2))
    got = O.embedding_backward(g, np.array([-5, 1, 4]), [0, 2, 4], 2)
    np.testing.assert_array_equal(got[0], [[0, 0], [1, 1]])
    np.testing.assert_array_equal(got[1], [[0, 0], [0, 0]])


def test_bf16_widening_exact():
    bits = np.array([0x3F80, 0xC000, 0x4049, 0x0000, 0x8000, 0x7F7F, 0x0001, 0xBF00], dtype=np.uint16)
    got = O.widen(bits, "bf16")
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 3.140625 and got[7] == -0.5
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(got, ref)
    allbits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    finite = ((allbits >> 7) & 0xFF) != 0xFF
    a = O.widen(allbits[finite], "bf16")
    b = torch.from_numpy(allbits[finite].view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- sharded combine
@pytest.mark.parametrize("V", [1000, 50304, 128256, 152064, 256000])
@pytest.mark.parametrize("t", [1, 2, 4, 8, 16])
def test_pages_combine_equals_unsharded(V, t):
    s = 6
    z, y = _rand_case(s, V, scale=3.0, ignore=(2,))
    z[0, 5] += 25.0          # a spike in shard 0: the other shards must rescale
    z[1, V - 1] += 25.0      # a spike in the last shard
    vs = [(i * V) // t for i in range(t + 1)]
    partials = [O.shard_partials(z[:, vs[i]:vs[i + 1]], y, vs[i], vs[i + 1]) for i in range(t)]
    lse, row_loss, mean = O.combine_sharded(partials, y, V)
    ref = O.cross_entropy(z, y)
    valid = ref["valid"]
    np.testing.assert_allclose(lse[valid], ref["lse"][valid], rtol=1e-12)
    np.testing.assert_allclose(row_loss, ref["row_loss"], rtol=1e-12, atol=1e-12)
    assert mean == pytest.approx(ref["loss"], rel=1e-12)


@pytest.mark.parametrize("t,ranks", [(2, 1), (4, 2), (8, 2), (8, 4), (16, 8)])
def test_fold_equals_partials_of_the_union(t, ranks):
    # a rank's t / ranks shards folded to one pair per row is the pair of its
    # whole column range computed directly: max over the union, then the sum
    # of exp(z - max) over the union (no partials involved)
    V, s = 4000, 7
    z, y = _rand_case(s, V, scale=3.0)
    z[0, 3] += 30.0            # a spike in the first shard of rank 0
    z[1, V // ranks - 1] += 30.0  # a spike in the last shard of rank 0
    z[2, V - 2] += 30.0        # a spike in the last rank's last shard
    vs = [(i * V) // t for i in range(t + 1)]
    per = t // ranks
    folded = []
    for r in range(ranks):
        lo, hi = vs[r * per], vs[(r + 1) * per]
        parts = [O.shard_partials(z[:, vs[i]:vs[i + 1]], y, vs[i], vs[i + 1]) for i in range(r * per, (r + 1) * per)]
        M, S = O.fold_partials(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        block = z[:, lo:hi]
        M_ref = block.max(axis=1)
        S_ref = np.array([math.fsum(np.exp(block[k] - M_ref[k])) for k in range(s)])
        np.testing.assert_array_equal(M, M_ref)
        np.testing.assert_allclose(S, S_ref, rtol=1e-13)
        tgt = sum(p[2] for p in parts)
        folded.append((M, S, tgt))
    # the ranks' folded pairs combined as the pages combine the cards' pairs
    lse, row_loss, mean = O.combine_sharded(folded, y, V)
    ref = O.cross_entropy(z, y)
    np.testing.assert_allclose(lse, ref["lse"], rtol=1e-12)
    assert mean == pytest.approx(ref["loss"], rel=1e-12)


def test_fold_of_one_card_is_the_identity():
    m = np.array([[1.5, -2.0, 40.0]])
    se = np.array([[3.0, 1.0, 7.25]])
    M, S = O.fold_partials(m, se)
    np.testing.assert_array_equal(M, m[0])
    np.testing.assert_array_equal(S, se[0])


def test_assemble_roundtrip_with_padding():
    z = RNG.normal(size=(4, 23)).astype(np.float32)
    vs = [0, 5, 6, 23]
    shards = []
    for i in range(3):
        w = vs[i + 1] - vs[i]
        buf = np.full((4, w + 3), np.nan, dtype=np.float32)
        buf[:, :w] = z[:, vs[i]:vs[i + 1]]
        shards.append(buf)
    full = O.assemble(shards, vs, "fp32")
    np.testing.assert_array_equal(full, z.astype(np.float64))
    back = O.split_columns(full, vs)
    assert [b.shape[1] for b in back] == [5, 1, 17]
