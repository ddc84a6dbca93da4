"""The seeded input generator shared by the oracle and the CUDA path (host side)."""
import os

import numpy as np
import pytest
import torch

from vocab_sharded_lm_gb300 import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def test_splitmix64_published_vectors():
    with open(os.path.join(HERE, "golden", "splitmix64_vectors.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for seed, idx, val in rows:
        got = int(synth.splitmix64_at(np.uint64(int(seed)), np.array([int(idx)]))[0])
        assert got == int(val)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.normal(0, 3, 200000), rng.normal(0, 1e-3, 1000),
                        np.array([1.00390625, 1.01171875, -1.00390625, 65504.0, 0.0, -0.0])]).astype(np.float32)
    got = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, ref)


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_row_subsets_are_consistent(name):
    w = synth.WORKLOADS[name]
    meta = synth.row_meta(w)
    rows = np.array([0, 3, w.s - 1])
    a = synth.logits_rows(w, rows, 0, 257, meta)
    b = synth.logits_rows(w, rows[1:2], 100, 257, meta)
    np.testing.assert_array_equal(a[1, 100:257], b[0])


def test_moments_and_counts():
    for name, w in synth.WORKLOADS.items():
        meta = synth.row_meta(w)
        y = meta.targets
        n_ign = int(np.sum(y == w.ignore_index))
        assert n_ign == int(round(w.ignore_frac * w.s))
        valid = y[y != w.ignore_index]
        assert valid.min() >= 0 and valid.max() < w.V
        if w.boost_frac:
            assert int(np.sum(meta.boost_col >= 0)) == int(round(w.boost_frac * w.s))
            hit = meta.boost_col >= 0
            np.testing.assert_array_equal(meta.boost_col[hit], y[hit])
        if w.spike:
            assert np.all(meta.boost_col >= 0) and meta.boost_col.max() < w.V
        v = synth.logits_rows(w, np.array([1, 2]), 0, min(w.V, 60000), meta)
        f = v if w.dtype == "fp32" else (v.astype(np.uint32) << 16).view(np.float32)
        f = f.astype(np.float64)
        mask = np.ones_like(f, dtype=bool)
        for j, r in enumerate([1, 2]):
            if meta.boost_col[r] >= 0 and meta.boost_col[r] < f.shape[1]:
                mask[j, meta.boost_col[r]] = False
        n = int(mask.sum())
        assert abs(f[mask].mean()) < 5 * w.sigma / np.sqrt(n)
        assert abs(f[mask].std() / w.sigma - 1) < 5 / np.sqrt(2 * n)


def test_boost_lands_on_the_target_column():
    w = synth.WORKLOADS["s8192_v128256"]
    meta = synth.row_meta(w)
    r = int(np.nonzero(meta.boost_col >= 0)[0][0])
    c = int(meta.boost_col[r])
    plain = synth.RowMeta(meta.targets, np.full_like(meta.boost_col, -1), 0.0)
    a = synth.logits_rows(w, [r], c, c + 1, meta)
    b = synth.logits_rows(w, [r], c, c + 1, plain)
    fa = (a.astype(np.uint32) << 16).view(np.float32)[0, 0]
    fb = (b.astype(np.uint32) << 16).view(np.float32)[0, 0]
    assert abs((fa - fb) - 5.0) < 0.07  # one bf16 step at |z| < 16


def test_zipf_targets_follow_the_law():
    w = synth.WORKLOADS["s32768_v256000"]
    y = synth.row_meta(w).targets
    H = np.sum(np.arange(1, w.V + 1, dtype=np.float64) ** -1.1)
    for k in (0, 1, 9):
        p = (k + 1) ** -1.1 / H
        freq = np.mean(y == k)
        assert abs(freq - p) < 5 * np.sqrt(p * (1 - p) / w.s)


def test_even_vocab_start():
    assert synth.even_vocab_start(128256, 8)[1] == 16032
    vs = synth.even_vocab_start(50257, 8)
    assert vs[-1] == 50257 and max(np.diff(vs)) - min(np.diff(vs)) == 1


def test_shards_host_padding_canary():
    w = synth.WORKLOADS["tiny_s64_v1000"]
    meta = synth.row_meta(w)
    sh = synth.shards_host(w, meta, ld=512)
    assert sh[0].shape == (64, 512) and np.isnan(sh[0][:, 500:]).all()
    full = synth.shards_host(w, meta)
    np.testing.assert_array_equal(sh[1][:, :500], full[1])
