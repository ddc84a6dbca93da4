"""Seeded synthetic inputs for vocab-parallel cross-entropy.

This module is the ONLY thing the CUDA path and the oracle share: it draws the
logits and the row metadata (targets, ignored rows, boosted rows, spike
columns).  It holds none of the loss arithmetic.

Generator (published definitions, restated):

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014): output ``n`` (0-based) of the generator seeded with
  ``key`` is ``mix(key + (n + 1) * GAMMA) mod 2**64``, with ``mix`` the
  xor-shift-multiply finaliser of that paper.  It is counter based, so any
  element can be drawn on its own, on the host or on the device, with integer
  arithmetic only (bit exact on both).
* Box-Muller (Box & Muller, 1958), cosine branch, in float64:
  ``n = sqrt(-2 ln u1) * cos(2 pi u2)`` with ``u1 = (a + 1) / 2**53`` in (0, 1]
  and ``u2 = b / 2**53`` in [0, 1), ``a``/``b`` the top 53 bits of outputs
  ``2g`` and ``2g + 1`` of the value stream for the element's global index
  ``g = r * V + c``.  The stored logit is ``float32(sigma * n + boost)``
  (float64 multiply, then add, then one round-to-nearest-even to binary32) and,
  for bf16 logits, that binary32 rounded to nearest-even bfloat16.

The device twin of the element generator lives in ``csrc/synth_gen.cu``
(library ``libvpce_synth.so``); the float64 ``log``/``cos`` of the two sides may
differ in the last bit, so a stored value can (rarely) differ by one ulp.  Row
metadata is drawn only here, on the host, and uploaded.

Workloads: the five configurations the method is exercised on, with the
shapes, value distributions and row structure of the LM-head cross-entropy:
the pages' Llama-3-70B head (V = 128256, t = 8, 16032 columns per card) plus
smaller and larger vocabularies.
"""
from __future__ import annotations

import dataclasses
import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_TWO_PI = 6.283185307179586  # float64 nearest to 2*pi
_INV_2_53 = 1.0 / 9007199254740992.0

# stream numbers (outputs of the generator seeded with the workload seed)
STREAM_VALUES = 0
STREAM_TARGETS = 1
STREAM_IGNORE = 2
STREAM_BOOST = 3
STREAM_SPIKE = 4


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64_at(key, n) -> np.ndarray:
    """Output number ``n`` (array, 0-based) of SplitMix64 seeded with ``key``."""
    with np.errstate(over="ignore"):
        n = np.asarray(n, dtype=np.uint64)
        return _mix(np.uint64(key) + (n + np.uint64(1)) * GAMMA)


def stream_key(seed: int, stream: int) -> np.uint64:
    return np.uint64(splitmix64_at(np.uint64(seed), np.uint64(stream)))


def uniform_int(h: np.ndarray, n: int) -> np.ndarray:
    """Map 64-bit hashes to [0, n) by the top 32 bits (multiply-shift)."""
    return ((h >> np.uint64(32)) * np.uint64(n)) >> np.uint64(32)


def _normals_from_index(key: np.uint64, g: np.ndarray) -> np.ndarray:
    g = np.asarray(g, dtype=np.uint64)
    with np.errstate(over="ignore"):
        h1 = splitmix64_at(key, g * np.uint64(2))
        h2 = splitmix64_at(key, g * np.uint64(2) + np.uint64(1))
    u1 = ((h1 >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * _INV_2_53
    u2 = (h2 >> np.uint64(11)).astype(np.float64) * _INV_2_53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(_TWO_PI * u2)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to nearest-even bfloat16; returns uint16 patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


# --------------------------------------------------------------------------
# workload recipes
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int            # 1..5; seed = 20261202 + index
    s: int                # rows (tokens)
    V: int                # vocabulary
    t: int                # shards
    dtype: str            # 'fp32' | 'bf16'
    sigma: float          # logits ~ N(0, sigma^2)
    targets: str          # 'uniform' | 'zipf1.1'
    ignore_frac: float = 0.0
    boost_frac: float = 0.0   # rows whose target column gets +boost
    boost: float = 0.0
    spike: float = 0.0        # +spike at one uniform column of every row
    ignore_index: int = -100

    @property
    def seed(self) -> int:
        return 20261202 + self.index

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_s64_v1000", 1, 64, 1000, 2, "fp32", 1.0, "uniform"),
        Workload("s4096_v50304", 2, 4096, 50304, 4, "bf16", 2.0, "uniform", ignore_frac=0.02),
        Workload("s8192_v128256", 3, 8192, 128256, 8, "bf16", 3.0, "uniform",
                 boost_frac=0.30, boost=5.0),
        Workload("s16384_v152064", 4, 16384, 152064, 8, "fp32", 1.0, "uniform",
                 ignore_frac=0.05, spike=20.0),
        Workload("s32768_v256000", 5, 32768, 256000, 16, "bf16", 2.0, "zipf1.1"),
    ]
}
BENCH_WORKLOAD = "s8192_v128256"


def even_vocab_start(V: int, t: int) -> list[int]:
    """Shard boundaries for t shards; widths differ by at most one column
    when t does not divide V (the first V % t shards are one wider)."""
    base, extra = divmod(V, t)
    out = [0]
    for i in range(t):
        out.append(out[-1] + base + (1 if i < extra else 0))
    return out


@dataclasses.dataclass
class RowMeta:
    targets: np.ndarray      # int64[s]; ignore_index on ignored rows
    boost_col: np.ndarray    # int64[s]; global column that gets +boost_val, -1 if none
    boost_val: float


def _pick_rows(seed: int, stream: int, s: int, count: int) -> np.ndarray:
    """Exactly ``count`` distinct rows: the first ``count`` of a seeded shuffle
    (rows ordered by a 64-bit key each)."""
    keys = splitmix64_at(stream_key(seed, stream), np.arange(s, dtype=np.uint64))
    order = np.argsort(keys, kind="stable")
    return np.sort(order[:count])


def row_meta(w: Workload, s: int | None = None) -> RowMeta:
    """Targets and per-row boost columns of workload ``w`` (first ``s`` rows
    of a batch of ``s`` rows; ``s`` defaults to ``w.s``)."""
    s = w.s if s is None else s
    rows = np.arange(s, dtype=np.uint64)
    if w.targets == "uniform":
        h = splitmix64_at(stream_key(w.seed, STREAM_TARGETS), rows)
        y = uniform_int(h, w.V).astype(np.int64)
    elif w.targets == "zipf1.1":
        # truncated Zipf over ranks k = 1..V with P(k) ~ k^-1.1; token id = k-1;
        # inverse-CDF sampling with a 53-bit uniform
        k = np.arange(1, w.V + 1, dtype=np.float64)
        cdf = np.cumsum(k ** -1.1)
        cdf /= cdf[-1]
        h = splitmix64_at(stream_key(w.seed, STREAM_TARGETS), rows)
        u = (h >> np.uint64(11)).astype(np.float64) * _INV_2_53
        y = np.minimum(np.searchsorted(cdf, u, side="right"), w.V - 1).astype(np.int64)
    else:
        raise ValueError(w.targets)
    boost_col = np.full(s, -1, dtype=np.int64)
    boost_val = 0.0
    if w.boost_frac > 0:
        picked = _pick_rows(w.seed, STREAM_BOOST, s, int(round(w.boost_frac * s)))
        boost_col[picked] = y[picked]
        boost_val = w.boost
    if w.spike > 0:
        h = splitmix64_at(stream_key(w.seed, STREAM_SPIKE), rows)
        boost_col[:] = uniform_int(h, w.V).astype(np.int64)
        boost_val = w.spike
    if w.ignore_frac > 0:
        picked = _pick_rows(w.seed, STREAM_IGNORE, s, int(round(w.ignore_frac * s)))
        y = y.copy()
        y[picked] = w.ignore_index
    return RowMeta(targets=y, boost_col=boost_col, boost_val=boost_val)


def logits_rows(w: Workload, rows, col_lo: int, col_hi: int, meta: RowMeta) -> np.ndarray:
    """Stored logits of ``rows`` x global columns [col_lo, col_hi).

    Returns float32 for fp32 workloads and uint16 bfloat16 patterns for bf16.
    """
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.arange(col_lo, col_hi, dtype=np.int64)
    key = stream_key(w.seed, STREAM_VALUES)
    g = (rows[:, None].astype(np.uint64) * np.uint64(w.V) + cols[None, :].astype(np.uint64))
    v = _normals_from_index(key, g) * w.sigma
    bc = meta.boost_col[rows]
    hit = bc[:, None] == cols[None, :]
    if hit.any():
        v = np.where(hit, v + meta.boost_val, v)
    f = v.astype(np.float32)
    return f32_to_bf16_bits(f) if w.dtype == "bf16" else f


def shards_host(w: Workload, meta: RowMeta, vocab_start=None, ld=None, rows=None):
    """Host shard arrays ``[len(rows), ld_i]`` (padding columns hold a NaN
    canary).  ``ld`` is None (each shard as wide as its columns) or one row
    stride (elements) for all shards."""
    vs = even_vocab_start(w.V, w.t) if vocab_start is None else list(vocab_start)
    rows = np.arange(w.s) if rows is None else np.asarray(rows)
    out = []
    for i in range(len(vs) - 1):
        width = vs[i + 1] - vs[i]
        lda = width if ld is None else int(ld)
        vals = logits_rows(w, rows, vs[i], vs[i + 1], meta)
        if lda == width:
            out.append(np.ascontiguousarray(vals))
            continue
        if w.dtype == "bf16":
            buf = np.full((len(rows), lda), 0x7FC1, dtype=np.uint16)
        else:
            buf = np.full((len(rows), lda), np.nan, dtype=np.float32)
        buf[:, :width] = vals
        out.append(buf)
    return out


# --------------------------------------------------------------------------
# device twin (libvpce_synth.so): fills device shards with the same values
# --------------------------------------------------------------------------
_SYNTH_LIB = None


def _synth_lib():
    global _SYNTH_LIB
    if _SYNTH_LIB is None:
        import ctypes
        import os

        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libvpce_synth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is not built: run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.vpce_synth_fill.restype = ctypes.c_int
        lib.vpce_synth_fill.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_longlong,
                                        ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
                                        ctypes.c_longlong, ctypes.c_ulonglong, ctypes.c_double,
                                        ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p]
        _SYNTH_LIB = lib
    return _SYNTH_LIB


def device_shards(w: Workload, meta: RowMeta, vocab_start=None, ld=None, device="cuda", row0: int = 0,
                  s: int | None = None):
    """Allocate and fill the t device shards of workload ``w`` (rows
    ``row0 .. row0+s-1`` of the batch described by ``meta``).  Returns a list
    of torch tensors ``[s, w_i]`` (views with row stride ``ld`` if given;
    padding columns hold a NaN canary)."""
    import ctypes
    import torch

    s = w.s if s is None else s
    vs = even_vocab_start(w.V, w.t) if vocab_start is None else list(vocab_start)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    boost = torch.from_numpy(np.ascontiguousarray(meta.boost_col)).to(device)
    key = int(stream_key(w.seed, STREAM_VALUES))
    stream = torch.cuda.current_stream(device).cuda_stream
    out = []
    for i in range(len(vs) - 1):
        width = vs[i + 1] - vs[i]
        lda = width if ld is None else int(ld)
        if lda == width:
            buf = torch.empty((s, lda), dtype=tdt, device=device)
        else:
            buf = torch.full((s, lda), float("nan"), dtype=tdt, device=device)
        err = _synth_lib().vpce_synth_fill(ctypes.c_void_p(buf.data_ptr()), 1 if w.dtype == "bf16" else 0,
                                           s, row0, vs[i], width, lda, w.V, key, float(w.sigma),
                                           ctypes.c_void_p(boost.data_ptr()), float(meta.boost_val),
                                           ctypes.c_void_p(stream))
        if err != 0:
            raise RuntimeError(f"vpce_synth_fill failed with CUDA error {err}")
        out.append(buf[:, :width])
    torch.cuda.current_stream(device).synchronize()
    del boost
    return out


# --------------------------------------------------------------------------
# LM-head inputs: hidden states X [s, h] and the vocabulary-sharded head
# W [V, h] (one row per vocabulary entry), both bf16, drawn element by
# element from their own streams of the same generator.
# --------------------------------------------------------------------------
STREAM_HIDDEN = 5
STREAM_WEIGHT = 6


@dataclasses.dataclass(frozen=True)
class LmHead:
    name: str
    index: int              # seed = 20261202 + index
    s: int                  # rows (tokens)
    h: int                  # hidden size (K of the contraction)
    V: int                  # vocabulary
    t: int                  # shards
    sigma_x: float = 1.0    # X ~ N(0, sigma_x^2)
    logit_sigma: float = 3.0  # W ~ N(0, (logit_sigma / sqrt(h))^2): logits ~ N(0, logit_sigma^2)
    ignore_frac: float = 0.0
    ignore_index: int = -100

    @property
    def seed(self) -> int:
        return 20261202 + self.index

    @property
    def sigma_w(self) -> float:
        return self.logit_sigma / float(np.sqrt(self.h))

    def replace(self, **kw) -> "LmHead":
        return dataclasses.replace(self, **kw)

    def as_workload(self) -> Workload:
        """The loss-side recipe with the same rows, vocabulary and targets."""
        return Workload(self.name, self.index, self.s, self.V, self.t, "bf16", self.logit_sigma, "uniform",
                        ignore_frac=self.ignore_frac, ignore_index=self.ignore_index)


LMHEADS = {
    m.name: m for m in [
        # the pages' Llama-3-70B LM head: [128256, 8192], t = 8, s = 8192
        LmHead("lmhead_s8192_h8192_v128256", 6, 8192, 8192, 128256, 8),
        LmHead("lmhead_s300_h512_v5000", 7, 300, 512, 5000, 3, ignore_frac=0.05),
    ]
}
LMHEAD_BENCH = "lmhead_s8192_h8192_v128256"


def dense_host(seed: int, stream: int, rows, cols: int, sigma: float) -> np.ndarray:
    """bf16 patterns (uint16) of rows ``rows`` of a [*, cols] matrix whose
    element (r, c) is the generator's normal number r * cols + c of the
    stream, times sigma, rounded to binary32 and then to bfloat16."""
    rows = np.asarray(rows, dtype=np.int64)
    key = stream_key(seed, stream)
    g = rows[:, None].astype(np.uint64) * np.uint64(cols) + np.arange(cols, dtype=np.uint64)[None, :]
    v = (_normals_from_index(key, g) * sigma).astype(np.float32)
    return f32_to_bf16_bits(v)


def lmhead_meta(m: LmHead) -> RowMeta:
    return row_meta(m.as_workload())


def _dense_device(buf, seed: int, stream: int, row0: int, cols: int, sigma: float) -> None:
    import ctypes
    import torch

    key = int(stream_key(seed, stream))
    st = torch.cuda.current_stream(buf.device).cuda_stream
    err = _synth_lib().vpce_synth_fill(ctypes.c_void_p(buf.data_ptr()), 1, buf.shape[0], row0, 0, cols,
                                       buf.stride(0), cols, key, float(sigma), None, 0.0, ctypes.c_void_p(st))
    if err != 0:
        raise RuntimeError(f"vpce_synth_fill failed with CUDA error {err}")


def lmhead_device(m: LmHead, vocab_start=None, device="cuda"):
    """Device X [s, h] and the t weight shards [w_i, h] (bf16), filled by the
    device twin of the generator (the values of :func:`dense_host`)."""
    import torch

    vs = even_vocab_start(m.V, m.t) if vocab_start is None else list(vocab_start)
    x = torch.empty((m.s, m.h), dtype=torch.bfloat16, device=device)
    _dense_device(x, m.seed, STREAM_HIDDEN, 0, m.h, m.sigma_x)
    ws = []
    for i in range(len(vs) - 1):
        wi = torch.empty((vs[i + 1] - vs[i], m.h), dtype=torch.bfloat16, device=device)
        _dense_device(wi, m.seed, STREAM_WEIGHT, vs[i], m.h, m.sigma_w)
        ws.append(wi)
    torch.cuda.current_stream(device).synchronize()
    return x, ws


# --------------------------------------------------------------------------
# embedding inputs: the table [V, h] (stream 7), output gradients [s, h]
# (stream 8), ids from the loss workloads' target recipes
# --------------------------------------------------------------------------
STREAM_TABLE = 7
STREAM_GRAD = 8


def table_device(seed: int, vocab_start, h: int, sigma: float = 1.0, device="cuda"):
    """Device bf16 table shards [w_i, h]: element (v, k) is normal number
    v * h + k of stream 7 (the values of dense_host(seed, STREAM_TABLE, ...))."""
    import torch

    out = []
    for i in range(len(vocab_start) - 1):
        e = torch.empty((vocab_start[i + 1] - vocab_start[i], h), dtype=torch.bfloat16, device=device)
        _dense_device(e, seed, STREAM_TABLE, vocab_start[i], h, sigma)
        out.append(e)
    torch.cuda.current_stream(device).synchronize()
    return out


def grad_device(seed: int, s: int, h: int, sigma: float = 1.0, device="cuda"):
    """Device bf16 output gradient [s, h] (stream 8)."""
    import torch

    g = torch.empty((s, h), dtype=torch.bfloat16, device=device)
    _dense_device(g, seed, STREAM_GRAD, 0, h, sigma)
    torch.cuda.current_stream(device).synchronize()
    return g
