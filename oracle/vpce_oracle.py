"""fp64 CPU oracle for vocab-parallel cross-entropy.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may use it.  It shares no code
with the CUDA library (no kernels, headers, helpers or constants); the only
thing both sides see is the seeded synthetic input.

What it computes, and where the method is defined
-------------------------------------------------
* "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16 notes),
  §5.5 "Embedding and output layer": when the output layer is split by
  vocabulary each card holds a slice of the logits; the cross-entropy is
  CE = logsumexp(z) - z[target]; the logsumexp is taken blockwise, with the
  per-block maxima combined first for stability, then the per-block sums of
  exponentials, and the target logit, which lives on exactly one card, is
  combined once more -- three scalars per token.  The lecture's script matched
  ``F.cross_entropy`` to about 1e-15 in float64, i.e. the sharded method reaches
  the plain unsharded cross-entropy up to rounding order.
* "LLM Internals" §7.3 "Model and tensor parallelism", §7.3.4 (attention,
  SwiGLU, embedding and LM head splits): the LM-head logits are ``[s, V]``
  (``[8192, 128256]`` for Llama-3-70B, 16032 columns per card at t = 8); the
  vocab-parallel cross-entropy reduces, per position, only the maximum, the
  target logit and the sum of exponentials, with the math in FP32.

Because the sharded method equals the unsharded definition up to rounding
order, :func:`cross_entropy` and :func:`dlogits` are that plain definition
written out in fp64 over the re-assembled full rows.  :func:`shard_partials` and
:func:`combine_sharded` restate the pages' three-scalar combine separately; the
tests check that it agrees with the unsharded definition, and nothing on the
GPU side calls it.

Readings taken where the pages are silent:
* backward: d(mean CE)/dz = g * (softmax(z) - onehot(y)) / n_valid  (the
  standard derivative of the mean loss; the pages give no backward);
* reduction: mean over rows whose target is not ``ignore_index`` (the default
  of ``F.cross_entropy``, the routine the pages compare against); 'sum' and
  'none' follow the same routine's other modes;
* ``ignore_index`` rows contribute no loss, are not counted in n_valid and get
  zero gradient; n_valid = 0 gives loss NaN (0/0) and an all-zero gradient;
* a target outside [0, V) that is not ``ignore_index`` makes that row's loss,
  lse and gradient NaN and raises the error flag;
* bf16 inputs are used as stored: the 16-bit pattern is widened exactly.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "widen",
    "assemble",
    "cross_entropy",
    "dlogits",
    "split_columns",
    "shard_partials",
    "fold_partials",
    "combine_sharded",
    "lmhead_logits",
    "lmhead_backward",
    "embedding_forward",
    "embedding_backward",
]


# --------------------------------------------------------------------------
# input widening and shard re-assembly
# --------------------------------------------------------------------------
def widen(values: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored logits to fp64 exactly.

    ``dtype == 'bf16'``: ``values`` holds raw bfloat16 bit patterns (uint16);
    a bfloat16 is the upper half of an IEEE binary32, so shifting the pattern
    16 bits left gives the binary32 with the same value, which widens exactly.
    ``dtype == 'fp32'``: ``values`` is float32 and widens exactly.
    """
    if dtype == "bf16":
        bits = np.asarray(values, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    if dtype == "fp32":
        return np.asarray(values, dtype=np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def assemble(shards, vocab_start, dtype: str) -> np.ndarray:
    """Re-assemble the full fp64 rows ``z[r, k]`` from t vocabulary shards.

    ``shards[i]`` is a 2-D array ``[s, ld_i]`` whose first
    ``vocab_start[i+1] - vocab_start[i]`` columns hold global vocabulary columns
    ``vocab_start[i] .. vocab_start[i+1]-1`` (columns past that are padding
    and ignored).  ``vocab_start`` has t+1 entries, starts at 0 and increases.
    """
    t = len(shards)
    vs = [int(v) for v in vocab_start]
    if len(vs) != t + 1 or vs[0] != 0:
        raise ValueError("vocab_start must have t+1 entries starting at 0")
    s = shards[0].shape[0]
    V = vs[-1]
    z = np.empty((s, V), dtype=np.float64)
    for i, sh in enumerate(shards):
        w = vs[i + 1] - vs[i]
        if w < 1:
            raise ValueError("empty shard")
        z[:, vs[i]:vs[i + 1]] = widen(sh[:, :w], dtype)
    return z


def split_columns(full: np.ndarray, vocab_start):
    """Cut a ``[s, V]`` array back into the t column blocks of ``vocab_start``."""
    vs = [int(v) for v in vocab_start]
    return [full[:, vs[i]:vs[i + 1]] for i in range(len(vs) - 1)]


# --------------------------------------------------------------------------
# the unsharded definition
# --------------------------------------------------------------------------
def _row_status(y: np.ndarray, V: int, ignore_index: int):
    y = np.asarray(y, dtype=np.int64)
    ignored = y == ignore_index
    bad = (~ignored) & ((y < 0) | (y >= V))
    valid = (~ignored) & (~bad)
    return valid, ignored, bad


def cross_entropy(z: np.ndarray, y: np.ndarray, ignore_index: int = -100,
                  reduction: str = "mean", n_valid: int | None = None) -> dict:
    """Cross-entropy of full fp64 rows: CE_r = logsumexp(z_r) - z_r[y_r].

    logsumexp is taken in the numerically stable form M + log(sum exp(z - M))
    with M the row maximum (the reason the pages combine the maxima first).

    Returns a dict with per-row ``lse`` (NaN for ignored rows), ``row_loss``
    (0 for ignored rows, NaN for out-of-range targets, as 'none' reduction
    gives), ``valid`` mask, ``n_valid``, ``error_flag`` (1 when some target is
    neither ``ignore_index`` nor in [0, V)) and ``loss`` for the requested
    reduction ('mean', 'sum' or 'none' -> the per-row vector).

    ``n_valid`` may be given when ``z`` holds only a sample of a batch's rows
    (the mean divides by the count of the whole batch).
    """
    z = np.asarray(z, dtype=np.float64)
    s, V = z.shape
    y = np.asarray(y, dtype=np.int64)
    valid, ignored, bad = _row_status(y, V, ignore_index)
    lse = np.full(s, np.nan)
    row_loss = np.zeros(s)
    if s:
        M = z.max(axis=1)
        S = np.exp(z - M[:, None]).sum(axis=1)
        lse_all = M + np.log(S)
        lse = np.where(ignored, np.nan, lse_all)
        lse = np.where(bad, np.nan, lse)
        rows = np.nonzero(valid)[0]
        row_loss[rows] = lse_all[rows] - z[rows, y[rows]]
        row_loss[bad] = np.nan
    nv = int(valid.sum()) if n_valid is None else int(n_valid)
    total = float(row_loss.sum()) if s else 0.0
    if reduction == "mean":
        loss = total / nv if nv > 0 else float("nan")
    elif reduction == "sum":
        loss = total
    elif reduction == "none":
        loss = row_loss.copy()
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    return {
        "loss": loss,
        "row_loss": row_loss,
        "lse": lse,
        "valid": valid,
        "n_valid": nv,
        "error_flag": int(bad.any()),
    }


def dlogits(z: np.ndarray, y: np.ndarray, ignore_index: int = -100,
            grad=1.0, reduction: str = "mean",
            n_valid: int | None = None, lse: np.ndarray | None = None) -> np.ndarray:
    """Gradient of the reduced cross-entropy w.r.t. the logits, in fp64.

    For a valid row r: d_rk = g * (exp(z_rk - lse_r) - [k == y_r]) / n_valid
    ('mean'; the division is dropped for 'sum').  For 'none' the loss is the
    per-row vector and ``grad`` is its upstream gradient, one g_r per row (a
    scalar is applied to every row): d_rk = g_r * (exp(z_rk - lse_r) -
    [k == y_r]).  Ignored rows are zero whatever their g_r; rows with an
    out-of-range target are NaN.  ``n_valid`` defaults to the count in
    ``y``; pass the batch count when ``z`` holds a sample of the rows.
    """
    z = np.asarray(z, dtype=np.float64)
    s, V = z.shape
    y = np.asarray(y, dtype=np.int64)
    valid, ignored, bad = _row_status(y, V, ignore_index)
    if lse is None:
        lse = cross_entropy(z, y, ignore_index)["lse"]
    nv = int(valid.sum()) if n_valid is None else int(n_valid)
    if reduction == "mean":
        scale = np.full(s, grad / nv if nv > 0 else 0.0)
    elif reduction == "sum":
        scale = np.full(s, float(grad))
    elif reduction == "none":
        scale = np.broadcast_to(np.asarray(grad, dtype=np.float64), (s,))
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    d = np.zeros((s, V))
    rows = np.nonzero(valid)[0]
    if rows.size:
        p = np.exp(z[rows] - lse[rows][:, None])
        p[np.arange(rows.size), y[rows]] -= 1.0
        d[rows] = scale[rows][:, None] * p
    d[bad] = np.nan
    return d


# --------------------------------------------------------------------------
# the LM head in front of the loss
# --------------------------------------------------------------------------
def lmhead_logits(x, w_shards, vocab_start, dtype: str = "bf16") -> np.ndarray:
    """Full fp64 logits of a vocabulary-split LM head, ``z = X W^T``.

    "LLM Internals" §7.3.4 splits the LM head ``[V, h]`` (``[128256, 8192]``
    for Llama-3-70B) along the vocabulary, ``[16032, h]`` per card at t = 8;
    card i's logits are the columns ``vocab_start[i] .. vocab_start[i+1]-1``
    of ``z``.  ``x`` is ``[s, h]``, ``w_shards[i]`` is ``[w_i, h]`` (one row
    per vocabulary entry), both in the stored form of ``dtype`` (bf16 bit
    patterns or float32), widened exactly; the product is a plain fp64 matrix
    multiply, so z is the exact dot product up to fp64 rounding.
    """
    X = widen(x, dtype)
    vs = [int(v) for v in vocab_start]
    if len(vs) != len(w_shards) + 1 or vs[0] != 0:
        raise ValueError("vocab_start must have t+1 entries starting at 0")
    z = np.empty((X.shape[0], vs[-1]), dtype=np.float64)
    for i, w in enumerate(w_shards):
        W = widen(w, dtype)
        if W.shape != (vs[i + 1] - vs[i], X.shape[1]):
            raise ValueError(f"shard {i} has shape {W.shape}")
        z[:, vs[i]:vs[i + 1]] = X @ W.T
    return z


def lmhead_backward(x, w_shards, vocab_start, y, ignore_index: int = -100, grad=1.0,
                    reduction: str = "mean", dtype: str = "bf16"):
    """Gradients of the reduced cross-entropy of ``z = X W^T`` with respect
    to X and to each head shard, in fp64.

    The pages give no backward; this is the chain rule through the plain
    product: with ``dZ = dlogits(z, ...)`` (the loss's own gradient, per-row
    ``grad`` for 'none'), ``dX = dZ W`` and ``dW_i = dZ_i^T X``.  Returns
    ``(dX [s, h], [dW_i [w_i, h]], dZ)``.
    """
    vs = [int(v) for v in vocab_start]
    X = widen(x, dtype)
    z = lmhead_logits(x, w_shards, vs, dtype)
    dz = dlogits(z, y, ignore_index, grad=grad, reduction=reduction)
    dX = np.zeros_like(X)
    dW = []
    for i, w in enumerate(w_shards):
        W = widen(w, dtype)
        dzi = dz[:, vs[i]:vs[i + 1]]
        dX += dzi @ W
        dW.append(dzi.T @ X)
    return dX, dW, dz


# --------------------------------------------------------------------------
# the vocabulary-parallel input embedding
# --------------------------------------------------------------------------
def embedding_forward(table_shards, vocab_start, ids, dtype: str = "bf16"):
    """Output rows of a vocabulary-split embedding table, in fp64.

    "Distributed Training III: Model Parallelism" (CMU 11-868 Lecture 16
    notes), §5.5: card i holds only the embeddings of the ids in its range,
    fills every other position with zeros, and an all-reduce sums the cards.
    "LLM Internals" §7.3.4: the table [128256, 8192] is split into [16032,
    8192] per card, ids outside a card's range give zero vectors there.
    Written out in that order: card i's masked lookup, then the sum over
    cards.  An id outside [0, V) is in no card's range, so its row is zero;
    ``bad`` reports whether any id was.  Returns ``(out [s, h], bad)``.
    """
    vs = [int(v) for v in vocab_start]
    ids = np.asarray(ids, dtype=np.int64)
    shards = [widen(e, dtype) for e in table_shards]
    h = shards[0].shape[1]
    out = np.zeros((ids.size, h))
    for i, e in enumerate(shards):
        mine = (ids >= vs[i]) & (ids < vs[i + 1])
        part = np.zeros((ids.size, h))
        part[mine] = e[ids[mine] - vs[i]]
        out += part
    bad = bool(np.any((ids < 0) | (ids >= vs[-1])))
    return out, bad


def embedding_backward(grad_out, ids, vocab_start, h: int):
    """Gradient of the embedding lookup with respect to each table shard, fp64.

    The pages give no backward.  The standard one is the adjoint of the
    lookup: row j of shard i receives the sum of the output gradients of the
    positions whose id is ``vocab_start[i] + j``.  Ids outside [0, V) send
    their gradient nowhere, matching their zero output rows.  ``grad_out`` is
    ``[s, h]`` fp64.  Returns the list of shard gradients ``[w_i, h]``.
    """
    vs = [int(v) for v in vocab_start]
    ids = np.asarray(ids, dtype=np.int64)
    g = np.asarray(grad_out, dtype=np.float64)
    out = []
    for i in range(len(vs) - 1):
        d = np.zeros((vs[i + 1] - vs[i], h))
        mine = np.nonzero((ids >= vs[i]) & (ids < vs[i + 1]))[0]
        for r in mine:
            d[ids[r] - vs[i]] += g[r]
        out.append(d)
    return out


# --------------------------------------------------------------------------
# the pages' three-scalar combine, restated on its own
# --------------------------------------------------------------------------
def shard_partials(z_shard: np.ndarray, y: np.ndarray, vocab_lo: int, vocab_hi: int):
    """What one card reduces from its slice of the logits, per row.

    Returns ``(m, se, tgt)``: the local maximum, the local sum of
    exp(z - m), and the target logit when vocab_lo <= y < vocab_hi (0.0
    otherwise, so that summing over cards picks the one card that holds it).
    """
    z_shard = np.asarray(z_shard, dtype=np.float64)
    y = np.asarray(y, dtype=np.int64)
    m = z_shard.max(axis=1)
    se = np.exp(z_shard - m[:, None]).sum(axis=1)
    mine = (y >= vocab_lo) & (y < vocab_hi)
    tgt = np.zeros(z_shard.shape[0])
    rows = np.nonzero(mine)[0]
    tgt[rows] = z_shard[rows, y[rows] - vocab_lo]
    return m, se, tgt


def fold_partials(ms: np.ndarray, ses: np.ndarray):
    """Several cards' (max, sum exp) pairs of one row set merged into the
    pair of their union of columns, the first and third steps of the pages'
    combine without the logarithm: M = max_i m_i, S = sum_i se_i exp(m_i - M).
    ``ms``, ``ses``: [cards, rows].  Returns ``(M, S)``; the pair equals
    :func:`shard_partials` of the concatenated columns up to rounding, which
    is what lets a process send one pair per row for all of its shards."""
    ms = np.asarray(ms, dtype=np.float64)
    ses = np.asarray(ses, dtype=np.float64)
    M = ms.max(axis=0)
    S = (ses * np.exp(ms - M[None, :])).sum(axis=0)
    return M, S


def combine_sharded(partials, y: np.ndarray, V: int, ignore_index: int = -100):
    """Combine the t cards' partials as the pages do, in fp64.

    1. all-reduce(MAX) of the local maxima gives the row maximum M;
    2. all-reduce(SUM) of the target logits gives z[y] (one card holds it);
    3. all-reduce(SUM) of the local sums, each rescaled to the common maximum
       by exp(m_i - M), gives sum exp(z - M); lse = M + log of it.
    Returns ``(lse, row_loss, mean_loss)`` with ignored rows excluded from the
    mean (and given row loss 0), as in :func:`cross_entropy`.
    """
    y = np.asarray(y, dtype=np.int64)
    ms = np.stack([p[0] for p in partials])
    ses = np.stack([p[1] for p in partials])
    tgts = np.stack([p[2] for p in partials])
    M = ms.max(axis=0)
    zy = tgts.sum(axis=0)
    S = (ses * np.exp(ms - M[None, :])).sum(axis=0)
    lse = M + np.log(S)
    valid, ignored, bad = _row_status(y, V, ignore_index)
    row_loss = np.where(valid, lse - zy, 0.0)
    row_loss = np.where(bad, np.nan, row_loss)
    nv = int(valid.sum())
    mean = float(row_loss.sum()) / nv if nv > 0 else float("nan")
    return lse, row_loss, mean
