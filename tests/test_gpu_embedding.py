"""GPU parity of the vocabulary-parallel embedding (vpce_embedding_forward /
vpce_embedding_backward) against the fp64 oracle.

* Forward: a copy of table rows, so bit-exact; ids outside [0, V) give zero
  rows and the flag.
* Backward: each table row receives the fp32 sum of its ids' gradient rows in
  a fixed order (ascending rows; ids with more than 64 rows in a chunk as
  eight ascending slices, then the slices in order), then one fp32 add.
  Against fp64 that is at most (count + 1) * 2^-24 * sum |g| per element (the
  recursive-summation bound, which holds for any summation tree of count + 1
  terms), checked element by element; results are bitwise repeatable."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def _ids(seed, s, V, kind="uniform", extra=()):
    w = synth.Workload("ids", seed, s, V, 1, "bf16", 1.0, kind)
    y = synth.row_meta(w).targets.copy()
    for r, v in extra:
        y[r] = v
    return y


@pytest.mark.parametrize("V,h,vs,s", [
    (1000, 64, None, 300),
    (5000, 136, [0, 1, 2, 2500, 5000], 513),        # one-row shards; 272-byte rows
    (300, 8, [0, 100, 300], 70),
])
def test_embedding_forward_bitexact(V, h, vs, s):
    vs = vs or synth.even_vocab_start(V, 4)
    ids = _ids(31, s, V, extra=[(0, 0), (1, V - 1), (2, -1), (3, V), (4, -100)])
    tab = synth.table_device(31, vs, h)
    flag = torch.zeros((), dtype=torch.int32, device="cuda")
    out = vpce.vpce_embedding_forward(tab, torch.from_numpy(ids).cuda(), vs, flag=flag)
    torch.cuda.synchronize()
    ref, bad = O.embedding_forward([_bits(e) for e in tab], vs, ids)
    np.testing.assert_array_equal(O.widen(_bits(out), "bf16"), ref)
    assert bool(int(flag.item()) & vpce.VPCE_FLAG_BAD_TARGET) == bad == True


def test_embedding_forward_fp32_padded_and_misaligned():
    V, h, s = 700, 37, 90                 # odd h: rows are not 16-byte multiples (element path)
    vs = [0, 350, 700]
    ids = _ids(32, s, V)
    tab = [e.float() for e in synth.table_device(32, vs, h)]
    padded = []
    for e in tab:
        b = torch.full((e.shape[0], h + 3), float("nan"), device="cuda")
        b[:, :h] = e
        padded.append(b[:, :h])
    out_buf = torch.full((s, h + 5), -1.0, device="cuda")
    vpce.vpce_embedding_forward(padded, torch.from_numpy(ids).cuda(), vs, out=out_buf[:, :h])
    torch.cuda.synchronize()
    ref, bad = O.embedding_forward([e.cpu().numpy() for e in tab], vs, ids, dtype="fp32")
    np.testing.assert_array_equal(out_buf[:, :h].cpu().numpy(), ref)
    assert np.all(out_buf[:, h:].cpu().numpy() == -1.0)   # padding untouched
    assert not bad


def _check_backward(V, h, vs, s, kind, grad_dtype, seed, extra=(), ld=None):
    ids = _ids(seed, s, V, kind, extra)
    g = synth.grad_device(seed, s, ld or h)[:, :h]  # ld: padded rows
    if grad_dtype == "fp32":
        g = g.float()
    gh = O.widen(_bits(g), "bf16") if grad_dtype == "bf16" else g.cpu().numpy().astype(np.float64)
    init = [torch.full((vs[i + 1] - vs[i], h), 0.25, dtype=torch.float32, device="cuda") for i in range(len(vs) - 1)]
    vpce.vpce_embedding_backward(g, torch.from_numpy(ids).cuda(), init, vs)
    torch.cuda.synchronize()
    got = np.concatenate([d.cpu().numpy().astype(np.float64) for d in init])
    ref = np.concatenate(O.embedding_backward(gh, ids, vs, h)) + 0.25
    valid = (ids >= 0) & (ids < V)
    count = np.bincount(ids[valid], minlength=V)
    absum = np.zeros((V, h))
    np.add.at(absum, ids[valid], np.abs(gh[valid]))
    bound = (count[:, None] + 1) * 2.0 ** -24 * (absum + 0.25)
    assert np.all(np.abs(got - ref) <= bound)
    return init


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("kind", ["uniform", "zipf1.1"])
def test_embedding_backward(kind, grad_dtype):
    _check_backward(2000, 64, [0, 1, 999, 2000], 3000, kind, grad_dtype, 41,
                    extra=[(5, -1), (6, 2000), (7, -100)])


@pytest.mark.parametrize("grad_dtype", ["bf16", "fp32"])
def test_embedding_backward_ragged_column_blocks(grad_dtype):
    # h = 516: two full 256-column blocks and a 4-column tail (for bf16 half
    # of a 16-byte piece; rows padded to 520 for 16-byte row strides), with
    # long and short runs of Zipf ids
    _check_backward(900, 516, [0, 450, 900], 2500, "zipf1.1", grad_dtype, 45, extra=[(3, -1)], ld=520)


@pytest.mark.parametrize("V", [262142, 300000])
def test_embedding_backward_vocabulary_sizes(V):
    # the largest vocabulary sorted with 32-bit (id, row) keys, and one past
    # it (64-bit keys); the largest ids are present
    _check_backward(V, 16, [0, V // 3, 2 * V // 3, V], 3000, "uniform", "bf16", 47,
                    extra=[(0, V - 1), (1, V - 1), (2, V - 2), (3, 0), (4, V)])


def test_embedding_backward_error_flag_is_clear():
    V, h, s = 1000, 264, 700
    vs = [0, 500, 1000]
    ids = torch.from_numpy(_ids(46, s, V, "zipf1.1", ())).cuda()
    g = synth.grad_device(46, s, h)
    grads = [torch.zeros((500, h), dtype=torch.float32, device="cuda") for _ in range(2)]
    wk = torch.full((vpce.vpce_embedding_backward_workspace_bytes(),), 0xFF, dtype=torch.uint8, device="cuda")
    vpce.vpce_embedding_backward(g, ids, grads, vs, workspace=wk)
    assert vpce.vpce_read_error_flag(wk) == 0


def test_embedding_backward_multi_chunk_is_deterministic():
    # 40000 rows: three 16384-row chunks accumulated in order
    a = _check_backward(500, 16, [0, 250, 500], 40000, "zipf1.1", "bf16", 42)
    b = _check_backward(500, 16, [0, 250, 500], 40000, "zipf1.1", "bf16", 42)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x.cpu().numpy(), y.cpu().numpy())


def test_embedding_full_size_sampled_rows():
    """The pages' table [128256, 8192] bf16 split t = 8, 8192 ids: the forward
    checked on sampled rows (bit-exact against the host generator), the
    backward on the rows of sampled ids (Zipf ids, so some repeat)."""
    V, h, s, t = 128256, 8192, 8192, 8
    vs = synth.even_vocab_start(V, t)
    ids = _ids(43, s, V, "zipf1.1")
    tab = synth.table_device(43, vs, h)
    dev_ids = torch.from_numpy(ids).cuda()
    out = vpce.vpce_embedding_forward(tab, dev_ids, vs)
    torch.cuda.synchronize()
    rng = np.random.default_rng(9)
    rows = np.concatenate([[0, s - 1], rng.integers(1, s - 1, size=30)])
    got = _bits(out[torch.from_numpy(rows).cuda()])
    ref = synth.dense_host(43, synth.STREAM_TABLE, ids[rows], h, 1.0)
    diff = np.abs(got.astype(np.int64) - ref.astype(np.int64))
    assert diff.max() <= 1 and np.count_nonzero(diff) <= 2   # device log/cos last bit
    del tab, out
    g = synth.grad_device(44, s, h)
    grads = [torch.zeros((vs[i + 1] - vs[i], h), dtype=torch.float32, device="cuda") for i in range(t)]
    vpce.vpce_embedding_backward(g, dev_ids, grads, vs)
    torch.cuda.synchronize()
    gh_bits = _bits(g)
    uniq, counts = np.unique(ids, return_counts=True)
    pick = np.concatenate([uniq[np.argsort(-counts)[:3]], rng.choice(uniq, size=5, replace=False)])
    for v in pick:
        i = np.searchsorted(vs, v, side="right") - 1
        gotrow = grads[i][v - vs[i]].cpu().numpy().astype(np.float64)
        rs = np.nonzero(ids == v)[0]
        gr = O.widen(gh_bits[rs], "bf16")
        refrow = gr.sum(axis=0)
        bound = (len(rs) + 1) * 2.0 ** -24 * np.abs(gr).sum(axis=0)
        assert np.all(np.abs(gotrow - refrow) <= bound), v
