"""CUDA-graph capture of the stream-ordered entry points: after a first call
on the device (its one-time set-up: architecture check, shared-memory
limits), the split path, the fused path, the per-row backward, the LM head
and the embedding launch only kernels (and, for the embedding flag, a
memset), so a stream capture records them and replays them with identical
results."""
import numpy as np
import pytest
import torch

from oracle import vpce_oracle as O
from vocab_sharded_lm_gb300 import synth, vpce

from _parity import from_device, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from vocab_sharded_lm_gb300 import _build

    _build.build()
    vpce.load_library()


def _capture(fn):
    """Warm up on a side stream, capture fn() into a graph, return it."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("path,wl", [("split", "s8192_v128256"), ("fused", "s8192_v128256"),
                                     ("rows", "s8192_v128256"), ("fused", "s32768_v256000")])
def test_loss_paths_replay_identically(path, wl):
    # s32768_v256000: 512 KB rows, the fused kernel's two-CTA cluster launch
    w = synth.WORKLOADS[wl].replace(s=64)
    vs = synth.even_vocab_start(w.V, w.t)
    meta = synth.row_meta(w)
    host = synth.shards_host(w, meta, vs)
    y = torch.from_numpy(meta.targets).cuda()
    work = to_device(host, w.dtype)
    pristine = [d.clone() for d in work]
    ws = vpce.new_workspace(w.t, w.s, "cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    rl = torch.empty(w.s, dtype=torch.float32, device="cuda")
    gr = torch.linspace(-1.0, 1.0, w.s, device="cuda")

    def step():
        for d, p in zip(work, pristine):
            d.copy_(p)
        if path == "split":
            vpce.vpce_forward(work, y, vs, loss_out=loss, row_loss_out=rl, workspace=ws)
            vpce.vpce_backward(work, y, ws, vs)
        elif path == "fused":
            vpce.vpce_forward_backward(work, y, vs, loss_out=loss, row_loss_out=rl, workspace=ws)
        else:
            vpce.vpce_forward_backward(work, y, vs, grad_rows=gr, loss_out=loss, row_loss_out=rl, workspace=ws)

    step()
    torch.cuda.synchronize()
    ref_loss, ref_rl = float(loss), rl.cpu().numpy().copy()
    ref_d = [from_device(d, w.dtype).copy() for d in work]
    g = _capture(step)
    for _ in range(3):
        loss.fill_(-1.0)
        g.replay()
        torch.cuda.synchronize()
        assert float(loss) == ref_loss
        np.testing.assert_array_equal(rl.cpu().numpy(), ref_rl)
        for a, b in zip(ref_d, work):
            np.testing.assert_array_equal(a, from_device(b, w.dtype))
    # and the eager result itself is the oracle's
    z = O.assemble(host, vs, w.dtype)
    assert abs(ref_loss - O.cross_entropy(z, meta.targets)["loss"]) <= 1e-5 * abs(ref_loss)


def test_lmhead_and_embedding_replay_identically():
    m = synth.LmHead("graph", 23, 256, 128, 1000, 2)
    mvs = synth.even_vocab_start(m.V, m.t)
    x, wsh = synth.lmhead_device(m, mvs)
    y = torch.from_numpy(synth.lmhead_meta(m).targets).cuda()
    wk = torch.empty(vpce.vpce_lmhead_workspace_bytes(m.s), dtype=torch.uint8, device="cuda")
    loss = torch.empty((), dtype=torch.float32, device="cuda")
    tvs = [0, 400, 1000]
    tab = synth.table_device(24, tvs, 64)
    ids = torch.from_numpy(np.random.default_rng(1).integers(0, 1000, size=300)).cuda()
    out = torch.empty((300, 64), dtype=torch.bfloat16, device="cuda")
    flag = torch.zeros((), dtype=torch.int32, device="cuda")
    gout = synth.grad_device(25, 300, 64)
    gtab = [torch.zeros((tvs[i + 1] - tvs[i], 64), dtype=torch.float32, device="cuda") for i in range(2)]
    ewk = torch.empty(vpce.vpce_embedding_backward_workspace_bytes(), dtype=torch.uint8, device="cuda")

    dx = torch.empty_like(x)
    dw = [torch.zeros(sh.shape, dtype=torch.float32, device="cuda") for sh in wsh]
    bwk = torch.empty(vpce.vpce_lmhead_backward_workspace_bytes(m.V, m.h), dtype=torch.uint8, device="cuda")
    # the one-call training step: prologue, logits-keeping GEMM, row kernel, dX and dW products, loss sum
    loss2 = torch.empty((), dtype=torch.float32, device="cuda")
    dx2 = torch.empty_like(x)
    dw2 = [torch.zeros(sh.shape, dtype=torch.float32, device="cuda") for sh in wsh]
    twk = torch.empty(vpce.vpce_lmhead_forward_backward_workspace_bytes(m.s, m.V, m.h), dtype=torch.uint8,
                      device="cuda")

    def step():
        vpce.vpce_lmhead_forward(x, wsh, y, mvs, loss_out=loss, workspace=wk)
        for d in dw:
            d.zero_()
        vpce.vpce_lmhead_backward(x, wsh, y, wk, mvs, grad_hidden=dx, grad_weight_shards=dw, workspace=bwk)
        for d in dw2:
            d.zero_()
        vpce.vpce_lmhead_forward_backward(x, wsh, y, mvs, loss_out=loss2, grad_hidden=dx2, grad_weight_shards=dw2,
                                          workspace=twk)
        vpce.vpce_embedding_forward(tab, ids, tvs, out=out, flag=flag)
        for t_ in gtab:
            t_.zero_()
        vpce.vpce_embedding_backward(gout, ids, gtab, tvs, workspace=ewk)

    step()
    torch.cuda.synchronize()
    ref = (float(loss), out.clone(), [t_.clone() for t_ in gtab], dx.clone(), [d.clone() for d in dw],
           float(loss2), dx2.clone(), [d.clone() for d in dw2])
    g = _capture(step)
    for _ in range(3):
        loss.fill_(-1.0)
        out.zero_()
        dx.zero_()
        dx2.zero_()
        loss2.fill_(-1.0)
        g.replay()
        torch.cuda.synchronize()
        assert float(loss) == ref[0]
        assert torch.equal(out, ref[1])
        for a, b in zip(ref[2], gtab):
            assert torch.equal(a, b)
        assert torch.equal(dx, ref[3])
        for a, b in zip(ref[4], dw):
            assert torch.equal(a, b)
        assert float(loss2) == ref[5]
        assert torch.equal(dx2, ref[6])
        for a, b in zip(ref[7], dw2):
            assert torch.equal(a, b)
