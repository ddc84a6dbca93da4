"""A CPU backend for vocab_sharded_lm_gb300.distributed, built on the fp64
oracle: lets world-size-2 gloo ranks exercise the multi-process
orchestration (the exchange, its order, the combine on every rank and the
communication-free backward) without a GPU.  Test infrastructure only."""
import numpy as np
import torch

from oracle import vpce_oracle as O


class OracleBackend:
    def new_workspace(self, t_local, s, device):
        return {}

    def partials(self, shards, vocab_start, targets, ignore_index, workspace, stream=None):
        y = targets.numpy()
        part, tgt = [], np.zeros(len(y))
        for i, z in enumerate(shards):
            m, se, tg = O.shard_partials(z.numpy(), y, vocab_start[i], vocab_start[i + 1])
            part.append(np.stack([m, se], axis=1))
            tgt += tg
        return torch.tensor(np.stack(part)), torch.tensor(tgt)

    def fold(self, part, stream=None):
        p = part.numpy()
        m, se = O.fold_partials(p[:, :, 0], p[:, :, 1])
        return torch.tensor(np.stack([m, se], axis=1)[None])

    def combine(self, part, tgt, V, targets, ignore_index, reduction, t_local, workspace, stream=None):
        y = targets.numpy()
        p = part.numpy()
        cards = [(p[i, :, 0], p[i, :, 1], tgt.numpy() if i == 0 else np.zeros(len(y))) for i in range(p.shape[0])]
        lse, row_loss, mean = O.combine_sharded(cards, y, V, ignore_index)
        workspace["lse"] = lse
        workspace["n_valid"] = int(np.sum((y != ignore_index) & (y >= 0) & (y < V)))
        workspace["reduction"] = reduction
        loss = {"mean": mean, "sum": float(np.nansum(row_loss)), "none": row_loss}[reduction]
        return torch.tensor(loss, dtype=torch.float64), torch.tensor(row_loss, dtype=torch.float64)

    def backward(self, shards, vocab_start, targets, ignore_index, workspace, grad_output, stream=None):
        y = targets.numpy()
        lse = workspace["lse"]
        scale = grad_output / workspace["n_valid"] if workspace["reduction"] == "mean" else grad_output
        for i, z in enumerate(shards):
            lo, hi = vocab_start[i], vocab_start[i + 1]
            d = np.exp(z.numpy() - lse[:, None])
            rows = np.nonzero((y >= lo) & (y < hi))[0]
            d[rows, y[rows] - lo] -= 1.0
            d *= scale
            d[y == ignore_index] = 0.0
            z.copy_(torch.tensor(d))
        return shards
