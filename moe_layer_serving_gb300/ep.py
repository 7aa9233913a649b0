"""Expert-parallel forward of the fused MoE layer across ranks.

The pages run the operator expert-parallel over eight GPUs with all-to-all
dispatch and combine ("sglang PR #35619", launch settings).  Here each rank
is one ``MegaMoE`` handle that owns a contiguous range of the physical
experts (``set_expert_parallel``); a forward is

    op.ep_dispatch      route, quantise and pack the rank's tokens; rows for
                        rank d are send[row_off[d]:row_off[d+1]]
    exchange.dispatch   all-to-all: every rank receives its ranges
    op.ep_experts       the rank's experts over the received rows
    exchange.combine    all-to-all back: y rows return in send order
    op.ep_combine       weighted combine into the output

This module only moves rows between ranks and keeps the split sizes: every
step of the layer's arithmetic runs in the library's kernels.  Two exchanges:
``DistExchange`` over ``torch.distributed`` (NCCL between GPUs, gloo on CPU),
and ``LoopbackExchange`` for ranks held by one process (device copies).
"""
from __future__ import annotations

import numpy as np


def splits(row_off) -> list[int]:
    """Rows per destination rank from the row offsets of one dispatch."""
    off = np.asarray(row_off, np.int64)
    if off.ndim != 1 or off.size < 2 or off[0] != 0 or np.any(np.diff(off) < 0):
        raise ValueError(f"row offsets must start at 0 and not decrease: {off}")
    return [int(x) for x in np.diff(off)]


class DistExchange:
    """All-to-all of the dispatch rows and of the returned y rows over a
    torch.distributed process group (one rank per process)."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist, self.group = dist, group
        self.world = dist.get_world_size(group)

    def _counts(self, send_splits, device):
        import torch
        if len(send_splits) != self.world:
            raise ValueError(f"{len(send_splits)} splits for {self.world} ranks")
        s = torch.tensor(send_splits, dtype=torch.int64, device=device)
        r = torch.empty_like(s)
        self.dist.all_to_all_single(r, s, group=self.group)
        return [int(x) for x in r.cpu()]

    def _rows(self, t, send_splits, recv_splits):
        import torch
        out = torch.empty((sum(recv_splits),) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        self.dist.all_to_all_single(out, t[:sum(send_splits)].contiguous(), recv_splits, send_splits,
                                    group=self.group)
        return out

    def dispatch(self, send_xq, send_xs, send_eid, send_splits):
        """-> (recv_xq, recv_xs, recv_eid, recv_splits): this rank's rows from every
        rank, concatenated in source-rank order."""
        recv_splits = self._counts(send_splits, send_eid.device)
        return (self._rows(send_xq, send_splits, recv_splits), self._rows(send_xs, send_splits, recv_splits),
                self._rows(send_eid, send_splits, recv_splits), recv_splits)

    def combine(self, y_recv, send_splits, recv_splits):
        """-> y_back: the y rows of this rank's own dispatch, in its send order."""
        return self._rows(y_recv, recv_splits, send_splits)


class LoopbackExchange:
    """The same exchange for all ranks held by one process (one GPU, or one
    process driving several): rows move by device copies."""

    def dispatch(self, sends, row_offs):
        """sends[s] = (send_xq, send_xs, send_eid) of rank s, row_offs[s] its row
        offsets.  -> per destination rank d: (recv_xq, recv_xs, recv_eid), rows
        from ranks 0, 1, ... in that order."""
        import torch
        world = len(sends)
        sp = [splits(o) for o in row_offs]
        recvs = []
        for d in range(world):
            parts = [[], [], []]
            for s in range(world):
                lo, hi = int(row_offs[s][d]), int(row_offs[s][d + 1])
                for i in range(3):
                    parts[i].append(sends[s][i][lo:hi])
            recvs.append(tuple(torch.cat(p) for p in parts))
        self._sp = sp
        return recvs

    def combine(self, y_recvs):
        """y_recvs[d] = y rows of destination d in its receive order -> per source
        rank s: y_back in s's send order."""
        import torch
        world = len(y_recvs)
        sp = self._sp
        # where source s's rows start inside destination d's receive buffer
        start = [[sum(sp[q][d] for q in range(s)) for d in range(world)] for s in range(world)]
        backs = []
        for s in range(world):
            backs.append(torch.cat([y_recvs[d][start[s][d]:start[s][d] + sp[s][d]] for d in range(world)]))
        return backs


class ExpertParallelMoE:
    """One rank of the expert-parallel layer over a torch.distributed group."""

    def __init__(self, op, exchange: DistExchange, max_tokens: int, max_recv_rows: int):
        """op: a MegaMoE handle already made a rank (set_expert_parallel) with its
        experts' weights set."""
        import torch
        self.op, self.ex = op, exchange
        op.ep_reserve(max_tokens, max_recv_rows)
        rows = op.ep_send_rows(max_tokens)
        dev = torch.device("cuda", torch.cuda.current_device())
        self.send_xq = torch.empty((rows, op.H), dtype=torch.uint8, device=dev)
        self.send_xs = torch.empty((rows, op.H // 32), dtype=torch.uint8, device=dev)
        self.send_eid = torch.empty((rows,), dtype=torch.int32, device=dev)

    def forward(self, hidden, logits, bias, out, stream=None):
        import torch
        row_off = self.op.ep_dispatch(hidden, logits, bias, self.send_xq, self.send_xs, self.send_eid,
                                      stream=stream)
        sp = splits(row_off)
        rxq, rxs, reid, rsp = self.ex.dispatch(self.send_xq, self.send_xs, self.send_eid, sp)
        y_recv = torch.empty((reid.shape[0], self.op.H), dtype=torch.bfloat16, device=reid.device)
        self.op.ep_experts(rxq, rxs, reid, y_recv, stream=stream)
        y_back = self.ex.combine(y_recv, sp, rsp)
        self.op.ep_combine(y_back, out, stream=stream)
        return out
