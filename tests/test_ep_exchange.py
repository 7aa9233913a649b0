"""The expert-parallel exchange on CPU: two gloo ranks, each with its own
batch, move their dispatch rows to the ranks owning the experts and the y
rows back through moe_layer_serving_gb300.ep.DistExchange.  The rows are
built in the send-buffer layout mm_ep_dispatch writes (segments of each
destination's experts in expert order, pairs in (token, slot) order, padded
to 16 rows with expert id -1), computed by the oracle, and the combined
output of every rank must equal oracle.forward of that rank's batch bit for
bit: the exchange's bookkeeping -- split sizes, source order, the way back --
may not move any row.  No GPU."""
import dataclasses
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg():
    import synthetic
    return dataclasses.replace(synthetic.CONFIGS[0], T=40, E=8, P=10, k=2)


def _send_buffer(cfg, hidden, logits, bias, pmap, first):
    """The send buffer of one rank from the oracle's stages, in the layout of
    mm_ep_dispatch; returns (xq, xs, eid, row_off, row of each pair, w)."""
    import oracle
    idx, w = oracle.route(logits, bias, cfg.k)
    phys = oracle.eplb(idx, *pmap)
    xq, xs = oracle.mxfp8_quant_bf16(hidden)
    off, order, _ = oracle.permute(phys, cfg.P)
    rows = []
    eid = []
    row_of_pair = np.empty(idx.size, np.int64)
    row_off = [0]
    for d in range(len(first) - 1):
        for p in range(first[d], first[d + 1]):
            pairs = order[off[p]:off[p + 1]]
            for q in pairs:
                row_of_pair[q] = len(rows)
                rows.append(q // cfg.k)
                eid.append(p - first[d])
            pad = (-pairs.size) % 16
            rows.extend([-1] * pad)
            eid.extend([-1] * pad)
        row_off.append(len(rows))
    rows = np.array(rows)
    bx = np.zeros((rows.size, cfg.H), np.uint8)
    bs = np.zeros((rows.size, cfg.H // 32), np.uint8)
    bx[rows >= 0] = xq[rows[rows >= 0]]
    bs[rows >= 0] = xs[rows[rows >= 0]]
    return bx, bs, np.array(eid, np.int32), row_off, row_of_pair, w


def _rank(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    import synthetic
    from moe_layer_serving_gb300 import ep
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = _cfg()
        W = synthetic.make_all_weights(cfg)
        m, rc, _ = synthetic.make_eplb_map(cfg)
        first = [0, 4, 10]                                  # uneven expert ranges
        hidden, logits, bias = synthetic.make_activations(dataclasses.replace(cfg, seed=rank), cfg.T + 7 * rank)
        bx, bs, eid, row_off, row_of_pair, w = _send_buffer(cfg, hidden, logits, bias, (m, rc), first)
        ex = ep.DistExchange()
        sp = ep.splits(row_off)
        rxq, rxs, reid, rsp = ex.dispatch(torch.from_numpy(bx), torch.from_numpy(bs), torch.from_numpy(eid), sp)
        assert sum(rsp) == reid.shape[0]
        # the receiving rank's experts over the received rows (the oracle's FFN)
        y_recv = np.zeros((reid.shape[0], cfg.H), np.float32)
        reid = reid.numpy()
        for e in range(first[rank + 1] - first[rank]):
            at = np.nonzero(reid == e)[0]
            if at.size:
                p = first[rank] + e
                y_recv[at] = oracle.expert_ffn(rxq.numpy()[at], rxs.numpy()[at], *(a[p] for a in W))["y"]
        y_back = ex.combine(torch.from_numpy(y_recv), sp, rsp).numpy()
        assert y_back.shape[0] == row_off[-1]
        got = oracle.combine(w, y_back[row_of_pair])
        ref = oracle.forward(hidden, logits, bias, cfg.k, W, m, rc)
        out[rank] = (bool(np.array_equal(got, ref["out"])), rsp, sp)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_rows_and_return_y_in_send_order():
    world, port = 2, _free_port()
    with tmp.Manager() as mgr:
        out = mgr.dict()
        tmp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] and res[1][0]
    # what rank s sent to rank d is what d received from s
    assert res[0][1][1] == res[1][2][0] and res[1][1][0] == res[0][2][1]


def test_splits_and_loopback_bookkeeping():
    from moe_layer_serving_gb300 import ep
    assert ep.splits([0, 16, 16, 48]) == [16, 0, 32]
    with pytest.raises(ValueError):
        ep.splits([0, 16, 8])
    with pytest.raises(ValueError):
        ep.splits([4, 16])
    # loopback: three ranks, rows tagged (source, destination, index)
    lb = ep.LoopbackExchange()
    offs = [[0, 2, 2, 5], [0, 1, 4, 4], [0, 0, 3, 6]]
    sends = []
    for s, o in enumerate(offs):
        tag = torch.zeros(o[-1], dtype=torch.int32)
        for d in range(3):
            tag[o[d]:o[d + 1]] = 100 * s + 10 * d + torch.arange(o[d + 1] - o[d], dtype=torch.int32)
        sends.append((tag.clone(), tag.clone(), tag.clone()))
    recvs = lb.dispatch(sends, offs)
    for d in range(3):
        want = torch.cat([sends[s][0][offs[s][d]:offs[s][d + 1]] for s in range(3)])
        assert torch.equal(recvs[d][0], want)
    backs = lb.combine([r[0] for r in recvs])
    for s in range(3):
        assert torch.equal(backs[s], sends[s][0])
