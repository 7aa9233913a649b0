"""Expert-parallel forward on one GPU: several handles, each owning a range
of the physical experts, exchange rows by device copies (the loopback
exchange), and every rank's output must equal the single-handle forward of
its own batch bit for bit -- the rows meet the same codes, MMAs, epilogue and
combine order -- and so match the oracle at the layer tolerance.  Routing,
physical ids and the dispatch layout of each rank are checked exactly.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import synthetic
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch


def _batches(cfg, world, T):
    """One batch per rank: the same recipe, a different seed per rank."""
    return [synthetic.make_activations(dataclasses.replace(cfg, seed=cfg.seed + r), T) for r in range(world)]


def _ep_forward(torch, cfg, W, pmap, batches, first, recording=False):
    """Every rank's forward through the expert-parallel calls; the exchange is
    LoopbackExchange (device copies).  -> outputs, per-rank dumps, counts."""
    import moe_layer_serving_gb300 as mm
    from moe_layer_serving_gb300 import ep
    dev = torch.device("cuda:0")
    world = len(first) - 1
    ops, sends, offs, xs_dev = [], [], [], []
    for r in range(world):
        op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
        if pmap is not None:
            op.set_eplb_map(*pmap)
        op.set_expert_parallel(r, world, first)
        lo, hi = first[r], first[r + 1]
        op.set_weights(*[torch.from_numpy(np.ascontiguousarray(a[lo:hi])).to(dev) for a in W])
        T = batches[r][0].shape[0]
        op.ep_reserve(T, sum(op.ep_send_rows(b[0].shape[0]) for b in batches))
        op.set_recording(recording)
        hidden, logits, bias = batches[r]
        x = torch.from_numpy(hidden.view(np.int16)).to(dev).view(torch.bfloat16)
        lg, b = torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev)
        rows = op.ep_send_rows(T)
        sxq = torch.full((rows, cfg.H), 0x55, dtype=torch.uint8, device=dev)
        sxs = torch.full((rows, cfg.H // 32), 0x55, dtype=torch.uint8, device=dev)
        seid = torch.full((rows,), 12345, dtype=torch.int32, device=dev)
        off = op.ep_dispatch(x, lg, b, sxq, sxs, seid)
        assert off[-1] <= rows
        ops.append(op)
        sends.append((sxq, sxs, seid))
        offs.append(off)
        xs_dev.append(x)
    ex = ep.LoopbackExchange()
    recvs = ex.dispatch(sends, offs)
    y_recvs = []
    for r in range(world):
        rxq, rxs, reid = recvs[r]
        y = torch.empty((reid.shape[0], cfg.H), dtype=torch.bfloat16, device=dev)
        ops[r].ep_experts(rxq, rxs, reid, y)
        y_recvs.append(y)
    backs = ex.combine(y_recvs)
    outs, dumps, counts = [], [], []
    for r in range(world):
        out = torch.empty_like(xs_dev[r])
        ops[r].ep_combine(backs[r], out)
        torch.cuda.synchronize()
        assert ops[r].get_status() == 0
        outs.append(out.view(torch.int16).cpu().numpy().view(np.uint16))
        T = batches[r][0].shape[0]
        dumps.append({"idx": ops[r].debug_dump(0).reshape(T, cfg.k), "phys": ops[r].debug_dump(2).reshape(T, cfg.k),
                      "send": tuple(a.cpu().numpy() for a in sends[r]), "off": offs[r]})
        counts.append(ops[r].read_counts(0) if recording else None)
        ops[r].close()
    return outs, dumps, counts


def _single_forward(cfg, W, batch, recording=False):
    run = gpu_util.Run(cfg, W, cap=batch[0].shape[0])
    run.op.set_recording(recording)
    res = run.forward(*batch)
    counts = run.op.read_counts(0) if recording else None
    run.close()
    assert res["status"] == 0
    return res, counts


def _check_send_layout(cfg, dump, batch, first, pmap):
    """The send buffer of one rank against the oracle: routing, remap and the
    rows of every destination (codes, scales, local expert ids, pad rows)."""
    hidden, logits, bias = batch
    idx, _ = oracle.route(logits, bias, cfg.k)
    m, rc = pmap if pmap is not None else (np.arange(cfg.E, dtype=np.int32)[:, None], np.ones(cfg.E, np.int32))
    phys = oracle.eplb(idx, m, rc)
    assert np.array_equal(dump["idx"], idx)
    assert np.array_equal(dump["phys"], phys)
    xq_ref, xs_ref = oracle.mxfp8_quant_bf16(hidden)
    off_o, order, _ = oracle.permute(phys, cfg.P)
    sxq, sxs, seid = dump["send"]
    row_off = dump["off"]
    T = hidden.shape[0]
    row = 0
    for d in range(len(first) - 1):
        assert row_off[d] == row
        for p in range(first[d], first[d + 1]):
            pairs = order[off_o[p]:off_o[p + 1]]              # (t, j) in pair order
            n = pairs.size
            toks = pairs // cfg.k
            assert np.all(seid[row:row + n] == p - first[d])
            assert np.array_equal(sxq[row:row + n], xq_ref[toks])
            assert np.array_equal(sxs[row:row + n], xs_ref[toks])
            pad = (n + 15) // 16 * 16
            assert np.all(seid[row + n:row + pad] == -1)
            row += pad
    assert row_off[-1] == row
    assert T * cfg.k <= row


@pytest.mark.parametrize("world,T", [(2, 300), (3, 1100)])
def test_expert_parallel_matches_single_gpu_bit_for_bit(torch, world, T):
    # 20 physical experts (16 logical + 4 replicas) over 2 or 3 ranks, uneven
    # ranges; per rank a different batch; recording on
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=512, I=256, E=16, P=20, k=4, recording=True)
    W = gpu_util.weights(cfg)
    pmap = synthetic.make_eplb_map(cfg)[:2]
    first = [0, 9, 20] if world == 2 else [0, 5, 13, 20]
    batches = _batches(cfg, world, T)
    outs, dumps, counts = _ep_forward(torch, cfg, W, pmap, batches, first, recording=True)
    for r in range(world):
        _check_send_layout(cfg, dumps[r], batches[r], first, pmap)
        res, cnt = _single_forward(cfg, W, batches[r], recording=True)
        assert np.array_equal(outs[r], res["out"]), f"rank {r}: output differs from the single-GPU forward"
        assert np.array_equal(counts[r], cnt)
        ref = oracle.forward(*batches[r], cfg.k, W, *pmap)
        gpu_util.assert_out_close(outs[r], ref["out"], f"rank {r}")


def test_expert_parallel_decode_layer_two_ranks(torch):
    # the decode layer's shapes (H = 7168, I = 2048, 256 experts, top-6), two
    # ranks of 128 experts each, 64 tokens per rank
    cfg = synthetic.CONFIGS[1]
    W = gpu_util.weights(cfg)
    batches = _batches(cfg, 2, cfg.T)
    outs, dumps, _ = _ep_forward(torch, cfg, W, None, batches, [0, 128, 256])
    for r in range(2):
        _check_send_layout(cfg, dumps[r], batches[r], [0, 128, 256], None)
        res, _ = _single_forward(cfg, W, batches[r])
        assert np.array_equal(outs[r], res["out"]), f"rank {r}: output differs from the single-GPU forward"
    sel = gpu_util.sample_tokens(cfg.T, 12)
    ref = oracle.forward(batches[0][0][sel], batches[0][1][sel], batches[0][2], cfg.k, W, token_ids=sel)
    gpu_util.assert_out_close(outs[0][sel], ref["out"])


def test_expert_parallel_rank_with_no_rows_and_idle_batches(torch):
    # every token avoids rank 1's experts (it receives only what it sends to
    # itself: nothing), and an idle batch (T = 0) on one rank
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=40, E=8, P=8, k=2)
    W = gpu_util.weights(cfg)
    hidden, logits, bias = synthetic.make_activations(cfg)
    logits[:, 4:] -= 30.0                                  # experts 4..7 (rank 1) never selected
    first = [0, 4, 8]
    outs, dumps, _ = _ep_forward(torch, cfg, W, None, [(hidden, logits, bias)] * 2, first)
    assert dumps[0]["off"][1] == dumps[0]["off"][2]        # nothing bound for rank 1
    res, _ = _single_forward(cfg, W, (hidden, logits, bias))
    assert np.array_equal(outs[0], res["out"]) and np.array_equal(outs[1], res["out"])
    op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
    op.set_expert_parallel(0, 2, first)
    op.ep_reserve(16, 64)
    off = op.ep_dispatch(np.zeros((0, cfg.H), np.uint16), np.zeros((0, cfg.E), np.float32), None, None, None,
                         None, num_tokens=0)
    assert list(off) == [0, 0, 0]
    assert op.ep_send_rows(0) == 0
    # send buffers smaller than mm_ep_send_rows: refused before anything is enqueued
    dev = torch.device("cuda:0")
    x = torch.zeros((16, cfg.H), dtype=torch.bfloat16, device=dev)
    lg = torch.zeros((16, cfg.E), dtype=torch.float32, device=dev)
    short = op.ep_send_rows(16) - 1
    sxq = torch.empty((short, cfg.H), dtype=torch.uint8, device=dev)
    sxs = torch.empty((short, cfg.H // 32), dtype=torch.uint8, device=dev)
    seid = torch.empty((short,), dtype=torch.int32, device=dev)
    with pytest.raises(mm.MegaMoEError) as err:
        op.ep_dispatch(x, lg, None, sxq, sxs, seid)
    assert err.value.status == mm.MM_ERR_CAPACITY
    # the single-GPU calls are refused on an expert-parallel handle
    assert mm.lib().mm_forward(op.handle, None, None, None, None, 1, None) == mm.MM_ERR_UNSUPPORTED
    assert mm.lib().mm_set_shared_experts(op.handle, 1) == mm.MM_ERR_UNSUPPORTED
    assert mm.lib().mm_rebalance(op.handle, 0, 2) == mm.MM_ERR_UNSUPPORTED
    op.close()
