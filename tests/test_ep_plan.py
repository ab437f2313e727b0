"""Expert-parallel dispatch / combine plans with two and three gloo ranks on the CPU.

Each rank routes its own token batch with the oracle (router, permutation, 1x128
x quantisation), dispatches its permuted rows to the experts' owners with
all_to_all_single, the owners regroup what they received by expert, apply a
per-row stand-in for the expert GEMMs, return the rows, and each rank combines
its slots.  The result must equal the same stand-in applied on one rank to the
whole permutation, bit for bit: the plans move every row to the right owner and
back to the right slot.  (The expert arithmetic itself is checked on the GPU
against the oracle; here only where rows go.)
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth
from sparse_moe_layer_gb300 import ep

T, H, I, E, K = 48, 256, 256, 8, 2


def _batch(rank: int):
    cfg = synth.LayerConfig(f"ep_rank{rank}", T, H, I, E, K, 40 + rank, "normal", "normal")
    x = synth.x_rows(cfg)
    rw, rb = synth.router(synth.LayerConfig("ep_router", T, H, I, E, K, 7, "normal", "normal"))
    r = oracle.router(x, rw, rb, K)
    p = oracle.permute(r["idx"], E)
    xq, sx = oracle.quant_rows_bf16(x)
    tok = p["perm"] // K
    rows = xq[tok].astype(np.float64) * sx[tok].repeat(128, axis=1)  # dequantised permuted rows [R, Hp]
    wts = synth.bf16_to_f32(r["w_bf16"]).astype(np.float64).reshape(-1)[p["perm"]]  # routing weight per row
    expert = np.repeat(np.arange(E), p["count"])
    return r, p, rows, wts, expert


def _expert_standin(rows: np.ndarray, expert: np.ndarray, wts: np.ndarray) -> np.ndarray:
    """A per-row function standing in for w * (expert GEMMs): depends on the row,
    its expert and its routing weight only."""
    return wts[:, None] * (rows[:, :H] * (expert[:, None] + 1.0) + np.sin(expert[:, None] + 0.25))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _a2a(send: np.ndarray, send_counts, recv_counts, dtype=torch.float64) -> np.ndarray:
    inp = torch.from_numpy(np.ascontiguousarray(send)).to(dtype)
    width = int(np.prod(send.shape[1:])) if send.ndim > 1 else 1
    out = torch.empty((int(sum(recv_counts)),) + tuple(send.shape[1:]), dtype=dtype)
    dist.all_to_all_single(out.view(-1), inp.view(-1), [int(c) * width for c in recv_counts],
                           [int(c) * width for c in send_counts])
    return out.numpy()


def _rank(rank: int, world: int, port: int, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, p, rows, wts, expert = _batch(rank)
        first = ep.expert_ranges(E, world)
        send = ep.dispatch_counts(p["offset"], first)
        # how many rows of each owned expert every source sends (one exchange of counts)
        per_dest = [ep.counts_by_expert(p["offset"], first, d) for d in range(world)]
        ne_max = int(np.diff(first).max())
        mat = np.zeros((world, ne_max), np.int64)
        for d in range(world):
            mat[d, :len(per_dest[d])] = per_dest[d]
        got = _a2a(mat, [1] * world, [1] * world, torch.int64).astype(np.int64)  # [source, local expert]
        recv_counts = got.sum(axis=1)
        ne = int(first[rank + 1] - first[rank])
        order, local_off = ep.regroup_order(got[:, :ne])
        # dispatch rows, their experts and routing weights
        rrows = _a2a(rows, send, recv_counts)
        rexp = _a2a(expert.astype(np.float64), send, recv_counts).astype(np.int64)
        rw = _a2a(wts, send, recv_counts)
        g_rows, g_exp, g_w = rrows[order], rexp[order], rw[order]
        assert np.all(np.diff(g_exp) >= 0) and np.all((g_exp >= first[rank]) & (g_exp < first[rank + 1]))
        assert np.array_equal(np.bincount(g_exp - first[rank], minlength=ne), np.diff(local_off))
        y = _expert_standin(g_rows, g_exp, g_w)
        back = _a2a(ep.ungroup(y, order), recv_counts, send)  # in this rank's permuted order again
        out_ep = ep.combine_slots(back, p["perm"], T, K)
        out_ref = ep.combine_slots(_expert_standin(rows, expert, wts), p["perm"], T, K)
        q.put((rank, bool(np.array_equal(out_ep, out_ref)), int(send[rank]), int(send.sum()),
               ep.exchange_bytes(send, rank, H)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ranks_dispatch_and_combine_equal_one_rank(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for pr in procs:
        pr.join(timeout=60)
        assert pr.exitcode == 0
    for rank, equal, local, total, nbytes in res:
        assert equal, f"rank {rank}: expert-parallel result differs from the one-rank result"
        assert total == T * K and 0 < local < total  # some rows stay, some travel
        assert nbytes["dispatch"] == nbytes["rows_remote"] * (256 + 4 * 2 + 8)


def test_plans_on_one_process():
    first = ep.expert_ranges(10, 3)
    assert first.tolist() == [0, 3, 6, 10]
    assert ep.owner_of(10, 3).tolist() == [0, 0, 0, 1, 1, 1, 2, 2, 2, 2]
    offset = np.array([0, 2, 2, 5, 6, 9, 9, 10, 12, 12, 15])
    assert ep.dispatch_counts(offset, first).tolist() == [5, 4, 6]
    assert ep.counts_by_expert(offset, first, 1).tolist() == [1, 3, 0]
    # two sources, two local experts: source 0 sent [2 of e0, 1 of e1], source 1 sent [0 of e0, 3 of e1]
    order, loff = ep.regroup_order(np.array([[2, 1], [0, 3]]))
    assert order.tolist() == [0, 1, 2, 3, 4, 5] and loff.tolist() == [0, 2, 6]
    order, loff = ep.regroup_order(np.array([[1, 1], [2, 1]]))
    assert order.tolist() == [0, 2, 3, 1, 4] and loff.tolist() == [0, 3, 5]
    g = np.arange(5.0)[:, None]
    assert np.array_equal(ep.ungroup(g[order], order), g)
    with pytest.raises(ValueError):
        ep.expert_ranges(2, 3)
