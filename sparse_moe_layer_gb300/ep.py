"""Expert-parallel dispatch and combine plans for the layer (host-side index logic).

Several GPUs can serve one MoE layer by partitioning its experts ("Hosting
Qwen on Blackwell", the sections on expert-parallel dispatch and combine;
"GPT-OSS on Day 0", combine paragraph: the weighted accumulation of the
experts' outputs): rank r owns the experts [first[r], first[r+1]).  Each rank
routes its own tokens and groups their rows by expert -- the permutation the
library's routing step already produces (moe_route_debug: offset, perm) -- so
the rows bound for one owner are one contiguous run of the permuted rows.

  dispatch  rank s sends rank r the rows [offset[first[r]], offset[first[r+1]])
            of its permuted xq / sx, with each row's expert
  regroup   rank r orders what it received by (expert, source rank, source row)
            so that every expert's rows are contiguous for the grouped GEMMs
  compute   the expert GEMMs on the regrouped rows (w[t,j] * y rows)
  return    the results go back in the order they arrived, so rank s gets its
            rows back in its own permuted order
  combine   rank s scatters row r to slot perm[r] and sums the k slots of every
            token in slot order, as the single-GPU combine does

Every row's expert arithmetic depends only on that row, so the result is the
single-GPU result bit for bit.  This module computes the plans and the bytes
the exchanges move; it moves no data.
"""
from __future__ import annotations

import numpy as np


def expert_ranges(E: int, world: int) -> np.ndarray:
    """First expert of each rank (int64 [world+1]): contiguous, sizes differing by at most one."""
    if world < 1 or E < world:
        raise ValueError("need 1 <= world <= E")
    return np.array([r * E // world for r in range(world + 1)], dtype=np.int64)


def owner_of(E: int, world: int) -> np.ndarray:
    """Rank owning each expert (int64 [E])."""
    first = expert_ranges(E, world)
    return np.searchsorted(first, np.arange(E), side="right") - 1


def dispatch_counts(offset: np.ndarray, first: np.ndarray) -> np.ndarray:
    """Rows this rank sends to each rank (int64 [world]): the permuted rows of the
    destination's experts, one contiguous run [offset[first[r]], offset[first[r+1]])."""
    offset = np.asarray(offset, np.int64)
    return offset[first[1:]] - offset[first[:-1]]


def counts_by_expert(offset: np.ndarray, first: np.ndarray, rank: int) -> np.ndarray:
    """Rows this rank sends for each expert that `rank` owns (int64 [experts of rank])."""
    offset = np.asarray(offset, np.int64)
    return np.diff(offset[first[rank]:first[rank + 1] + 1])


def regroup_order(recv_counts: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """recv_counts [sources, local experts]: rows received from each source rank
    for each owned expert, the sources' runs concatenated in source order and,
    inside a run, grouped by expert.  Returns (order, local_offset): the grouped
    buffer is received[order], and the rows of local expert e are
    [local_offset[e], local_offset[e+1]) in it, ordered by (source, source row)."""
    recv_counts = np.asarray(recv_counts, np.int64)
    nsrc, ne = recv_counts.shape
    run_start = np.concatenate([[0], np.cumsum(recv_counts.sum(axis=1))])  # where source s's run begins
    in_run = np.concatenate([np.zeros((nsrc, 1), np.int64), np.cumsum(recv_counts, axis=1)], axis=1)
    order = []
    for e in range(ne):
        for s in range(nsrc):
            a = run_start[s] + in_run[s, e]
            order.append(np.arange(a, a + recv_counts[s, e], dtype=np.int64))
    order = np.concatenate(order) if order else np.zeros(0, np.int64)
    local_offset = np.concatenate([[0], np.cumsum(recv_counts.sum(axis=0))]).astype(np.int64)
    return order, local_offset


def ungroup(grouped: np.ndarray, order: np.ndarray) -> np.ndarray:
    """Rows of the grouped buffer back in the order they were received."""
    out = np.empty_like(grouped)
    out[order] = grouped
    return out


def combine_slots(rows: np.ndarray, perm: np.ndarray, T: int, k: int) -> np.ndarray:
    """Permuted result rows (w[t,j] * y, [R, H]) -> token outputs [T, H]: row r goes
    to slot perm[r] = t*k + j, and the k slots of a token are summed in slot order."""
    slots = np.empty_like(rows)
    slots[np.asarray(perm, np.int64)] = rows
    slots = slots.reshape(T, k, -1)
    out = slots[:, 0].copy()
    for j in range(1, k):
        out = out + slots[:, j]
    return out


def exchange_bytes(send_counts: np.ndarray, rank: int, H: int) -> dict:
    """Bytes this rank puts on the wire per step for rows bound to other ranks:
    dispatch = e4m3 codes (Hp) + fp32 1x128 scales + the row's expert and slot
    (int32 each); combine = the fp32 result rows (H) coming back."""
    Hp = (H + 127) // 128 * 128
    remote = int(np.asarray(send_counts).sum() - np.asarray(send_counts)[rank])
    return dict(rows_remote=remote, dispatch=remote * (Hp + 4 * (Hp // 128) + 8), combine=remote * H * 4)
