"""Data-parallel helpers for HSTU jagged attention.

The attention path shards by sequence with no exchange inside it: each rank
runs whole sequences.  A data-parallel training step needs one exchange, the
sum over ranks of the gradients of the shared parameters: the d_rab tables
(H x (P + Tb) floats) and, for the full layer, dW1 and dW2; the benchmark
needs the step time (max over ranks) and the work done (sum over ranks).  Everything here is host logic plus torch.distributed collectives on
whatever backend the process group uses (NCCL on GPUs, gloo on CPUs).
"""
from __future__ import annotations

import heapq
from typing import List, Sequence

import numpy as np

from . import synth


def sequence_costs(batch) -> np.ndarray:
    """Allowed (query, key) pairs of each sequence (the work it brings)."""
    n = batch.lengths.astype(np.int64)
    c = batch.num_contexts.astype(np.int64) if batch.num_contexts is not None else np.zeros_like(n)
    m = batch.num_targets.astype(np.int64) if batch.num_targets is not None else np.zeros_like(n)
    h_end = n - m
    return h_end * (h_end + 1) // 2 + c * (c - 1) // 2 + m * (h_end + 1)


def lpt_shard(costs: Sequence[int], world: int) -> List[List[int]]:
    """Longest-processing-time-first assignment of sequences to ranks: each
    sequence, largest first, goes to the rank with the least work so far.
    Ties break by rank, then by sequence index, so every rank computes the
    same answer.  Returns the sequence indices of each rank, in index order."""
    order = sorted(range(len(costs)), key=lambda i: (-int(costs[i]), i))
    heap = [(0, r) for r in range(world)]
    out: List[List[int]] = [[] for _ in range(world)]
    for i in order:
        load, r = heapq.heappop(heap)
        out[r].append(i)
        heapq.heappush(heap, (load + int(costs[i]), r))
    return [sorted(x) for x in out]


def gather_sequences(batch, idx: Sequence[int]):
    """A new jagged batch holding the sequences idx of batch (same N, alpha,
    tables and, for a layer batch, the same weights): data movement only."""
    idx = list(idx)
    off = batch.offsets
    rows = np.concatenate([np.arange(off[i], off[i + 1]) for i in idx]) if idx else np.zeros(0, np.int64)
    take = lambda a: None if a is None else a[rows]
    lengths = batch.lengths[idx].copy()
    return synth.Batch(
        name=batch.name, seed=batch.seed, dtype=batch.dtype, B=len(idx), H=batch.H, d_qk=batch.d_qk,
        d_v=batch.d_v, lengths=lengths, offsets=synth.offsets_from_lengths(lengths),
        num_targets=None if batch.num_targets is None else batch.num_targets[idx].copy(),
        num_contexts=None if batch.num_contexts is None else batch.num_contexts[idx].copy(),
        timestamps=take(batch.timestamps), q=batch.q[rows], k=batch.k[rows], v=batch.v[rows],
        u=take(batch.u), dy=take(batch.dy), rab_pos=batch.rab_pos, rab_time=batch.rab_time,
        alpha=batch.alpha, max_seq_len=batch.max_seq_len, norm=batch.norm, eps=batch.eps,
        backward=batch.backward, x=take(batch.x), w1=batch.w1, w2=batch.w2, dout=take(batch.dout))


def allreduce_sum_(tensors, group=None):
    """In-place sum over ranks of each tensor (the d_rab gradients)."""
    import torch.distributed as dist
    for t in tensors:
        if t is not None:
            dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return tensors


def reduce_step_time(elapsed_ms: float, work: float, device="cpu", group=None):
    """(max elapsed over ranks, sum of work over ranks) for a timed region."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
    w = torch.tensor([float(work)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(w, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(w.item())
