"""Padded-dense brute force of HSTU attention, used only to pin the oracle.

It is deliberately built another way than the oracle: every sequence is padded
to a dense n_max x n_max problem, the mask is assembled from whole-matrix
pieces (lower triangle, context block, candidate diagonal), the buckets come
from vectorised NumPy (``np.frexp`` for the log2 time bucket), and the
attention is a batched dense matmul.  A torch float64 version of the same
dense construction gives autograd gradients.
"""
from __future__ import annotations

import numpy as np


def dense_mask(n, c, m):
    """Boolean [n, n] visibility matrix from whole-matrix pieces."""
    h_end = n - m
    M = np.tril(np.ones((n, n), dtype=bool))           # causal incl. diagonal
    M[:c, :c] = True                                    # context block, both ways
    M[:, h_end:] = False                                # nobody sees candidates ...
    idx = np.arange(h_end, n)
    M[idx, idx] = True                                  # ... except themselves
    return M


def dense_buckets(n, m, ts, P=128, Tb=64):
    h_end = n - m
    pos = np.minimum(np.arange(n), h_end)
    bp = np.minimum(np.abs(pos[:, None] - pos[None, :]), P - 1)
    bt = None
    if ts is not None:
        d = np.abs(ts[:, None].astype(np.int64) - ts[None, :].astype(np.int64))
        _, e = np.frexp(d.astype(np.float64))           # d = f * 2**e, f in [0.5, 1)
        bt = np.where(d == 0, 0, np.minimum(e, Tb - 1))
    return bp, bt


def pad_batch(offsets, arr, n_max):
    """[T, ...] jagged -> [B, n_max, ...] zero padded."""
    B = len(offsets) - 1
    out = np.zeros((B, n_max) + arr.shape[1:], dtype=arr.dtype)
    for b in range(B):
        s, e = offsets[b], offsets[b + 1]
        out[b, : e - s] = arr[s:e]
    return out


def forward(offsets, q, k, v, alpha, N, nt=None, nc=None, ts=None, rp=None, rt=None, u=None,
            norm="layernorm", eps=1e-5):
    """Returns (o [T,H,dv], y [T,H*dv]) in float64."""
    offsets = np.asarray(offsets)
    B = len(offsets) - 1
    T, H, _ = q.shape
    dv = v.shape[2]
    o = np.zeros((T, H, dv))
    for b in range(B):
        s, e = int(offsets[b]), int(offsets[b + 1])
        n = e - s
        if n == 0:
            continue
        c = int(nc[b]) if nc is not None else 0
        m = int(nt[b]) if nt is not None else 0
        M = dense_mask(n, c, m)
        bp, bt = dense_buckets(n, m, None if ts is None else ts[s:e],
                               rp.shape[1] if rp is not None else 128,
                               rt.shape[1] if rt is not None else 64)
        Q = np.transpose(q[s:e].astype(np.float64), (1, 0, 2))   # [H, n, d]
        K = np.transpose(k[s:e].astype(np.float64), (1, 0, 2))
        V = np.transpose(v[s:e].astype(np.float64), (1, 0, 2))
        Z = alpha * np.einsum("hid,hjd->hij", Q, K)
        if rp is not None:
            Z = Z + np.asarray(rp, np.float64)[:, bp]
        if rt is not None and ts is not None:
            Z = Z + np.asarray(rt, np.float64)[:, bt]
        A = np.where(M[None], Z / (1.0 + np.exp(-Z)) / N, 0.0)
        o[s:e] = np.transpose(np.einsum("hij,hjd->hid", A, V), (1, 0, 2))
    x = o.reshape(T, H * dv)
    if norm == "layernorm":
        mu = x.mean(axis=1, keepdims=True)
        var = ((x - mu) ** 2).mean(axis=1, keepdims=True)
        x = (x - mu) / np.sqrt(var + eps)
    y = x * (np.asarray(u, np.float64) if u is not None else 1.0)
    return o, y


def torch_forward(offsets, q, k, v, alpha, N, nt=None, nc=None, ts=None, rp=None, rt=None, u=None,
                  norm="layernorm", eps=1e-5):
    """Same dense construction in torch float64 (autograd-able inputs)."""
    import torch
    offsets = np.asarray(offsets)
    B = len(offsets) - 1
    T, H, _ = q.shape
    dv = v.shape[2]
    rows = []
    for b in range(B):
        s, e = int(offsets[b]), int(offsets[b + 1])
        n = e - s
        if n == 0:
            continue
        c = int(nc[b]) if nc is not None else 0
        m = int(nt[b]) if nt is not None else 0
        M = torch.from_numpy(dense_mask(n, c, m))
        bp, bt = dense_buckets(n, m, None if ts is None else ts[s:e],
                               rp.shape[1] if rp is not None else 128,
                               rt.shape[1] if rt is not None else 64)
        Q, K, V = (x[s:e].transpose(0, 1) for x in (q, k, v))
        Z = alpha * Q @ K.transpose(1, 2)
        if rp is not None:
            Z = Z + rp[:, torch.from_numpy(bp)]
        if rt is not None and ts is not None:
            Z = Z + rt[:, torch.from_numpy(bt)]
        A = torch.where(M[None], torch.nn.functional.silu(Z) / N, torch.zeros_like(Z))
        rows.append((A @ V).transpose(0, 1))
    o = torch.cat(rows, 0)
    x = o.reshape(T, H * dv)
    if norm == "layernorm":
        x = torch.nn.functional.layer_norm(x, (H * dv,), eps=eps)
    return o, (x * u if u is not None else x)
