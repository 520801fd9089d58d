"""Seeded synthetic inputs for HSTU jagged attention.

This module only draws random numbers and lays them out in the jagged format.
It holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can take their inputs from it without sharing any computation.

Layout (the KeyedJaggedTensor convention from the TorchRec section,
"3.1.2 KeyedJaggedTensor" of the ai6s.net generative-recommendation survey):
sequences are packed back to back with no padding, and ``offsets`` is the
exclusive prefix sum of ``lengths`` (``offsets[b]`` is where sequence ``b``
starts, ``offsets[B]`` is the total token count T).

Per token the sequence holds, in order: ``num_contexts`` contextual prefix
tokens, the user history, then ``num_targets`` candidate items appended at the
end (ranking task, section "2.1.2", the candidates-at-the-end paragraph).

Value recipe (all from ``numpy.random.default_rng(seed)``, drawn in the order
lengths -> timestamps -> q, k, v, u, dy -> rab tables -> layer weights):

* q, k, v, u, dy ~ N(0, 1) float32, then rounded to bfloat16 (round to
  nearest even) when the batch dtype is bf16, so both sides read the same
  representable values.
* rab tables ~ N(0, 0.02): 128 relative-position buckets, 64 time buckets.
* timestamps: int64 seconds. Each sequence starts at 1.7e9 plus a random
  offset below 1e6; context tokens share that start time; each history token
  adds a gap round(Exp(mean 600 s)); all candidates share one request time,
  one more gap after the last history token.
* stochastic length (section "2.1.3", sparse optimisation): Zipf(1.2)
  lengths on [1, 8192] drawn by inverse CDF; a history longer than
  L = floor(8192**0.8) is cut to a uniform random ordered subset of L tokens
  with probability 1 - 8192**1.6 / n**2.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

NUM_POS_BUCKETS = 128
NUM_TIME_BUCKETS = 64


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)).astype(np.uint32)
    return r.view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of bf16-representable float32 values, as uint16."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def offsets_from_lengths(lengths) -> np.ndarray:
    """Exclusive prefix sum: offsets[0] = 0, offsets[b+1] = offsets[b] + lengths[b]."""
    lengths = np.asarray(lengths, dtype=np.int64)
    out = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(lengths, out=out[1:])
    return out


@dataclasses.dataclass
class Batch:
    name: str
    seed: int
    dtype: str                      # "bf16" or "fp32"
    B: int
    H: int
    d_qk: int
    d_v: int
    lengths: np.ndarray             # int64 [B], total length incl. context and targets
    offsets: np.ndarray             # int64 [B+1]
    num_targets: Optional[np.ndarray]   # int32 [B] or None
    num_contexts: Optional[np.ndarray]  # int32 [B] or None
    timestamps: Optional[np.ndarray]    # int64 [T] or None
    q: np.ndarray                   # float32 [T, H, d_qk]
    k: np.ndarray                   # float32 [T, H, d_qk]
    v: np.ndarray                   # float32 [T, H, d_v]
    u: Optional[np.ndarray]         # float32 [T, H*d_v] or None
    dy: Optional[np.ndarray]        # float32 [T, H*d_v] or None (forward-only batches)
    rab_pos: Optional[np.ndarray]   # float32 [H, 128] or None
    rab_time: Optional[np.ndarray]  # float32 [H, 64] or None
    alpha: float
    max_seq_len: int                # N of the 1/N scale
    norm: str = "layernorm"         # "layernorm" or "none"
    eps: float = 1e-5
    backward: bool = True
    # full-layer extras (model dim D = H*d_v)
    x: Optional[np.ndarray] = None      # float32 [T, D]
    w1: Optional[np.ndarray] = None     # float32 [D, 4*D]  (columns: U | V | Q | K)
    w2: Optional[np.ndarray] = None     # float32 [D, D]
    dout: Optional[np.ndarray] = None   # float32 [T, D]

    @property
    def T(self) -> int:
        return int(self.offsets[-1])


def _normal(rng, shape, dtype, std=1.0):
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return bf16_round(a) if dtype == "bf16" else a


def _zipf_lengths(rng, count, s=1.2, n_max=8192):
    support = np.arange(1, n_max + 1, dtype=np.float64)
    cdf = np.cumsum(support ** (-s))
    cdf /= cdf[-1]
    return np.searchsorted(cdf, rng.random(count), side="left").astype(np.int64) + 1


def _timestamps(rng, n_ctx, n_hist, n_tgt, n_hist_full=None, keep=None):
    """Integer-second timestamps for one sequence (see the module docstring)."""
    t0 = int(1_700_000_000 + rng.integers(0, 1_000_000))
    nh = n_hist if n_hist_full is None else n_hist_full
    gaps = np.rint(rng.exponential(600.0, size=nh + 1)).astype(np.int64)
    hist = t0 + np.cumsum(gaps[:nh])
    if keep is not None:
        hist = hist[keep]
    last = hist[-1] if len(hist) else t0
    req = last + gaps[nh]
    return np.concatenate([np.full(n_ctx, t0, np.int64), hist,
                           np.full(n_tgt, req, np.int64)]).astype(np.int64)


def make_batch(lengths_hist, *, H, d_qk, d_v, dtype="bf16", num_contexts=0,
               num_targets=0, with_time=True, with_rab=True, backward=True,
               seed=0, name="custom", alpha=None, max_seq_len=None,
               norm="layernorm", with_u=True, rng=None, sl_keep=None,
               hist_full=None) -> Batch:
    """Build a batch from per-sequence history lengths.

    ``num_contexts`` / ``num_targets`` are ints (same for every sequence) or
    per-sequence arrays.  Total length = contexts + history + targets.
    """
    rng = np.random.default_rng(seed) if rng is None else rng
    hist = np.asarray(lengths_hist, dtype=np.int64)
    B = len(hist)
    nc = np.broadcast_to(np.asarray(num_contexts, dtype=np.int64), (B,)).copy()
    nt = np.broadcast_to(np.asarray(num_targets, dtype=np.int64), (B,)).copy()
    lengths = nc + hist + nt
    offsets = offsets_from_lengths(lengths)
    T = int(offsets[-1])
    ts = None
    if with_time:
        parts = []
        for b in range(B):
            keep = None if sl_keep is None else sl_keep[b]
            full = None if hist_full is None else int(hist_full[b])
            parts.append(_timestamps(rng, int(nc[b]), int(hist[b]), int(nt[b]),
                                     n_hist_full=full, keep=keep))
        ts = np.concatenate(parts) if parts else np.zeros(0, np.int64)
        assert ts.shape[0] == T
    q = _normal(rng, (T, H, d_qk), dtype)
    k = _normal(rng, (T, H, d_qk), dtype)
    v = _normal(rng, (T, H, d_v), dtype)
    u = _normal(rng, (T, H * d_v), dtype) if with_u else None
    dy = _normal(rng, (T, H * d_v), dtype) if backward else None
    rp = rt = None
    if with_rab:
        rp = _normal(rng, (H, NUM_POS_BUCKETS), "fp32", std=0.02)
        rt = _normal(rng, (H, NUM_TIME_BUCKETS), "fp32", std=0.02) if with_time else None
    return Batch(
        name=name, seed=seed, dtype=dtype, B=B, H=H, d_qk=d_qk, d_v=d_v,
        lengths=lengths, offsets=offsets,
        num_targets=nt.astype(np.int32) if np.any(nt) else None,
        num_contexts=nc.astype(np.int32) if np.any(nc) else None,
        timestamps=ts, q=q, k=k, v=v, u=u, dy=dy, rab_pos=rp, rab_time=rt,
        alpha=float(alpha if alpha is not None else 1.0 / math.sqrt(d_qk)),
        max_seq_len=int(max_seq_len if max_seq_len is not None
                        else (max(int(lengths.max()), 1) if B else 1)),
        norm=norm, backward=backward)


# ---------------------------------------------------------------------------
# The five named workloads.

CONFIG_NAMES = ("tiny_fp32", "retrieval", "ranking", "heavy_tailed", "layer")


def tiny_fp32(seed=0) -> Batch:
    """4 sequences of lengths 7/16/31/50, 2 heads of 32, FP32, causal only,
    no rab, N = 50, alpha = 1/sqrt(32); forward and backward."""
    return make_batch([7, 16, 31, 50], H=2, d_qk=32, d_v=32, dtype="fp32",
                      with_time=False, with_rab=False, seed=seed,
                      name="tiny_fp32", max_seq_len=50)


def retrieval(seed=0) -> Batch:
    """32 sequences, lengths clip(round(LogNormal(5, 1)), 16, 1024), 4 heads
    of 64, BF16, causal, position+time rab; forward only."""
    rng = np.random.default_rng(seed)
    n = np.clip(np.rint(rng.lognormal(5.0, 1.0, size=32)), 16, 1024).astype(np.int64)
    return make_batch(n, H=4, d_qk=64, d_v=64, rng=rng, seed=seed,
                      name="retrieval", backward=False)


def ranking(seed=0) -> Batch:
    """16 sequences, history ~ U[256, 3968] plus 8 context tokens in front and
    64 candidates at the end, 4 heads of 128, BF16; forward and backward."""
    rng = np.random.default_rng(seed)
    hist = rng.integers(256, 3968, size=16, endpoint=True).astype(np.int64)
    return make_batch(hist, H=4, d_qk=128, d_v=128, num_contexts=8,
                      num_targets=64, rng=rng, seed=seed, name="ranking")


SL_N_MAX = 8192
SL_ALPHA = 1.6


def stochastic_length(rng, n_hist: np.ndarray):
    """Stochastic-length sampling: returns (kept lengths, per-sequence kept
    index arrays or None).  L = floor(8192**0.8); a history with n > L is cut
    to L with probability 1 - 8192**1.6 / n**2."""
    L = int(math.floor(SL_N_MAX ** (SL_ALPHA / 2)))
    out = n_hist.copy()
    keeps = []
    for b, n in enumerate(n_hist):
        n = int(n)
        keep = None
        if n > L:
            p_cut = 1.0 - (SL_N_MAX ** SL_ALPHA) / float(n * n)
            if rng.random() < p_cut:
                keep = np.sort(rng.choice(n, size=L, replace=False))
                out[b] = L
        keeps.append(keep)
    return out, keeps


def heavy_tailed(seed=0) -> Batch:
    """64 sequences, Zipf(1.2) history lengths on [1, 8192] after
    stochastic-length sampling, plus 32 candidates each, 4 heads of 128,
    BF16, causal + target mask + rab; forward and backward."""
    rng = np.random.default_rng(seed)
    full = _zipf_lengths(rng, 64)
    kept, keeps = stochastic_length(rng, full)
    return make_batch(kept, H=4, d_qk=128, d_v=128, num_targets=32, rng=rng,
                      seed=seed, name="heavy_tailed", sl_keep=keeps,
                      hist_full=full)


def layer(seed=0, n_lo=8192, n_hi=32768, B=8) -> Batch:
    """Full HSTU layer: 8 sequences with history ~ U[8192, 32768] plus 128
    candidates, model dim 512 = 4 heads of 128; X ~ N(0,1), W1 [512, 2048]
    and W2 [512, 512] ~ N(0, 0.02), all BF16; forward and backward.

    q/k/v/u of the returned batch are unused placeholders of shape [T,H,0]:
    the layer derives them from X @ W1."""
    rng = np.random.default_rng(seed)
    hist = rng.integers(n_lo, n_hi, size=B, endpoint=True).astype(np.int64)
    nt = 128
    lengths = hist + nt
    offsets = offsets_from_lengths(lengths)
    T = int(offsets[-1])
    H, d = 4, 128
    D = H * d
    ts = np.concatenate([_timestamps(rng, 0, int(h), nt) for h in hist])
    x = _normal(rng, (T, D), "bf16")
    dout = _normal(rng, (T, D), "bf16")
    rp = _normal(rng, (H, NUM_POS_BUCKETS), "fp32", std=0.02)
    rt = _normal(rng, (H, NUM_TIME_BUCKETS), "fp32", std=0.02)
    w1 = _normal(rng, (D, 4 * D), "bf16", std=0.02)
    w2 = _normal(rng, (D, D), "bf16", std=0.02)
    empty = np.zeros((T, H, 0), np.float32)
    return Batch(name="layer", seed=seed, dtype="bf16", B=B, H=H, d_qk=d, d_v=d,
                 lengths=lengths, offsets=offsets,
                 num_targets=np.full(B, nt, np.int32), num_contexts=None,
                 timestamps=ts, q=empty, k=empty, v=empty, u=None, dy=None,
                 rab_pos=rp, rab_time=rt, alpha=1.0 / math.sqrt(d),
                 max_seq_len=int(lengths.max()), x=x, w1=w1, w2=w2, dout=dout)


def by_name(name: str, seed: int = 0) -> Batch:
    return {"tiny_fp32": tiny_fp32, "retrieval": retrieval, "ranking": ranking,
            "heavy_tailed": heavy_tailed, "layer": layer}[name](seed)
