"""NumPy front end of the FP64 CPU oracle for HSTU jagged attention.

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  Nothing here is shared
with the CUDA path.

All floating-point inputs are widened to float64 (bf16/fp32 values widen
exactly), all computation is float64 in ``hstu_oracle.c`` or in NumPy.
The full HSTU layer (ai6s.net survey, section 2.1.2: pointwise projection
eq. (1), spatial aggregation eq. (2), pointwise transformation eq. (3), with
residual connections between layers) is composed here from NumPy matmuls and
the C attention routines:

    [U | V | Q | K] = SiLU(X W1)           (split in that order, no bias)
    Y   = LayerNorm(attention(Q, K, V)) * U
    out = X + Y W2                         (no bias)

The optional fused dropout on Y draws its keep decisions from Philox4x64-10
(a counter-based generator, written out here from its published
definition), so both sides derive the same mask from (seed, offset).
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from .build import build_oracle

_lib = None

P_DEFAULT = 128
TB_DEFAULT = 64


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build_oracle())
        i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        _lib.hstu_oracle_fwd.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp, i32,
                                         dbl, dbl, vp, vp, vp, vp, vp]
        _lib.hstu_oracle_norm_gate.argtypes = [i64, i32, i32, dbl, vp, vp, vp, vp, vp, vp]
        _lib.hstu_oracle_norm_gate_bwd.argtypes = [i64, i32, i32, dbl, vp, vp, vp, vp, vp, vp]
        _lib.hstu_oracle_attn_bwd.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, i32, vp, i32,
                                              dbl, dbl, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
        _lib.hstu_oracle_tile_count.argtypes = [i32, vp, i32, i32]
        _lib.hstu_oracle_tile_count.restype = i64
        _lib.hstu_oracle_tile_classes.argtypes = [i32, vp, vp, vp, i32, i32, vp, vp, vp, vp, vp]
        _lib.hstu_oracle_allowed_pairs.argtypes = [i32, vp, vp, vp, vp]
        _lib.hstu_oracle_time_bucket.argtypes = [i64, i64, i32]
        _lib.hstu_oracle_pos_bucket.argtypes = [i64, i64, i64, i32]
        _lib.hstu_oracle_num_threads.restype = i32
    return _lib


def num_threads() -> int:
    return int(lib().hstu_oracle_num_threads())


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.float64)


def _i64(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int64)


def _i32(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.int32)


def _u8(a):
    return None if a is None else np.ascontiguousarray(a, dtype=np.uint8)


def time_bucket(ti: int, tj: int, Tb: int = TB_DEFAULT) -> int:
    return int(lib().hstu_oracle_time_bucket(int(ti), int(tj), int(Tb)))


def pos_bucket(i: int, j: int, h_end: int, P: int = P_DEFAULT) -> int:
    return int(lib().hstu_oracle_pos_bucket(int(i), int(j), int(h_end), int(P)))


class Problem:
    """The attention inputs in float64 / int64, in the jagged layout."""

    def __init__(self, offsets, q, k, v, alpha, N, num_targets=None, num_contexts=None,
                 timestamps=None, rab_pos=None, rab_time=None):
        self.offsets = _i64(offsets)
        self.B = len(self.offsets) - 1
        self.q, self.k, self.v = _f64(q), _f64(k), _f64(v)
        self.T, self.H, self.dqk = self.q.shape
        self.dv = self.v.shape[2]
        self.alpha, self.N = float(alpha), float(N)
        self.nt, self.nc = _i32(num_targets), _i32(num_contexts)
        self.ts = _i64(timestamps)
        self.rp, self.rt = _f64(rab_pos), _f64(rab_time)
        self.P = self.rp.shape[1] if self.rp is not None else P_DEFAULT
        self.Tb = self.rt.shape[1] if self.rt is not None else TB_DEFAULT

    @classmethod
    def from_batch(cls, b, q=None, k=None, v=None):
        return cls(b.offsets, b.q if q is None else q, b.k if k is None else k,
                   b.v if v is None else v, b.alpha, b.max_seq_len, b.num_targets,
                   b.num_contexts, b.timestamps, b.rab_pos, b.rab_time)

    def _head(self):
        return (self.B, self.H, self.dqk, self.dv, _p(self.offsets), _p(self.nt), _p(self.nc),
                _p(self.ts), _p(self.rp), self.P, _p(self.rt), self.Tb, self.alpha, self.N)


def attn_fwd(pb: Problem, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """o [T, H, dv] float64; rows (bool/uint8 [T]) restricts the computed rows
    (the others are returned as zeros)."""
    o = np.zeros((pb.T, pb.H, pb.dv), np.float64)
    rows = _u8(rows)
    rc = lib().hstu_oracle_fwd(*pb._head(), _p(pb.q), _p(pb.k), _p(pb.v), _p(o), _p(rows))
    if rc != 0:
        raise ValueError("oracle: invalid jagged metadata")
    return o


def norm_gate(o, u, norm="layernorm", eps=1e-5, rows=None):
    """y [T, F], mean [T], rstd [T] from o [T, H, dv] (or [T, F]) and u [T, F] (or None)."""
    o = _f64(o).reshape(o.shape[0], -1)
    T, F = o.shape
    u = _f64(u)
    y = np.zeros((T, F), np.float64)
    mean = np.zeros(T, np.float64)
    rstd = np.zeros(T, np.float64)
    lib().hstu_oracle_norm_gate(T, F, 1 if norm == "layernorm" else 0, float(eps), _p(o), _p(u),
                                _p(y), _p(mean), _p(rstd), _p(_u8(rows)))
    return y, mean, rstd


def norm_gate_bwd(o, u, dy, norm="layernorm", eps=1e-5, rows=None):
    """(dx [T, F], du [T, F] or None)."""
    o = _f64(o).reshape(o.shape[0], -1)
    T, F = o.shape
    u, dy = _f64(u), _f64(dy).reshape(T, F)
    dx = np.zeros((T, F), np.float64)
    du = np.zeros((T, F), np.float64) if u is not None else None
    lib().hstu_oracle_norm_gate_bwd(T, F, 1 if norm == "layernorm" else 0, float(eps), _p(o), _p(u),
                                    _p(dy), _p(dx), _p(du), _p(_u8(rows)))
    return dx, du


# ------------------------------------------------------------------ dropout
# Dropout on y = Norm(o) * u, fused with the norm-gate (ai6s.net survey,
# section 2.1.3, "memory optimisation": dropout fused with its neighbouring
# operators).  The keep decision of element (t, f) of the [T, F] output comes
# from the counter-based generator Philox4x64-10 (Salmon, Moraes, Dror, Shaw,
# "Parallel random numbers: as easy as 1, 2, 3", SC 2011), so the backward
# regenerates the forward's mask from (seed, offset) alone:
#   e = t F + f;  (r0, r1, r2, r3) = Philox4x64-10(counter (e >> 3, offset, 0, 0), key (seed, 0))
#   w = 32-bit word (e & 7) of r0..r3, low half of each 64-bit word first
#   keep iff w >= floor(p 2^32);  kept elements are scaled by 1 / (1 - p)
# p is the descriptor's float32 value.

_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)
_LO32 = np.uint64(0xFFFFFFFF)
_PHILOX_M0 = np.uint64(0xD2E7470EE14C6C93)   # round multipliers
_PHILOX_M1 = np.uint64(0xCA5A826395121157)
_PHILOX_W0 = np.uint64(0x9E3779B97F4A7C15)   # key schedule (Weyl) increments
_PHILOX_W1 = np.uint64(0xBB67AE8584CAA73B)


def _mulhilo64(a, b):
    """(high, low) 64-bit halves of the 128-bit products a * b (uint64 arrays)."""
    s32 = np.uint64(32)
    al, ah = a & _LO32, a >> s32
    bl, bh = b & _LO32, b >> s32
    p0, p1, p2, p3 = al * bl, al * bh, ah * bl, ah * bh
    mid = (p0 >> s32) + (p1 & _LO32) + (p2 & _LO32)
    hi = p3 + (p1 >> s32) + (p2 >> s32) + (mid >> s32)
    return hi, a * b


def philox4x64_10(c0, c1, c2, c3, k0, k1):
    """Philox4x64 with 10 rounds on uint64 arrays (broadcast): returns the four
    output words.  A round multiplies c0 and c2 by the two round constants and
    crosses the halves with c1, c3 and the key; the key advances by the Weyl
    increments between rounds."""
    with np.errstate(over="ignore"):
        c = [np.asarray(x, np.uint64) for x in (c0, c1, c2, c3)]
        k = [np.asarray(k0, np.uint64), np.asarray(k1, np.uint64)]
        for r in range(10):
            if r > 0:
                k = [k[0] + _PHILOX_W0, k[1] + _PHILOX_W1]
            hi0, lo0 = _mulhilo64(_PHILOX_M0, c[0])
            hi1, lo1 = _mulhilo64(_PHILOX_M1, c[2])
            c = [hi1 ^ c[1] ^ k[0], lo1, hi0 ^ c[3] ^ k[1], lo0]
    return c


def dropout_threshold(p) -> int:
    """floor(p 2^32) for the float32 probability p (0 <= p < 1)."""
    p32 = float(np.float32(p))
    if not 0.0 <= p32 < 1.0:
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(np.floor(p32 * 4294967296.0))


def dropout_mask(T, F, p, seed, offset, rows=None):
    """(keep bool [T, F], scale) of the fused dropout; rows (bool [T]) limits
    the evaluation to those rows (the others are reported kept)."""
    p32 = float(np.float32(p))
    thr = dropout_threshold(p)
    keep = np.ones((T, F), bool)
    if p32 == 0.0 or T == 0:
        return keep, 1.0
    t_idx = np.arange(T, dtype=np.uint64) if rows is None else np.nonzero(np.asarray(rows, bool))[0].astype(np.uint64)
    e = t_idx[:, None] * np.uint64(F) + np.arange(F, dtype=np.uint64)[None, :]
    r = philox4x64_10(e >> np.uint64(3), np.uint64(offset), np.uint64(0), np.uint64(0),
                      np.uint64(seed), np.uint64(0))
    k = (e & np.uint64(7)).astype(np.int64)
    word64 = np.choose(k >> 1, r)
    w = (word64 >> (np.uint64(32) * (k & 1).astype(np.uint64))) & _LO32
    keep[t_idx.astype(np.int64)] = w >= np.uint64(thr)
    return keep, 1.0 / (1.0 - p32)


def apply_dropout(y, p, seed, offset, rows=None):
    """y [T, F] with the fused dropout applied (the identity when p == 0)."""
    y = _f64(y)
    keep, scale = dropout_mask(y.shape[0], y.shape[1], p, seed, offset, rows)
    return np.where(keep, y * scale, 0.0)


def attn_bwd(pb: Problem, dO, q_rows=None, kv_rows=None, want_rab=True):
    """dq, dk, dv [T, H, d] and d_rab_pos [H, P], d_rab_time [H, Tb] (None when
    the table is absent or rows are restricted)."""
    dO = _f64(dO).reshape(pb.T, pb.H, pb.dv)
    dq = np.zeros_like(pb.q)
    dk = np.zeros_like(pb.k)
    dv = np.zeros_like(pb.v)
    full = q_rows is None and kv_rows is None
    drp = np.zeros((pb.H, pb.P), np.float64) if (pb.rp is not None and full and want_rab) else None
    drt = (np.zeros((pb.H, pb.Tb), np.float64)
           if (pb.rt is not None and pb.ts is not None and full and want_rab) else None)
    rc = lib().hstu_oracle_attn_bwd(*pb._head(), _p(pb.q), _p(pb.k), _p(pb.v), _p(dO),
                                    _p(dq), _p(dk), _p(dv), _p(drp), _p(drt),
                                    _p(_u8(q_rows)), _p(_u8(kv_rows)))
    if rc != 0:
        raise ValueError("oracle: invalid jagged metadata")
    return dq, dk, dv, drp, drt


def forward(b, rows=None, dropout=None):
    """Whole forward of a synth.Batch: dict with o [T,H,dv], y [T,F], mean, rstd.
    dropout = (p, seed, offset) applies the fused dropout to y."""
    pb = Problem.from_batch(b)
    o = attn_fwd(pb, rows)
    y, mean, rstd = norm_gate(o, b.u, b.norm, b.eps, rows)
    if dropout is not None:
        y = apply_dropout(y, *dropout, rows=rows)
    return {"o": o, "y": y, "mean": mean, "rstd": rstd}


def backward(b, o=None, dropout=None):
    """Whole backward of a synth.Batch given its dy: dict with dq, dk, dv, du,
    d_rab_pos, d_rab_time (and the forward's o, y).  dropout = (p, seed,
    offset): dy is the gradient w.r.t. the dropped-out y, so it passes the
    forward's mask and scale before the norm-gate backward."""
    pb = Problem.from_batch(b)
    if o is None:
        o = attn_fwd(pb)
    dy = b.dy if dropout is None else apply_dropout(_f64(b.dy).reshape(pb.T, -1), *dropout)
    dO, du = norm_gate_bwd(o, b.u, dy, b.norm, b.eps)
    dq, dk, dv, drp, drt = attn_bwd(pb, dO)
    return {"o": o, "dO": dO.reshape(pb.T, pb.H, pb.dv), "dq": dq, "dk": dk, "dv": dv, "du": du,
            "d_rab_pos": drp, "d_rab_time": drt}


def tile_classes(offsets, num_targets, num_contexts, BM, BN):
    """Brute-force tile classes: structured array of (b, qb, kb, cls, allowed),
    cls 0 = skip, 1 = partial, 2 = full."""
    off = _i64(offsets)
    B = len(off) - 1
    n = int(lib().hstu_oracle_tile_count(B, _p(off), BM, BN))
    cols = [np.zeros(n, np.int32) for _ in range(4)]
    allowed = np.zeros(n, np.int64)
    lib().hstu_oracle_tile_classes(B, _p(off), _p(_i32(num_targets)), _p(_i32(num_contexts)), BM, BN,
                                   *[_p(c) for c in cols], _p(allowed))
    return {"b": cols[0], "qb": cols[1], "kb": cols[2], "cls": cols[3], "allowed": allowed}


def allowed_pairs(offsets, num_targets=None, num_contexts=None):
    off = _i64(offsets)
    out = np.zeros(len(off) - 1, np.int64)
    lib().hstu_oracle_allowed_pairs(len(off) - 1, _p(off), _p(_i32(num_targets)),
                                    _p(_i32(num_contexts)), _p(out))
    return out


# ------------------------------------------------------------- full layer

def _silu(x):
    return x / (1.0 + np.exp(-x))


def _silu_grad(x):
    s = 1.0 / (1.0 + np.exp(-x))
    return s * (1.0 + x * (1.0 - s))


def _split_uvqk(a, H, d):
    T = a.shape[0]
    D = H * d
    return (a[:, 0:D], a[:, D:2 * D].reshape(T, H, d), a[:, 2 * D:3 * D].reshape(T, H, d),
            a[:, 3 * D:4 * D].reshape(T, H, d))


def bf16_round(a):
    """Round float64 values to the nearest bfloat16 value (8 significant bits,
    ties to even), returned as float64.  Values stay in the normal range of
    the layer's activations; no overflow or subnormal handling."""
    a = np.asarray(a, np.float64)
    m, e = np.frexp(a)                      # a = m * 2**e, 0.5 <= |m| < 1
    return np.ldexp(np.round(m * 256.0) / 256.0, e)   # np.round: half to even


def layer_forward(b, rows=None, act_dtype=None, dropout=None):
    """Full HSTU layer forward in float64: dict with z1, u, v, q, k, o, y, out.

    act_dtype="bf16" rounds the values a BF16 layer stores once: V, Q and
    K = SiLU(X W1) are rounded to bfloat16 before the attention.  The gate U
    and Y (which such a layer carries at about 16 bits) are not rounded.
    rows (bool [T]) restricts o, y and out to those rows (the others are
    zero); z1 and the U/V/Q/K split are always complete.  dropout = (p, seed,
    offset) applies the fused dropout to y (before y W2)."""
    rnd = bf16_round if act_dtype == "bf16" else (lambda a: a)
    x, w1, w2 = _f64(b.x), _f64(b.w1), _f64(b.w2)
    z1 = x @ w1
    u, v, q, k = _split_uvqk(_silu(z1), b.H, b.d_v)
    v, q, k = rnd(v), rnd(q), rnd(k)
    pb = Problem(b.offsets, q, k, v, b.alpha, b.max_seq_len, b.num_targets, b.num_contexts,
                 b.timestamps, b.rab_pos, b.rab_time)
    o = attn_fwd(pb, rows)
    y, mean, rstd = norm_gate(o, u, "layernorm", b.eps, rows)
    if dropout is not None:
        y = apply_dropout(y, *dropout, rows=rows)
    y_op = y
    out = x + y_op @ w2
    if rows is not None:
        out[~np.asarray(rows, bool)] = 0.0
    return {"z1": z1, "u": u, "v": pb.v, "q": pb.q, "k": pb.k, "o": o, "y": y, "out": out,
            "mean": mean, "rstd": rstd, "pb": pb, "y_op": y_op, "act_dtype": act_dtype, "rows": rows,
            "dropout": dropout}


def layer_backward(b, fwd=None, act_dtype=None, rows=None, dropout=None):
    """Full HSTU layer backward given d(out) = b.dout: dict with dx, dw1, dw2
    and the attention intermediates dq, dk, dv, du, d_rab_pos, d_rab_time.

    act_dtype="bf16" also rounds d(out), an input, to bfloat16 as the
    operand of the two W2 products; dZ1 is not rounded (carried at about 16
    bits).

    rows (bool [T]) computes dx (and dq, dk, dv, du) only on those rows and
    leaves dw1, dw2 and the bias-table gradients out (None).  This is exact
    for every row whose key is attended only by queries inside rows (the
    candidate rows and the last history row of a sequence, when rows holds
    all the candidates of that sequence), because dO is formed on rows only."""
    f = layer_forward(b, rows=rows, act_dtype=act_dtype, dropout=dropout) if fwd is None else fwd
    rnd = bf16_round if act_dtype == "bf16" else (lambda a: a)
    x, w1, w2, dout = _f64(b.x), _f64(b.w1), _f64(b.w2), _f64(b.dout)
    dout_op = rnd(dout)
    dw2 = f["y_op"].T @ dout_op if rows is None else None
    dy = dout_op @ w2.T
    if f.get("dropout") is not None:
        dy = apply_dropout(dy, *f["dropout"], rows=rows)
    dO, du = norm_gate_bwd(f["o"], f["u"], dy, "layernorm", b.eps, rows)
    dq, dk, dv, drp, drt = attn_bwd(f["pb"], dO, q_rows=rows, kv_rows=rows)
    T = x.shape[0]
    sel = slice(None) if rows is None else np.asarray(rows, bool)
    da1 = np.concatenate([du, dv.reshape(T, -1), dq.reshape(T, -1), dk.reshape(T, -1)], axis=1)[sel]
    dz1 = da1 * _silu_grad(f["z1"][sel])
    dw1 = x.T @ dz1 if rows is None else None
    dx = np.zeros_like(dout)
    dx[sel] = dout[sel] + dz1 @ w1.T
    return {"dx": dx, "dw1": dw1, "dw2": dw2, "dq": dq, "dk": dk, "dv": dv, "du": du,
            "d_rab_pos": drp, "d_rab_time": drt, "dy": dy, "dO": dO}
