"""Pins of the FP64 oracle to things other than itself.

* the KeyedJaggedTensor worked example (lengths -> offsets convention),
* the bucket functions against their mathematical definitions,
* an independent padded-dense brute force on tiny inputs, every mask mode,
* the 1-token and 2-token closed forms,
* invariants: packing, candidate permutation, candidate isolation, masked
  pairs contribute exactly zero,
* LayerNorm against torch's library routine,
* the backward against central finite differences and torch autograd,
* allowed-pair counts and tile classes against the closed-form pair count.
"""
import json
import math
import os

import numpy as np
import pytest

from hstu_jagged_attention_02_gb300 import synth
from oracle import oracle as O
from tests import bruteforce as BF

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


# ----------------------------------------------------------- jagged layout

def test_kjt_worked_example_offsets():
    g = json.load(open(os.path.join(GOLDEN, "kjt_example.json")))
    off = synth.offsets_from_lengths(g["lengths"])
    assert off.tolist() == [0, 2, 5, 6, 8]
    vals = g["values"]
    segs = [vals[off[i]:off[i + 1]] for i in range(len(g["lengths"]))]
    # keys own consecutive groups of segments (2 per key here)
    per_key = len(segs) // len(g["keys"])
    got = {key: segs[i * per_key:(i + 1) * per_key] for i, key in enumerate(g["keys"])}
    assert got == g["printed"]


# ------------------------------------------------------------------ buckets

@pytest.mark.parametrize("delta", [0, 1, 2, 3, 4, 5, 7, 8, 600, 1023, 1024, 1025,
                                   2**31 - 1, 2**31, 2**40 + 3, 2**62, 2**63 - 1])
def test_time_bucket_is_binary_length(delta):
    # floor(log2 d) + 1 == number of binary digits; 0 for d == 0; clamp at 63
    want = min(63, delta.bit_length())
    if delta > 0:
        assert want == min(63, math.floor(math.log2(delta)) + 1) or delta >= 2**53
    assert O.time_bucket(10**12 + delta if delta < 2**62 else delta, 10**12 if delta < 2**62 else 0) == want
    # symmetric in its arguments
    assert O.time_bucket(0, delta) == want


def test_time_bucket_random():
    r = np.random.default_rng(5)
    for d in r.integers(0, 2**45, size=200):
        assert O.time_bucket(int(d) + 7, 7) == min(63, int(d).bit_length())


def test_pos_bucket_special_cases():
    h_end = 300
    assert O.pos_bucket(5, 5, h_end) == 0
    assert O.pos_bucket(10, 3, h_end) == 7 and O.pos_bucket(3, 10, h_end) == 7
    assert O.pos_bucket(200, 0, h_end) == 127          # clamped
    # all candidates sit at position h_end
    assert O.pos_bucket(h_end + 5, h_end + 9, h_end) == 0
    assert O.pos_bucket(h_end + 5, h_end - 4, h_end) == 4


# -------------------------------------------------------------- brute force

def _random_case(lengths, H=2, d=8, dv=None, nc=None, nt=None, time=True, rab=True, seed=0,
                 u=True):
    r = np.random.default_rng(seed)
    dv = dv or d
    lengths = np.asarray(lengths)
    off = synth.offsets_from_lengths(lengths)
    T = int(off[-1])
    ts = None
    if time:
        ts = np.concatenate([np.sort(r.integers(0, 5000, size=n)) + 1_700_000_000 for n in lengths]
                            ).astype(np.int64) if T else np.zeros(0, np.int64)
    case = dict(
        offsets=off, q=r.standard_normal((T, H, d)), k=r.standard_normal((T, H, d)),
        v=r.standard_normal((T, H, dv)), alpha=1 / math.sqrt(d), N=float(max(lengths.max(), 1)),
        nt=None if nt is None else np.asarray(nt, np.int32),
        nc=None if nc is None else np.asarray(nc, np.int32), ts=ts,
        rp=r.normal(0, 0.3, (H, 128)) if rab else None,
        rt=r.normal(0, 0.3, (H, 64)) if (rab and time) else None,
        u=r.standard_normal((T, H * dv)) if u else None)
    return case


def _oracle_fwd(c, norm="layernorm"):
    pb = O.Problem(c["offsets"], c["q"], c["k"], c["v"], c["alpha"], c["N"], c["nt"], c["nc"],
                   c["ts"], c["rp"], c["rt"])
    o = O.attn_fwd(pb)
    y, _, _ = O.norm_gate(o, c["u"], norm)
    return o, y


MASK_CASES = [
    dict(lengths=[1, 2, 5, 17, 33], nc=None, nt=None),
    dict(lengths=[6, 9, 40], nc=None, nt=[2, 9, 5]),           # a sequence of only candidates
    dict(lengths=[6, 9, 40], nc=[3, 9, 8], nt=None),           # a sequence of only context
    dict(lengths=[12, 30, 64], nc=[2, 4, 8], nt=[3, 7, 16]),
    dict(lengths=[1, 3], nc=[1, 0], nt=[0, 3]),
]


@pytest.mark.parametrize("mc", MASK_CASES)
@pytest.mark.parametrize("time,rab", [(True, True), (False, True), (False, False)])
def test_oracle_matches_dense_bruteforce(mc, time, rab):
    c = _random_case(mc["lengths"], nc=mc["nc"], nt=mc["nt"], time=time, rab=rab, seed=len(mc["lengths"]))
    o, y = _oracle_fwd(c)
    ob, yb = BF.forward(c["offsets"], c["q"], c["k"], c["v"], c["alpha"], c["N"], c["nt"], c["nc"],
                        c["ts"], c["rp"], c["rt"], c["u"])
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(y, yb, rtol=1e-10, atol=1e-11)


def test_large_time_gaps_hit_the_clamp():
    c = _random_case([20], time=True, seed=3)
    c["ts"] = np.sort(RNG.integers(0, 2**62, size=20)).astype(np.int64)
    o, _ = _oracle_fwd(c)
    ob, _ = BF.forward(c["offsets"], c["q"], c["k"], c["v"], c["alpha"], c["N"], None, None,
                       c["ts"], c["rp"], c["rt"], c["u"])
    np.testing.assert_allclose(o, ob, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------- closed forms

def _silu(z):
    return z / (1 + math.exp(-z))


def test_one_token_closed_form():
    r = np.random.default_rng(7)
    H, d = 3, 16
    q, k, v = (r.standard_normal((1, H, d)) for _ in range(3))
    rp, rt = r.normal(0, 0.1, (H, 128)), r.normal(0, 0.1, (H, 64))
    ts = np.array([1_700_000_123], np.int64)
    N = 7.0
    pb = O.Problem([0, 1], q, k, v, 0.25, N, None, None, ts, rp, rt)
    o = O.attn_fwd(pb)
    for h in range(H):
        z = 0.25 * float(q[0, h] @ k[0, h]) + rp[h, 0] + rt[h, 0]
        np.testing.assert_allclose(o[0, h], _silu(z) / N * v[0, h], rtol=1e-14)


def test_two_token_causal_closed_form():
    r = np.random.default_rng(8)
    H, d = 2, 8
    q, k, v = (r.standard_normal((2, H, d)) for _ in range(3))
    rp, rt = r.normal(0, 0.1, (H, 128)), r.normal(0, 0.1, (H, 64))
    ts = np.array([100, 107], np.int64)      # gap 7 -> time bucket floor(log2 7)+1 = 3
    N, a = 2.0, 0.5
    o = O.attn_fwd(O.Problem([0, 2], q, k, v, a, N, None, None, ts, rp, rt))
    for h in range(H):
        z00 = a * q[0, h] @ k[0, h] + rp[h, 0] + rt[h, 0]
        z10 = a * q[1, h] @ k[0, h] + rp[h, 1] + rt[h, 3]
        z11 = a * q[1, h] @ k[1, h] + rp[h, 0] + rt[h, 0]
        np.testing.assert_allclose(o[0, h], _silu(z00) * v[0, h] / N, rtol=1e-13)
        np.testing.assert_allclose(o[1, h], (_silu(z10) * v[0, h] + _silu(z11) * v[1, h]) / N,
                                   rtol=1e-13)


# ---------------------------------------------------------------- invariants

def test_packing_equals_per_sequence_runs():
    c = _random_case([5, 23, 11, 40], nc=[1, 2, 0, 4], nt=[2, 5, 3, 8], seed=11)
    o, y = _oracle_fwd(c)
    off = c["offsets"]
    for b in range(4):
        s, e = off[b], off[b + 1]
        pb = O.Problem([0, e - s], c["q"][s:e], c["k"][s:e], c["v"][s:e], c["alpha"], c["N"],
                       c["nt"][b:b + 1], c["nc"][b:b + 1], c["ts"][s:e], c["rp"], c["rt"])
        assert np.array_equal(O.attn_fwd(pb), o[s:e])


def test_candidate_permutation_equivariance():
    n, m = 30, 8
    c = _random_case([n], nt=[m], seed=12)
    # give each candidate its own timestamp so the permutation moves real data
    c["ts"][n - m:] = c["ts"][n - m - 1] + RNG.integers(1, 1000, size=m)
    o, _ = _oracle_fwd(c)
    perm = np.arange(n)
    perm[n - m:] = n - m + RNG.permutation(m)
    c2 = dict(c)
    for key in ("q", "k", "v", "ts"):
        c2[key] = c[key][perm]
    c2["u"] = c["u"][perm]
    o2, _ = _oracle_fwd(c2)
    assert np.array_equal(o2, o[perm])


def test_one_candidate_does_not_touch_others():
    n, m = 25, 6
    c = _random_case([n], nt=[m], seed=13)
    o, _ = _oracle_fwd(c)
    c2 = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in c.items()}
    j = n - m + 2
    c2["q"][j] += 5.0
    c2["k"][j] -= 3.0
    c2["v"][j] *= -7.0
    o2, _ = _oracle_fwd(c2)
    others = [i for i in range(n) if i != j]
    assert np.array_equal(o2[others], o[others])
    assert not np.array_equal(o2[j], o[j])


def test_masked_pairs_contribute_exact_zero():
    n, cx, m = 20, 3, 4
    c = _random_case([n], nc=[cx], nt=[m], seed=14)
    o, _ = _oracle_fwd(c)
    # row 8 (history) cannot see 9..n-1; row 1 (context) cannot see 3..n-1
    for row, hidden in ((8, range(9, n)), (1, range(3, n))):
        c2 = {key: (val.copy() if isinstance(val, np.ndarray) else val) for key, val in c.items()}
        for j in hidden:
            c2["k"][j] = 1e30
            c2["v"][j] = 1e30
        o2, _ = _oracle_fwd(c2)
        assert np.array_equal(o2[row], o[row])


# ---------------------------------------------------------------- LayerNorm

def test_layernorm_against_torch():
    torch = pytest.importorskip("torch")
    r = np.random.default_rng(15)
    o = r.standard_normal((37, 4, 16)) * 3 + 1
    u = r.standard_normal((37, 64))
    y, mean, rstd = O.norm_gate(o, u, "layernorm", 1e-5)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(o.reshape(37, 64)), (64,), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy() * u, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(mean, o.reshape(37, 64).mean(1), rtol=1e-12)
    y0, _, _ = O.norm_gate(o, u, "none")
    np.testing.assert_array_equal(y0, o.reshape(37, 64) * u)


# ----------------------------------------------------------------- backward

def _loss_and_grads(c, dy, norm="layernorm"):
    pb = O.Problem(c["offsets"], c["q"], c["k"], c["v"], c["alpha"], c["N"], c["nt"], c["nc"],
                   c["ts"], c["rp"], c["rt"])
    o = O.attn_fwd(pb)
    y, _, _ = O.norm_gate(o, c["u"], norm)
    dO, du = O.norm_gate_bwd(o, c["u"], dy, norm)
    dq, dk, dv, drp, drt = O.attn_bwd(pb, dO)
    return float((y * dy).sum()), dict(q=dq, k=dk, v=dv, u=du, rp=drp, rt=drt)


@pytest.mark.parametrize("norm", ["layernorm", "none"])
def test_backward_central_differences(norm):
    c = _random_case([4, 9, 13], nc=[1, 2, 3], nt=[1, 3, 4], H=2, d=4, seed=21)
    r = np.random.default_rng(22)
    dy = r.standard_normal(c["u"].shape)
    _, g = _loss_and_grads(c, dy, norm)
    h = 1e-6
    for key in ("q", "k", "v", "u", "rp", "rt"):
        for trial in range(2):
            delta = r.standard_normal(c[key].shape)
            cp = dict(c); cp[key] = c[key] + h * delta
            cm = dict(c); cm[key] = c[key] - h * delta
            fd = (_loss_and_grads(cp, dy, norm)[0] - _loss_and_grads(cm, dy, norm)[0]) / (2 * h)
            an = float((g[key] * delta).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (key, fd, an)


def test_backward_against_torch_autograd():
    torch = pytest.importorskip("torch")
    c = _random_case([3, 11, 20], nc=[0, 2, 5], nt=[1, 3, 6], H=2, d=8, seed=23)
    r = np.random.default_rng(24)
    dy = r.standard_normal(c["u"].shape)
    _, g = _loss_and_grads(c, dy)
    tt = {key: torch.tensor(c[key], dtype=torch.float64, requires_grad=True)
          for key in ("q", "k", "v", "u", "rp", "rt")}
    _, y = BF.torch_forward(c["offsets"], tt["q"], tt["k"], tt["v"], c["alpha"], c["N"], c["nt"],
                            c["nc"], c["ts"], tt["rp"], tt["rt"], tt["u"])
    (y * torch.from_numpy(dy)).sum().backward()
    for key in tt:
        np.testing.assert_allclose(g[key], tt[key].grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=key)


def test_restricted_rows_match_full_backward():
    c = _random_case([7, 19, 33], nc=[1, 2, 3], nt=[2, 3, 4], H=2, d=8, seed=25)
    r = np.random.default_rng(26)
    dO = r.standard_normal(c["v"].shape)
    pb = O.Problem(c["offsets"], c["q"], c["k"], c["v"], c["alpha"], c["N"], c["nt"], c["nc"],
                   c["ts"], c["rp"], c["rt"])
    full = O.attn_bwd(pb, dO)
    rows = np.zeros(pb.T, bool); rows[[0, 8, 30, 58]] = True
    part = O.attn_bwd(pb, dO, q_rows=rows, kv_rows=rows)
    for a, b in zip(full[:3], part[:3]):
        np.testing.assert_array_equal(a[rows], b[rows])


# --------------------------------------------------------- pair / tile counts

def _closed_form_pairs(n, c, m):
    h_end = n - m
    return h_end * (h_end + 1) // 2 + c * (c - 1) // 2 + m * (h_end + 1)


def test_allowed_pair_count_closed_form():
    r = np.random.default_rng(27)
    lengths = r.integers(1, 90, size=30)
    nc = np.array([r.integers(0, n + 1) for n in lengths])
    nt = np.array([r.integers(0, n - c + 1) for n, c in zip(lengths, nc)])
    off = synth.offsets_from_lengths(lengths)
    got = O.allowed_pairs(off, nt, nc)
    want = [_closed_form_pairs(int(n), int(c), int(m)) for n, c, m in zip(lengths, nc, nt)]
    assert got.tolist() == want
    # and the dense mask of the brute force agrees
    for n, c, m in zip(lengths[:8], nc[:8], nt[:8]):
        assert BF.dense_mask(int(n), int(c), int(m)).sum() == _closed_form_pairs(int(n), int(c), int(m))


@pytest.mark.parametrize("BM,BN", [(128, 128), (64, 64), (16, 32)])
def test_tile_classes_partition_the_pairs(BM, BN):
    r = np.random.default_rng(28)
    lengths = r.integers(1, 400, size=12)
    nc = np.array([r.integers(0, min(n, 40) + 1) for n in lengths])
    nt = np.array([r.integers(0, min(n - c, 70) + 1) for n, c in zip(lengths, nc)])
    off = synth.offsets_from_lengths(lengths)
    tc = O.tile_classes(off, nt, nc, BM, BN)
    for b, (n, c, m) in enumerate(zip(lengths, nc, nt)):
        sel = tc["b"] == b
        assert tc["allowed"][sel].sum() == _closed_form_pairs(int(n), int(c), int(m))
        assert np.all((tc["cls"][sel] == 0) == (tc["allowed"][sel] == 0))
        assert np.all((tc["cls"][sel] == 2) == (tc["allowed"][sel] == BM * BN))
        assert sel.sum() == math.ceil(n / BM) * math.ceil(n / BN)


# ------------------------------------------------------------- full layer

def _tiny_layer(seed=30):
    r = np.random.default_rng(seed)
    H, d = 2, 4
    D = H * d
    lengths = np.array([5, 9, 14])
    off = synth.offsets_from_lengths(lengths + 3)
    T = int(off[-1])
    ts = np.concatenate([np.sort(r.integers(0, 4000, size=n + 3)) for n in lengths]).astype(np.int64)
    empty = np.zeros((T, H, 0))
    return synth.Batch(name="layer", seed=seed, dtype="fp32", B=3, H=H, d_qk=d, d_v=d,
                       lengths=lengths + 3, offsets=off, num_targets=np.full(3, 3, np.int32),
                       num_contexts=None, timestamps=ts, q=empty, k=empty, v=empty, u=None, dy=None,
                       rab_pos=r.normal(0, 0.2, (H, 128)), rab_time=r.normal(0, 0.2, (H, 64)),
                       alpha=0.5, max_seq_len=17, x=r.standard_normal((T, D)),
                       w1=r.normal(0, 0.3, (D, 4 * D)), w2=r.normal(0, 0.3, (D, D)),
                       dout=r.standard_normal((T, D)))


@pytest.mark.parametrize("dropout", [None, (0.3, 12, 4)])
def test_layer_backward_central_differences(dropout):
    b = _tiny_layer()
    g = O.layer_backward(b, dropout=dropout)
    r = np.random.default_rng(31)
    h = 1e-6

    def loss(bb):
        return float((O.layer_forward(bb, dropout=dropout)["out"] * bb.dout).sum())

    import copy
    for key, gk in (("x", "dx"), ("w1", "dw1"), ("w2", "dw2"), ("rab_pos", "d_rab_pos"),
                    ("rab_time", "d_rab_time")):
        delta = r.standard_normal(getattr(b, key).shape)
        bp = copy.copy(b); setattr(bp, key, getattr(b, key) + h * delta)
        bm = copy.copy(b); setattr(bm, key, getattr(b, key) - h * delta)
        fd = (loss(bp) - loss(bm)) / (2 * h)
        an = float((g[gk] * delta).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (key, fd, an)


def test_layer_split_order_and_residual():
    # with W2 = 0 the layer is the identity; the U slice is the first D columns of SiLU(X W1)
    b = _tiny_layer(32)
    b.w2 = np.zeros_like(b.w2)
    f = O.layer_forward(b)
    np.testing.assert_array_equal(f["out"], b.x)
    D = b.H * b.d_v
    a1 = f["z1"] / (1 + np.exp(-f["z1"]))
    np.testing.assert_array_equal(f["u"], a1[:, :D])
    np.testing.assert_array_equal(f["k"].reshape(-1, D), a1[:, 3 * D:])


def test_bf16_round_matches_torch_conversion():
    torch = pytest.importorskip("torch")
    # float32 -> bfloat16 rounding to nearest even as torch performs it, including exact ties
    r = np.random.default_rng(33)
    a = (r.standard_normal(4000) * np.exp(r.uniform(-20, 20, 4000))).astype(np.float32)
    bits = a.view(np.uint32)
    ties = ((bits[:1000] & np.uint32(0xFFFF0000)) | np.uint32(0x8000)).view(np.float32)
    a = np.concatenate([a, ties, np.float32([1.0, -2.5, 3.0e-3])])
    want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(a.astype(np.float64)), want)


def _layer_sample_rows(b):
    # every candidate row and the last history row of each sequence: the keys of
    # these rows are attended only by queries of the same set
    rows = np.zeros(b.T, bool)
    for i in range(b.B):
        s, e = int(b.offsets[i]), int(b.offsets[i + 1])
        rows[e - int(b.num_targets[i]) - 1:e] = True
    return rows


def test_layer_backward_on_rows_equals_full_backward():
    b = _tiny_layer(34)
    rows = _layer_sample_rows(b)
    full = O.layer_backward(b)
    part = O.layer_backward(b, rows=rows)
    assert part["dw1"] is None and part["dw2"] is None and part["d_rab_pos"] is None
    np.testing.assert_allclose(part["dx"][rows], full["dx"][rows], rtol=1e-12, atol=1e-12)
    assert np.all(part["dx"][~rows] == 0)
    f = O.layer_forward(b, rows=rows)
    np.testing.assert_allclose(f["out"][rows], O.layer_forward(b)["out"][rows], rtol=1e-12, atol=1e-12)


def test_layer_bf16_storage_stays_within_rounding_error():
    # rounding the stored activations to bfloat16 (8 significant bits: relative
    # error <= 2^-8 each) moves every output by a small multiple of 2^-8 of its scale
    b = _tiny_layer(35)
    exact_f, round_f = O.layer_forward(b), O.layer_forward(b, act_dtype="bf16")
    exact_g, round_g = O.layer_backward(b, exact_f), O.layer_backward(b, round_f, act_dtype="bf16")
    np.testing.assert_array_equal(round_f["u"], exact_f["u"])       # the gate is not rounded
    assert np.all(np.abs(round_f["q"] - exact_f["q"]) <= 2.0 ** -8 * np.abs(exact_f["q"]))
    assert not np.array_equal(round_f["q"], exact_f["q"])
    for got, want in ((round_f["out"], exact_f["out"]), (round_g["dx"], exact_g["dx"]),
                      (round_g["dw1"], exact_g["dw1"]), (round_g["dw2"], exact_g["dw2"])):
        scale = math.sqrt(float(np.mean(want * want)))
        assert np.max(np.abs(got - want)) <= 16 * 2.0 ** -8 * scale
