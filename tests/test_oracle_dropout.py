"""Pins of the oracle's fused dropout (y = dropout(Norm(o) * u)).

* the Philox4x64-10 core against numpy's own implementation of the
  generator (numpy.random.Philox, an independent library routine): same
  128-bit products, round structure and key schedule, word for word;
* the keep decision: the keep rate is 1 - p and neighbouring elements of
  one generator block are independent (binomial bounds); p = 0 keeps all;
* the definition's invariants: the mask of element (t, f) depends only on
  (seed, offset, t F + f), so any [T, F] shape with the same flat layout and
  any row subset give the same bits; another seed or offset gives another
  mask;
* E[dropout(y)] = y (inverted scaling), and the backward of the composition
  against central finite differences.
"""
import math

import numpy as np
import pytest

from oracle import oracle as O


def _numpy_philox_block(c0, c1, c2, c3, k0, k1):
    # numpy's generator advances word 0 of its counter before each block
    bg = np.random.Philox(counter=np.array([c0 - 1, c1, c2, c3], np.uint64), key=np.array([k0, k1], np.uint64))
    return [int(x) for x in bg.random_raw(4)]


@pytest.mark.parametrize("ctr,key", [
    ((1, 0, 0, 0), (0, 0)),
    ((5, 7, 0, 0), (123, 0)),
    ((2**40 + 17, 3, 0, 0), (2**63 + 12345, 0)),
    ((2**64 - 1, 2**64 - 1, 2**64 - 1, 2**64 - 1), (2**64 - 1, 2**64 - 1)),
    ((0x243F6A8885A308D3, 0x13198A2E03707344, 0xA4093822299F31D0, 0x082EFA98EC4E6C89),
     (0x452821E638D01377, 0xBE5466CF34E90C6C)),
])
def test_philox_matches_numpy(ctr, key):
    want = _numpy_philox_block(*ctr, *key)
    got = [int(x) for x in O.philox4x64_10(*[np.uint64(c) for c in ctr], np.uint64(key[0]), np.uint64(key[1]))]
    assert got == want


def test_philox_vectorised_equals_scalar_blocks():
    r = np.random.default_rng(3)
    c0 = r.integers(1, 2**63, size=64, dtype=np.uint64)
    c1 = r.integers(0, 2**63, size=64, dtype=np.uint64)
    out = O.philox4x64_10(c0, c1, np.uint64(0), np.uint64(0), np.uint64(99), np.uint64(0))
    for i in range(0, 64, 9):
        assert [int(w[i]) for w in out] == _numpy_philox_block(int(c0[i]), int(c1[i]), 0, 0, 99, 0)


def _binomial_ok(k, n, q, sigmas=6.0):
    return abs(k - n * q) <= sigmas * math.sqrt(n * q * (1 - q)) + 1


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_keep_rate(p):
    keep, scale = O.dropout_mask(300, 512, p, seed=7, offset=11)
    assert _binomial_ok(int(keep.sum()), keep.size, 1 - float(np.float32(p)))
    assert scale == pytest.approx(1.0 / (1.0 - float(np.float32(p))), rel=1e-15)


def test_neighbours_in_a_block_are_independent():
    keep, _ = O.dropout_mask(256, 512, 0.5, seed=1, offset=0)
    flat = keep.reshape(-1)
    for lag in (1, 2, 4, 7, 8):
        both = int((flat[:-lag] & flat[lag:]).sum())
        assert _binomial_ok(both, flat.size - lag, 0.25), lag


def test_p_zero_keeps_everything():
    keep, scale = O.dropout_mask(10, 64, 0.0, seed=5, offset=5)
    assert keep.all() and scale == 1.0
    y = np.random.default_rng(0).standard_normal((10, 64))
    assert np.array_equal(O.apply_dropout(y, 0.0, 5, 5), y)


def test_threshold_is_floor_of_p_times_2_32():
    assert O.dropout_threshold(0.0) == 0
    assert O.dropout_threshold(0.5) == 2**31
    assert O.dropout_threshold(0.25) == 2**30
    p32 = float(np.float32(0.1))
    assert O.dropout_threshold(0.1) == math.floor(p32 * 2**32)
    with pytest.raises(ValueError):
        O.dropout_threshold(1.0)


def test_mask_depends_only_on_the_flat_element_index():
    a, _ = O.dropout_mask(6, 40, 0.3, seed=2, offset=9)
    b, _ = O.dropout_mask(3, 80, 0.3, seed=2, offset=9)
    c, _ = O.dropout_mask(240, 1, 0.3, seed=2, offset=9)
    assert np.array_equal(a.reshape(-1), b.reshape(-1))
    assert np.array_equal(a.reshape(-1), c.reshape(-1))
    rows = np.zeros(6, bool)
    rows[[1, 4]] = True
    d, _ = O.dropout_mask(6, 40, 0.3, seed=2, offset=9, rows=rows)
    assert np.array_equal(d[rows], a[rows]) and d[~rows].all()


def test_other_seed_or_offset_gives_another_mask():
    a, _ = O.dropout_mask(64, 128, 0.5, seed=2, offset=9)
    for seed, offset in ((3, 9), (2, 10)):
        b, _ = O.dropout_mask(64, 128, 0.5, seed=seed, offset=offset)
        agree = int((a == b).sum())
        assert _binomial_ok(agree, a.size, 0.5)


def test_inverted_scaling_keeps_the_mean():
    y = np.full((512, 512), 3.0)
    got = O.apply_dropout(y, 0.3, seed=4, offset=0)
    q = 1 - float(np.float32(0.3))
    sd = 3.0 / q * math.sqrt(q * (1 - q)) / math.sqrt(y.size)
    assert abs(got.mean() - 3.0) <= 6 * sd
    assert set(np.unique(got)) <= {0.0, 3.0 / q}


@pytest.mark.parametrize("norm", ["layernorm", "none"])
def test_norm_gate_dropout_backward_central_differences(norm):
    r = np.random.default_rng(31)
    T, F = 7, 24
    o, u, dy = r.standard_normal((T, F)), r.standard_normal((T, F)), r.standard_normal((T, F))
    drop = (0.4, 77, 5)

    def loss(o_, u_):
        y, _, _ = O.norm_gate(o_, u_, norm)
        return float((O.apply_dropout(y, *drop) * dy).sum())

    do, du = O.norm_gate_bwd(o, u, O.apply_dropout(dy, *drop), norm)
    h = 1e-6
    for which in ("o", "u"):
        for trial in range(3):
            delta = r.standard_normal((T, F))
            if which == "o":
                fd = (loss(o + h * delta, u) - loss(o - h * delta, u)) / (2 * h)
                an = float((do * delta).sum())
            else:
                fd = (loss(o, u + h * delta) - loss(o, u - h * delta)) / (2 * h)
                an = float((du * delta).sum())
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (which, fd, an)
