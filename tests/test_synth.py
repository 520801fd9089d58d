"""The seeded input recipe, checked against its definition on the CPU.

- History lengths: Zipf with exponent 1.2 on the finite support [1, 8192],
  drawn by inverse CDF (the heavy-tailed workload).
- Stochastic length (ai6s.net survey, section 2.1.3, sparse optimisation;
  the formula itself is lost there, so this is the stated reading): with
  L = floor(8192^0.8), a history of n > L tokens is cut to a uniform ordered
  subset of L tokens with probability 1 - 8192^1.6 / n^2; shorter ones stay.
- Timestamps: integer seconds; context tokens share the sequence's start,
  history times never decrease, and all candidates share one request time
  after the last history token.
Sampling checks use bounds of several standard errors, so a wrong exponent,
support or cut rule fails while seeded noise does not.
"""
import math

import numpy as np

from hstu_jagged_attention_02_gb300 import synth


def test_zipf_lengths_follow_the_finite_zipf_law():
    rng = np.random.default_rng(11)
    n = synth._zipf_lengths(rng, 400_000)
    assert n.min() >= 1 and n.max() <= 8192
    support = np.arange(1, 8193, dtype=np.float64)
    pmf = support ** -1.2 / np.sum(support ** -1.2)
    for lo, hi in ((1, 1), (2, 2), (3, 10), (11, 100), (101, 1000), (1001, 8192)):
        p = pmf[lo - 1:hi].sum()
        got = np.mean((n >= lo) & (n <= hi))
        se = math.sqrt(p * (1 - p) / n.size)
        assert abs(got - p) <= 5 * se + 1e-12, (lo, hi, got, p)


def test_stochastic_length_cut_rule():
    L = int(math.floor(8192 ** 0.8))
    assert L == 1351
    rng = np.random.default_rng(5)
    # never cut at or below L
    short = np.array([1, 100, L - 1, L] * 50, np.int64)
    kept, keeps = synth.stochastic_length(rng, short)
    assert np.array_equal(kept, short) and all(k is None for k in keeps)
    # above L: cut with probability 1 - 8192^1.6 / n^2, to exactly L sorted distinct indices
    for n in (1400, 2500, 8192):
        trials = 4000
        kept, keeps = synth.stochastic_length(rng, np.full(trials, n, np.int64))
        cut = kept == L
        p = 1.0 - 8192 ** 1.6 / n ** 2
        se = math.sqrt(p * (1 - p) / trials)
        assert abs(cut.mean() - p) <= 5 * se + 1e-12, (n, cut.mean(), p)
        assert np.all(kept[~cut] == n)
        for k in [x for x in keeps if x is not None][:50]:
            assert len(k) == L and np.all(np.diff(k) > 0) and k[0] >= 0 and k[-1] < n


def test_timestamp_structure():
    b = synth.make_batch([40, 0, 7], H=1, d_qk=32, d_v=32, num_contexts=[3, 2, 0], num_targets=[5, 4, 1],
                         seed=9)
    for s in range(b.B):
        a0, a1 = b.offsets[s], b.offsets[s + 1]
        c = 0 if b.num_contexts is None else int(b.num_contexts[s])
        m = int(b.num_targets[s])
        t = b.timestamps[a0:a1]
        ctx, hist, cand = t[:c], t[c:len(t) - m], t[len(t) - m:]
        if c:
            assert np.all(ctx == ctx[0])
            assert len(hist) == 0 or hist[0] >= ctx[0]
        assert np.all(np.diff(hist) >= 0)
        assert np.all(cand == cand[0])
        assert len(hist) == 0 or cand[0] >= hist[-1]


def test_heavy_tailed_batch_shape():
    b = synth.heavy_tailed(4)
    assert b.B == 64 and b.H == 4 and b.d_qk == b.d_v == 128
    assert np.all(b.num_targets == 32)
    hist = b.lengths - 32
    assert hist.min() >= 1 and hist.max() <= 8192
    assert b.max_seq_len == int(b.lengths.max())
    assert b.alpha == 1.0 / math.sqrt(128)
