"""Host side of the delta forward (KV-cached candidate scoring, wmrh.cn RecSDK
page: variable length with KV cache): splitting a jagged batch into the cached
part of each sequence and its candidates.  Properties checked on random
batches: the two row sets partition the tokens in order, the offsets count
each sequence's part, and every row sits on the right side of its
sequence's candidate boundary."""
import types

import numpy as np

from hstu_jagged_attention_02_gb300.delta import split_rows


def _batch(lengths, targets):
    lengths = np.asarray(lengths, np.int64)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    return types.SimpleNamespace(B=len(lengths), offsets=off,
                                 num_targets=None if targets is None else np.asarray(targets, np.int32))


def _check(b):
    cache_rows, cand_rows, cache_off, cand_off = split_rows(b)
    T = int(b.offsets[-1])
    m = np.zeros(b.B, np.int64) if b.num_targets is None else b.num_targets.astype(np.int64)
    assert np.array_equal(np.sort(np.concatenate([cache_rows, cand_rows])), np.arange(T))
    assert np.all(np.diff(cache_rows) > 0) and np.all(np.diff(cand_rows) > 0)   # token order kept
    assert np.array_equal(np.diff(cand_off), m)
    assert np.array_equal(np.diff(cache_off), np.diff(b.offsets) - m)
    for s in range(b.B):
        h_end = b.offsets[s + 1] - m[s]
        mine_cache = cache_rows[cache_off[s]:cache_off[s + 1]]
        mine_cand = cand_rows[cand_off[s]:cand_off[s + 1]]
        assert np.all((mine_cache >= b.offsets[s]) & (mine_cache < h_end))
        assert np.all((mine_cand >= h_end) & (mine_cand < b.offsets[s + 1]))


def test_split_rows_edge_cases():
    _check(_batch([5, 1, 7], [2, 1, 0]))     # a sequence of candidates only, one with none
    _check(_batch([4, 9], None))             # no candidates: everything is cache
    _check(_batch([0, 3, 0], [0, 3, 0]))     # empty sequences


def test_split_rows_random_batches():
    r = np.random.default_rng(3)
    for _ in range(50):
        n = r.integers(0, 40, size=int(r.integers(1, 9)))
        m = np.array([r.integers(0, k + 1) for k in n])
        _check(_batch(n, m))
