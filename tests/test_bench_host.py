"""Host arithmetic of bench.py, checked on the CPU against counts taken
element by element from the compound mask.

The metric counts useful FLOPs over allowed (query, key) pairs only: the
causal history/context pairs, the bidirectional context block and each
candidate's view of the history plus itself (ai6s.net survey, section 2.1.2,
ranking task; wmrh.cn RecSDK page, compound causal + context/target mask).
bench.py takes the count from a closed form per sequence; here it is the sum
of an explicit [n, n] visibility matrix built from whole-matrix pieces.
"""
import json
import types

import numpy as np
import pytest

import bench
from tests.bruteforce import dense_mask


def _batch(lengths, contexts, targets, H=3, d_qk=64, d_v=32):
    return types.SimpleNamespace(lengths=np.asarray(lengths, np.int64),
                                 num_contexts=None if contexts is None else np.asarray(contexts, np.int32),
                                 num_targets=None if targets is None else np.asarray(targets, np.int32),
                                 H=H, d_qk=d_qk, d_v=d_v)


def _dense_pairs(b, rows="all"):
    total = 0
    for i, n in enumerate(b.lengths):
        c = 0 if b.num_contexts is None else int(b.num_contexts[i])
        m = 0 if b.num_targets is None else int(b.num_targets[i])
        M = dense_mask(int(n), c, m)
        total += int(M[int(n) - m:].sum() if rows == "candidates" else M.sum())
    return total * b.H


CASES = [
    ([1, 2, 7, 50, 129], None, None),                       # causal only
    ([1, 5, 40, 64], [0, 2, 13, 64], None),                # context block, up to the whole sequence
    ([1, 9, 33, 300], None, [1, 4, 33, 32]),                # candidates, up to the whole sequence
    ([12, 70, 200, 5], [3, 0, 17, 1], [2, 8, 40, 4]),      # both
]


@pytest.mark.parametrize("lengths,contexts,targets", CASES)
def test_allowed_pairs_match_the_dense_mask(lengths, contexts, targets):
    b = _batch(lengths, contexts, targets)
    assert bench.allowed_pairs(b) == _dense_pairs(b)


def test_random_batches_allowed_pairs():
    r = np.random.default_rng(7)
    for _ in range(20):
        n = r.integers(1, 90, size=6)
        m = np.array([r.integers(0, k + 1) for k in n])
        c = np.array([r.integers(0, k - mm + 1) for k, mm in zip(n, m)])
        b = _batch(n, c, m, H=int(r.integers(1, 5)))
        assert bench.allowed_pairs(b) == _dense_pairs(b)


def test_useful_flops_count_each_pair_once_per_gemm():
    b = _batch([17, 80, 3], [2, 5, 0], [4, 10, 1], H=2, d_qk=64, d_v=32)
    fwd, bwd = bench.useful_flops(b)
    pairs = _dense_pairs(b)
    # forward: S = Q K^T (2 d_qk per pair) and O = A V (2 d_v);
    # backward: S recomputed, dQ, dK (3 x 2 d_qk) and dA, dV (2 x 2 d_v)
    assert fwd == pairs * (2 * 64 + 2 * 32)
    assert bwd == pairs * (3 * 2 * 64 + 2 * 2 * 32)


def test_delta_forward_counts_candidate_rows_only():
    b = _batch([300, 2100, 129], [0, 0, 0], [128, 128, 1], H=4, d_qk=128, d_v=128)
    f, bw, tot = bench.DeltaWorkload().flops(b)
    assert bw == 0 and tot == f
    assert f == _dense_pairs(b, rows="candidates") * 2 * (128 + 128)



def test_source_hash_ignores_comments_only():
    code = "int a = 1;  // one\n/* block\n comment */\nint b = a;\n\n"
    assert bench._code_only(code) == bench._code_only("int a = 1;\nint b = a;")
    assert bench._code_only(code) != bench._code_only("int a = 2;\nint b = a;")


def test_traffic_record_is_used_only_on_the_sources_it_was_taken_on(monkeypatch, tmp_path):
    # a DRAM-traffic record counts only while the kernel's code hashes to the
    # value stored with the capture; any other code gives no record (null)
    (tmp_path / "profiles").mkdir()
    rec = {"dram_bytes_per_token": 1.0, "sources_sha": "abc", "capture": "ncu ...", "capture_tokens": 10}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"w:bwd": rec}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda role: "abc" if role == "bwd" else "zzz")
    assert bench.traffic_record("w:bwd") == rec
    monkeypatch.setattr(bench, "kernel_sources_sha", lambda role: "def")
    assert bench.traffic_record("w:bwd") is None
    assert bench.traffic_record("w:fwd") is None
