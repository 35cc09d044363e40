"""Host-side arithmetic of bench.py: the algorithmic work it divides by time.

- dense causal pairs N(N+1)/2 equal a brute-force count of (i, j <= i);
- attended pairs of a page selection equal a brute-force count over the
  selected pages (full pages before the query page, causal inside it), per
  query head of each KV group;
- the oracle's own local and top-K lists give the counts the sparse workloads
  report;
- --context replaces N only by a multiple of the chunk and renames the workload.
"""
import argparse

import numpy as np
import pytest

import bench
import oracle


def test_dense_pairs_brute_force():
    for N in (1, 2, 7, 128, 1000):
        assert bench.pairs_dense(N) == sum(i + 1 for i in range(N))


def _brute_pairs(sel, q_start, P, g):
    n_qp, Hkv, _ = sel.shape
    total = 0
    for qp in range(n_qp):
        for h in range(Hkv):
            pages = set(int(p) for p in sel[qp, h] if p >= 0)
            for t in range(P):
                i = q_start + qp * P + t
                total += g * sum(1 for j in range(i + 1) if j // P in pages)
    return total


@pytest.mark.parametrize("ns,nl", [(0, 1), (1, 2), (2, 3)])
def test_sparse_pairs_of_local_lists_brute_force(ns, nl):
    P, Hkv, g, q_start, n_q = 8, 2, 3, 40, 32
    _, sel = oracle.chunk_local_selection(q_start, n_q, Hkv, P, ns, nl)
    assert bench.sparse_pairs(sel, P, g) == _brute_pairs(sel, q_start, P, g)


def test_sparse_pairs_of_topk_lists_brute_force():
    P, Hkv, Hq, d, q_start, n_q = 8, 2, 4, 16, 64, 32
    rng = np.random.default_rng(3)
    q = rng.standard_normal((n_q, Hq, d))
    k = rng.standard_normal((q_start + n_q, Hkv, d))
    _, sel = oracle.chunk_selection(q, q_start, k, P, 3, 1, 2)
    assert bench.sparse_pairs(sel, P, Hq // Hkv) == _brute_pairs(sel, q_start, P, Hq // Hkv)


def _args(**kw):
    ns = argparse.Namespace(workload="qwen7b_sparse_256k", context=0)
    for k, v in kw.items():
        setattr(ns, k, v)
    return ns


def test_context_override():
    w = bench.bench_workload(_args(context=65536))
    assert w.N == 65536 and w.n_chunks == 8 and "65536" in w.name
    assert bench.bench_workload(_args()).N == 262144
    with pytest.raises(SystemExit):
        bench.bench_workload(_args(context=65536 + 128))


def test_result_line_is_strict_json():
    import json
    out = bench.json_safe({"a": float("nan"), "b": [1.0, float("inf")], "c": {"d": 2.5}, "e": "x"})
    assert out == {"a": None, "b": [1.0, None], "c": {"d": 2.5}, "e": "x"}
    json.dumps(out, allow_nan=False)
