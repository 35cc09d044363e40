"""The parallel oracle helper (tests/oracle_pool.py) against the plain oracle.

The full-size GPU tests take their expected values from OraclePool, which
splits the oracle's work over processes and uses two restatements: a page's
dK/dV from a backward over that page's keys alone, shifted, and a page-sparse
row as dense causal attention over its selected pages laid end to end. Here
both must reproduce the oracle's own chunk-recurrent sweep
(oracle.chunk_recurrent_step) on small workloads: dense with a permuted block
table and grouped heads, and page-sparse with top-K selection.
"""
import numpy as np
import pytest

import oracle
from paged_kv_chunk_chunked_gb300 import synth

from oracle_pool import OraclePool


@pytest.fixture(scope="module")
def pool():
    with OraclePool(processes=4) as p:
        yield p


def _inputs(w):
    n = w.n_chunks
    return ([synth.chunk_q(w, c) for c in range(n)], [synth.chunk_k(w, c) for c in range(n)],
            [synth.chunk_v(w, c) for c in range(n)], [synth.chunk_do(w, c) for c in range(n)])


def test_dense_full_and_page_grads_equal_the_chunk_recurrent_oracle(pool):
    w = synth.workload("tiny_dense_f32", Hq=4, Hkv=2, table="perm", extra_pages=3)
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    got = pool.dense_full(w, block=24)
    for c in range(w.n_chunks):
        np.testing.assert_allclose(got["o"][c], ref["o"][c], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["lse"][c], ref["lse"][c], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["dq"][c], ref["dq"][c], rtol=0, atol=1e-12)
    dk = oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)
    dv = oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)
    np.testing.assert_allclose(got["dk"], dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dv"], dv, rtol=0, atol=1e-12)
    # every chunk: the final rows of a page of chunk 0, two pages on a chunk
    # boundary (the chunk is 4 pages) and the last page
    pages = [1, 7, 8, 15]
    pg = pool.dense_page_grads(w, pages, block=40)
    for p in pages:
        rows = slice(p * w.P, (p + 1) * w.P)
        np.testing.assert_allclose(pg[p][0], dk[rows], rtol=0, atol=1e-12)
        np.testing.assert_allclose(pg[p][1], dv[rows], rtol=0, atol=1e-12)
    # one chunk's contribution alone: the oracle's backward of that chunk
    c = 2
    s, e = w.chunk_range(c)
    K, V = np.concatenate(ks)[:e], np.concatenate(vs)[:e]
    o, lse = oracle.attention_forward(qs[c], K, V, s)
    _, dkc, dvc = oracle.attention_backward(qs[c], K, V, o, dos[c], lse, s)
    pg = pool.dense_page_grads(w, [1, 8, 11], chunks=[c], kvs=[1])
    for p in (1, 8, 11):
        rows = slice(p * w.P, (p + 1) * w.P)
        np.testing.assert_allclose(pg[p][0][:, 1], dkc[rows, 1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(pg[p][1][:, 1], dvc[rows, 1], rtol=0, atol=1e-12)
        assert not pg[p][0][:, 0].any()                 # KV head 0 not asked for


def test_sparse_full_and_page_grads_equal_the_chunk_recurrent_oracle(pool):
    w = synth.workload("qwen7b_sparse_256k", N=512, C=128, P=16, Hq=4, Hkv=2, d=64,
                       dtype="f32", extra_pages=2, topk=(3, 1, 2))
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk)
    lists = {c: {(i, kv): [int(x) for x in ref["sel"][c][i, kv] if x >= 0]
                 for i in range(ref["sel"][c].shape[0]) for kv in range(w.Hkv)}
             for c in range(w.n_chunks)}
    K, V = np.concatenate(ks), np.concatenate(vs)
    page_kv = lambda p: (K[p * w.P:(p + 1) * w.P], V[p * w.P:(p + 1) * w.P])
    got = pool.sparse_full(w, lists, page_kv)
    for c in range(w.n_chunks):
        np.testing.assert_allclose(got["o"][c], ref["o"][c], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["lse"][c], ref["lse"][c], rtol=0, atol=1e-12)
        np.testing.assert_allclose(got["dq"][c], ref["dq"][c], rtol=0, atol=1e-12)
    dk = oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)
    dv = oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)
    np.testing.assert_allclose(got["dk"], dk, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["dv"], dv, rtol=0, atol=1e-12)
    want = {0: [0, 5, 17], 1: [3, 20, 31]}
    pg, n_tasks = pool.sparse_page_grads(w, lists, want, page_kv)
    assert n_tasks > 0
    for kv, ps in want.items():
        for p in ps:
            rows = slice(p * w.P, (p + 1) * w.P)
            np.testing.assert_allclose(pg[(p, kv)][0], dk[rows, kv], rtol=0, atol=1e-12)
            np.testing.assert_allclose(pg[(p, kv)][1], dv[rows, kv], rtol=0, atol=1e-12)
