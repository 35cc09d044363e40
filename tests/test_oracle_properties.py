"""Randomised pins of the oracle (hypothesis, CPU only): over random shapes --
chunk length, page size, GQA grouping, head dimension, permuted block tables,
partial last pages and chunks -- the paged, chunk-recurrent forward and
backward equal one-shot full-sequence attention (which is itself pinned to
library attention), and the paging helpers and local page lists equal their
plain definitions. Small sizes keep the whole module to seconds."""
import numpy as np
import pytest

hyp = pytest.importorskip("hypothesis")
st = pytest.importorskip("hypothesis.strategies")
from hypothesis import given, settings  # noqa: E402

import oracle as orc  # noqa: E402

SETTINGS = dict(max_examples=25, deadline=None, derandomize=True)


@st.composite
def _shapes(draw):
    P = draw(st.sampled_from([1, 2, 4, 8]))
    C = P * draw(st.integers(1, 4))
    n_chunks = draw(st.integers(1, 4))
    tail = draw(st.integers(0, C - 1)) if n_chunks > 1 else 0
    N = C * n_chunks - tail                         # last chunk may be partial
    Hkv = draw(st.integers(1, 2))
    g = draw(st.integers(1, 3))
    d = draw(st.sampled_from([2, 4, 8]))
    extra = draw(st.integers(0, 3))
    seed = draw(st.integers(0, 2 ** 16))
    return P, C, N, Hkv, g, d, extra, seed


@settings(**SETTINGS)
@given(_shapes())
def test_paged_chunk_recurrence_equals_one_shot(shape):
    P, C, N, Hkv, g, d, extra, seed = shape
    Hq = Hkv * g
    rng = np.random.default_rng(seed)
    q, do = rng.standard_normal((N, Hq, d)), rng.standard_normal((N, Hq, d))
    k, v = rng.standard_normal((N, Hkv, d)), rng.standard_normal((N, Hkv, d))
    n_pages = (N + P - 1) // P
    bt = rng.permutation(n_pages + extra)[:n_pages].astype(np.int32)
    cut = list(range(0, N, C)) + [N]
    split = lambda x: [x[a:b] for a, b in zip(cut[:-1], cut[1:])]
    res = orc.chunk_recurrent_step(split(q), split(k), split(v), split(do), bt, P, n_pages + extra)
    o_ref, lse_ref = orc.full_causal_attention(q, k, v)
    dq_ref, dk_ref, dv_ref = orc.attention_backward(q, k, v, o_ref, do, lse_ref, 0)
    np.testing.assert_allclose(np.concatenate(res["o"]), o_ref, atol=1e-10)
    np.testing.assert_allclose(np.concatenate(res["lse"], axis=1), lse_ref, atol=1e-10)
    np.testing.assert_allclose(np.concatenate(res["dq"]), dq_ref, atol=1e-9)
    np.testing.assert_allclose(orc.logical_rows(res["dkpool"], bt, N, P), dk_ref, atol=1e-9)
    np.testing.assert_allclose(orc.logical_rows(res["dvpool"], bt, N, P), dv_ref, atol=1e-9)
    # pages outside the table hold nothing
    unused = np.setdiff1d(np.arange(n_pages + extra), bt)
    assert not res["kpool"][unused].any() and not res["dkpool"][unused].any()


@settings(**SETTINGS)
@given(st.integers(0, 60), st.integers(0, 5), st.integers(1, 6))
def test_local_pages_equal_their_definition(qp, n_sink, n_local):
    want = sorted({p for p in range(qp + 1) if p < n_sink or p > qp - n_local})
    assert orc.local_pages(qp, n_sink, n_local) == want


@settings(**SETTINGS)
@given(st.integers(1, 8), st.integers(1, 40), st.integers(0, 4), st.integers(0, 2 ** 16))
def test_scatter_then_logical_rows_round_trip(P, N, extra, seed):
    rng = np.random.default_rng(seed)
    n_pages = (N + P - 1) // P
    bt = rng.permutation(n_pages + extra)[:n_pages].astype(np.int32)
    rows = rng.standard_normal((N, 2, 3))
    pool = np.zeros((n_pages + extra, 2, P, 3))
    orc.scatter_rows(pool, bt, 0, rows, P)
    np.testing.assert_array_equal(orc.logical_rows(pool, bt, N, P), rows)
    orc.scatter_rows(pool, bt, 0, rows, P, accumulate=True)
    np.testing.assert_array_equal(orc.logical_rows(pool, bt, N, P), 2 * rows)
