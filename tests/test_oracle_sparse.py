"""Pins for the oracle's page-sparse path (representatives, selection, sparse attention).

- K at least the number of candidates reproduces dense attention exactly;
- a planted page whose centre lines up with the page query is selected;
- selection equals a brute-force rank count at tiny sizes, ties to the lower page;
- representatives and page queries equal constructed means (closed forms);
- sparse attention equals library attention under the explicit page mask, and
  its backward matches finite differences.
"""
import math

import numpy as np
import pytest
import torch

import oracle as orc
from paged_kv_chunk_chunked_gb300 import synth


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_representative_closed_form():
    # keys = c + e and c - e in pairs: the mean of the page is exactly c
    P, Hkv, d = 8, 2, 5
    c = _rand((3, Hkv, d), 1)
    e = _rand((3, P // 2, Hkv, d), 2)
    k = np.concatenate([c[:, None] + e, c[:, None] - e], axis=1).reshape(3 * P, Hkv, d)
    rep = orc.page_representatives(k, P)
    np.testing.assert_allclose(rep, c, atol=1e-14)
    # partial last page: mean of the rows it holds
    rep2 = orc.page_representatives(k[: 2 * P + 2], P)
    np.testing.assert_allclose(rep2[2], (k[2 * P] + k[2 * P + 1]) / 2, atol=1e-14)


def test_query_page_mean_closed_form():
    # one query page, 2 KV heads with g = 3: the mean runs over tokens and the group's heads
    P, Hq, Hkv, d = 4, 6, 2, 3
    q = np.zeros((P, Hq, d))
    q[:, 0:3] = 1.0              # group 0: every entry 1
    q[0, 3:6] = 12.0             # group 1: one token of 4 holds 12 in all 3 heads
    qb = orc.query_page_means(q, P, Hkv)
    np.testing.assert_allclose(qb[0, 0], 1.0)
    np.testing.assert_allclose(qb[0, 1], 3.0)


def _brute_force_select(qbar, rep, qp, K, n_sink, n_local):
    keep = {p for p in range(qp + 1) if p < n_sink or p > qp - n_local}
    cand = [p for p in range(n_sink, qp - n_local + 1)]
    score = {p: float(np.dot(qbar, rep[p])) for p in cand}
    for p in cand:
        # rank = how many candidates come first: higher score, or equal score and lower index
        rank = sum(1 for r in cand if score[r] > score[p] or (score[r] == score[p] and r < p))
        if rank < K:
            keep.add(p)
    return sorted(keep)


@pytest.mark.parametrize("K,n_sink,n_local", [(3, 1, 2), (5, 2, 1), (1, 1, 2), (0, 1, 2)])
def test_selection_matches_brute_force(K, n_sink, n_local):
    d = 6
    rep = _rand((20, d), 3)
    rep[7] = rep[4]               # an exact score tie between pages 4 and 7
    for qp in range(20):
        qbar = _rand((d,), 100 + qp)
        assert orc.select_pages(qbar, rep, qp, K, n_sink, n_local) == \
            _brute_force_select(qbar, rep, qp, K, n_sink, n_local)


def test_selection_tie_goes_to_lower_page():
    d = 4
    rep = np.zeros((10, d))
    rep[3] = rep[6] = np.ones(d)
    sel = orc.select_pages(np.ones(d), rep, 9, 1, 1, 2)
    assert sel == [0, 3, 8, 9]


def test_selection_small_pages():
    rep = _rand((5, 4), 4)
    qb = _rand((4,), 5)
    assert orc.select_pages(qb, rep, 0, 64, 1, 2) == [0]
    assert orc.select_pages(qb, rep, 1, 64, 1, 2) == [0, 1]
    assert orc.select_pages(qb, rep, 2, 64, 1, 2) == [0, 1, 2]
    assert orc.select_pages(qb, rep, 3, 0, 1, 2) == [0, 2, 3]
    assert orc.select_pages(qb, rep, 4, 64, 1, 2) == [0, 1, 2, 3, 4]


def _sparse_w(**kw):
    base = dict(N=384, C=128, P=16, Hq=4, Hkv=2, d=16, dtype="f32", keys="clustered",
                table="perm", extra_pages=4)
    base.update(kw)
    return synth.workload("qwen7b_sparse_256k", **base)


def _inputs(w):
    n = w.n_chunks
    return ([synth.chunk_q(w, c) for c in range(n)], [synth.chunk_k(w, c) for c in range(n)],
            [synth.chunk_v(w, c) for c in range(n)], [synth.chunk_do(w, c) for c in range(n)])


def test_sparse_with_all_pages_equals_dense():
    w = _sparse_w()
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    dense = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    sparse = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys,
                                      topk=(w.n_pages, 1, 2))
    for key in ("o", "lse", "dq"):
        for a, b in zip(dense[key], sparse[key]):
            np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(dense["dkpool"], sparse["dkpool"])
    np.testing.assert_array_equal(dense["dvpool"], sparse["dvpool"])


def test_planted_page_is_selected():
    # give page 5 of KV head 1 a centre parallel to the page query, with a large norm
    w = _sparse_w(N=256, C=256)
    q = synth.chunk_q(w, 0)
    k = synth.chunk_k(w, 0)
    qbar = orc.query_page_means(q, w.P, w.Hkv)
    target_qp = 15
    u = qbar[target_qp, 1] / np.linalg.norm(qbar[target_qp, 1])
    k[5 * w.P:6 * w.P, 1] += 50.0 * u
    lists, _ = orc.chunk_selection(q, 0, k, w.P, K=1, n_sink=1, n_local=2)
    assert lists[target_qp][1] == [0, 5, 14, 15]


def test_sparse_forward_matches_library_with_page_mask():
    w = _sparse_w(N=128, C=128)
    q, k, v = synth.chunk_q(w, 0), synth.chunk_k(w, 0), synth.chunk_v(w, 0)
    lists, _ = orc.chunk_selection(q, 0, k, w.P, K=2, n_sink=1, n_local=2)
    allowed = orc.page_allowed_from_lists(lists, w.n_pages)
    o, _ = orc.attention_forward(q, k, v, 0, w.P, allowed)
    for h in range(w.Hq):
        kv = h // w.g
        mask = np.zeros((w.N, w.N), bool)
        for i in range(w.N):
            for j in range(i + 1):
                mask[i, j] = j // w.P in lists[i // w.P][kv]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.tensor(q[:, h], dtype=torch.float64)[None],
            torch.tensor(k[:, kv], dtype=torch.float64)[None],
            torch.tensor(v[:, kv], dtype=torch.float64)[None], attn_mask=torch.tensor(mask))
        np.testing.assert_allclose(o[:, h], ref[0].numpy(), atol=1e-12)


def test_sparse_backward_finite_differences():
    w = _sparse_w(N=64, C=64, P=8, Hq=2, Hkv=1, d=4)
    q, k, v, do = (synth.chunk_q(w, 0).astype(np.float64), synth.chunk_k(w, 0).astype(np.float64),
                   synth.chunk_v(w, 0).astype(np.float64), synth.chunk_do(w, 0).astype(np.float64))
    lists, _ = orc.chunk_selection(q, 0, k, w.P, K=2, n_sink=1, n_local=2)
    allowed = orc.page_allowed_from_lists(lists, w.n_pages)

    def loss(q_, k_, v_):
        o_, _ = orc.attention_forward(q_, k_, v_, 0, w.P, allowed)
        return float((o_ * do).sum())

    o, lse = orc.attention_forward(q, k, v, 0, w.P, allowed)
    grads = orc.attention_backward(q, k, v, o, do, lse, 0, w.P, allowed)
    rng = np.random.default_rng(1)
    for which, x in enumerate((q, k, v)):
        for _ in range(10):
            idx = tuple(int(rng.integers(s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1e-6
            xm[idx] -= 1e-6
            a = [q, k, v]; b = [q, k, v]
            a[which], b[which] = xp, xm
            fd = (loss(*a) - loss(*b)) / 2e-6
            assert abs(fd - grads[which][idx]) < 1e-7 * max(1, abs(fd))


def test_padded_selection_layout():
    w = _sparse_w(N=128, C=64)
    q = synth.chunk_q(w, 1)
    k = np.concatenate([synth.chunk_k(w, 0), synth.chunk_k(w, 1)])
    lists, padded = orc.chunk_selection(q, 64, k, w.P, K=2, n_sink=1, n_local=2)
    assert padded.shape == (4, w.Hkv, 5)
    for i in range(4):
        for h in range(w.Hkv):
            n = len(lists[i][h])
            assert list(padded[i, h, :n]) == lists[i][h]
            assert (padded[i, h, n:] == -1).all()
            assert lists[i][h][-1] == 4 + i    # own page is always last


# ---------------------------------------------------------------- local attention layers

@pytest.mark.parametrize("n_sink,n_local", [(0, 1), (0, 2), (1, 2), (3, 4), (2, 1)])
def test_local_pages_counts_and_order(n_sink, n_local):
    """Closed forms: |list| = min(qp + 1, n_sink + n_local); the query page is
    last; a window reaching page 0 gives every page; K = 0 top-K gives the same
    list (nothing to score)."""
    rep, qb = np.zeros((40, 4)), np.ones(4)
    for qp in range(40):
        got = orc.local_pages(qp, n_sink, n_local)
        assert len(got) == min(qp + 1, n_sink + n_local)
        assert got == sorted(set(got)) and got[-1] == qp
        if qp < n_sink + n_local:
            assert got == list(range(qp + 1))
        else:
            assert got[:n_sink] == list(range(n_sink))
            assert got[n_sink:] == list(range(qp - n_local + 1, qp + 1))
        assert got == orc.select_pages(qb, rep, qp, 0, n_sink, n_local)


def test_local_one_page_equals_blockwise_library_attention():
    """n_local = 1, no sink: every query attends causally inside its own page only,
    i.e. independent causal attention per P-token block (library attention, fp64),
    forward and backward (autograd), through the paged chunk recurrence."""
    w = _sparse_w(N=96, C=32, P=16, Hq=4, Hkv=2, d=8, keys="normal")
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    res = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, local=(0, 1))
    q, k, v, do = (np.concatenate(x) for x in (qs, ks, vs, dos))
    o = np.concatenate(res["o"])
    dq = np.concatenate(res["dq"])
    dk = orc.logical_rows(res["dkpool"], bt, w.N, w.P)
    for b in range(w.N // w.P):
        sl = slice(b * w.P, (b + 1) * w.P)
        tq = torch.tensor(q[sl], dtype=torch.float64).permute(1, 0, 2).requires_grad_()
        tk = torch.tensor(k[sl], dtype=torch.float64).repeat_interleave(w.g, 1).permute(1, 0, 2).requires_grad_()
        tv = torch.tensor(v[sl], dtype=torch.float64).repeat_interleave(w.g, 1).permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
        (ref * torch.tensor(do[sl], dtype=torch.float64).permute(1, 0, 2)).sum().backward()
        np.testing.assert_allclose(o[sl], ref.permute(1, 0, 2).detach().numpy(), atol=1e-12)
        np.testing.assert_allclose(dq[sl], tq.grad.permute(1, 0, 2).numpy(), atol=1e-10)
        dk_ref = tk.grad.permute(1, 0, 2).numpy().reshape(w.P, w.Hkv, w.g, w.d).sum(2)
        np.testing.assert_allclose(dk[sl], dk_ref, atol=1e-10)


def test_local_window_covering_everything_equals_dense():
    w = _sparse_w()
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    dense = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    local = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, local=(0, w.n_pages))
    for key in ("o", "lse", "dq"):
        for a, b in zip(dense[key], local[key]):
            np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(dense["dkpool"], local["dkpool"])


def test_local_padded_layout():
    lists, padded = orc.chunk_local_selection(64, 40, 3, 16, 1, 2)
    assert padded.shape == (3, 3, 3)
    assert lists[0][2] == [0, 3, 4] and lists[2][0] == [0, 5, 6]
    assert (padded[:, 0] == padded[:, 2]).all()
    assert (padded[0, 0] == [0, 3, 4]).all()
    with pytest.raises(ValueError):
        orc.chunk_local_selection(8, 16, 1, 16, 0, 1)
