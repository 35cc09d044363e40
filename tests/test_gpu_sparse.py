"""GPU parity of the page-sparse path against the oracle, through the C ABI.

- pkv_page_topk: selected page sets equal the oracle's, except where a differing
  page's oracle score lies within 1e-5 of the K-th score (ties in fp32 vs fp64);
- sparse forward/backward: given the oracle's selection, O and LSE within
  max-abs 1e-2 (bf16) / 1e-4 (fp32), dQ/dK/dV within relative Frobenius
  2e-2 / 1e-4;
- the whole sparse sweep with the GPU's own selection.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_numpy

pytestmark = pytest.mark.gpu
TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-4, 1e-4)}
TIE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _w(**kw):
    base = dict(N=2048, C=1024, P=128, Hq=4, Hkv=2, d=128, dtype="bf16", table="perm",
                keys="clustered", extra_pages=3, topk=(3, 1, 2))
    base.update(kw)
    return synth.workload("qwen7b_sparse_256k", **base)


def _inputs(w):
    n = w.n_chunks
    return ([synth.chunk_q(w, c) for c in range(n)], [synth.chunk_k(w, c) for c in range(n)],
            [synth.chunk_v(w, c) for c in range(n)], [synth.chunk_do(w, c) for c in range(n)])


def _check_selection(sel_gpu, q, q_start, k_logical, P, K, n_sink, n_local):
    """Compare against the oracle with the tie rule; returns the number of tie mismatches."""
    lists, padded = oracle.chunk_selection(q, q_start, k_logical, P, K, n_sink, n_local)
    qbar = oracle.query_page_means(q, P, k_logical.shape[1])
    rep = oracle.page_representatives(k_logical[: q_start + q.shape[0]], P)
    ties = 0
    for i in range(len(lists)):
        for h in range(len(lists[0])):
            got = [int(x) for x in sel_gpu[i, h] if x >= 0]
            assert got == sorted(set(got)), (i, h, got)
            want = lists[i][h]
            if got == want:
                continue
            qpg = q_start // P + i
            cand = np.arange(n_sink, qpg - n_local + 1)
            scores = rep[cand, h] @ qbar[i, h]
            kth = np.sort(scores)[::-1][min(K, len(cand)) - 1]
            for pg in set(got) ^ set(want):
                assert n_sink <= pg <= qpg - n_local, (i, h, pg)
                assert abs(rep[pg, h] @ qbar[i, h] - kth) <= TIE, (i, h, pg, got, want)
            ties += 1
    return ties


@pytest.mark.parametrize("dtype,P,d,K", [("bf16", 128, 128, 3), ("f32", 16, 64, 5),
                                         ("bf16", 128, 128, 64), ("bf16", 128, 128, 0),
                                         ("f32", 16, 64, 0)])
def test_page_topk_matches_oracle(dtype, P, d, K):
    """K = 0 keeps no scored page: every row is its sink and local pages."""
    w = _w(dtype=dtype, P=P, d=d, N=2048 if P == 128 else 512, C=1024 if P == 128 else 256,
           topk=(K, 1, 2))
    qs, ks, vs, _ = _inputs(w)
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        k_all = np.concatenate(ks)
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            n_qp = (e - s + w.P - 1) // w.P
            sel = torch.full((n_qp, w.Hkv, K + 3), 7, dtype=torch.int32, device="cuda")
            cnt = torch.zeros((n_qp, w.Hkv), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, 1, 2, sel, cnt)
            torch.cuda.synchronize()
            B.pkv_check(sw.pool)
            got = sel.cpu().numpy()
            _check_selection(got, qs[c], s, k_all, w.P, K, 1, 2)
            np.testing.assert_array_equal(cnt.cpu().numpy(), (got >= 0).sum(-1))
    finally:
        sw.close()


def test_page_topk_beyond_sixteen_thousand_candidates():
    """More candidate pages than a 16,384-entry sort buffer holds: page size 8
    and 16,456 pages, so the last chunk's query pages have ~16,450 candidates
    each (a 4M-token context at page 128 has 32,768 pages). Selection against
    the oracle with the tie rule; counts equal the listed entries."""
    P, C, n_pages = 8, 64, 16456
    w = _w(dtype="f32", P=P, d=64, N=n_pages * P, C=C, Hq=2, Hkv=1, table="identity",
           extra_pages=0, topk=(64, 1, 2))
    K, ns, nl = w.topk
    ks = [synth.chunk_k(w, c) for c in range(w.n_chunks)]
    k_all = np.concatenate(ks)
    c = w.n_chunks - 1
    s, e = w.chunk_range(c)
    q = synth.chunk_q(w, c)
    pool = B.pkv_pool_create(P, w.Hkv, w.Hq, w.d, B.PKV_F32, w.n_phys)
    try:
        seq = B.pkv_seq_create(pool)
        kt = torch.from_numpy(k_all).cuda()
        B.pkv_append(seq, kt, kt, w.N)
        n_qp = (e - s) // P
        sel = torch.full((n_qp, w.Hkv, K + ns + nl), 7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros((n_qp, w.Hkv), dtype=torch.int32, device="cuda")
        B.pkv_page_topk(seq, torch.from_numpy(q).cuda(), s, e - s, K, ns, nl, sel, cnt)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        got = sel.cpu().numpy()
        assert s // P - nl - ns + 1 > 16384
        _check_selection(got, q, s, k_all, P, K, ns, nl)
        np.testing.assert_array_equal(cnt.cpu().numpy(), (got >= 0).sum(-1))
    finally:
        B.pkv_pool_destroy(pool)


def _sparse_sweep(w, use_oracle_selection: bool, flags=0):
    K, ns, nl = w.topk if w.topk else (0,) + tuple(w.local)
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk,
                                      local=w.local)
    sw = ChunkSweep(w, flags=flags).load_inputs()
    try:
        sw.reset()
        sels = []
        k_all = np.concatenate(ks)
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            n_qp = (e - s + w.P - 1) // w.P
            if use_oracle_selection:
                sel = torch.from_numpy(ref["sel"][c]).cuda()
            elif w.local:
                sel = torch.full((n_qp, w.Hkv, ns + nl), 9, dtype=torch.int32, device="cuda")
                B.pkv_page_local(sw.seq, s, e - s, ns, nl, sel)
                torch.cuda.synchronize()
                np.testing.assert_array_equal(sel.cpu().numpy(), ref["sel"][c])
            else:
                sel = torch.empty((n_qp, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
                B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sel)
                torch.cuda.synchronize()
                assert _check_selection(sel.cpu().numpy(), qs[c], s, k_all, w.P, K, ns, nl) == 0
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sels[c])
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, sel=sels[c])
        B.pkv_check(sw.pool)
        g = sw.gather()
        tol_abs, tol_rel = TOL[w.dtype]
        o = np.concatenate([to_numpy(x) for x in sw.o])
        lse = np.concatenate([to_numpy(x) for x in sw.lse], axis=1)
        err = dict(
            o=float(np.abs(o - np.concatenate(ref["o"])).max()),
            lse=float(np.abs(lse - np.concatenate(ref["lse"], axis=1)).max()),
            dq=_rel(np.concatenate([to_numpy(x) for x in sw.dq]), np.concatenate(ref["dq"])),
            dk=_rel(to_numpy(g["dk"]), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)),
            dv=_rel(to_numpy(g["dv"]), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)),
        )
        assert err["o"] <= tol_abs and err["lse"] <= tol_abs, err
        assert max(err["dq"], err["dk"], err["dv"]) <= tol_rel, err
        return err
    finally:
        sw.close()


def test_sparse_attention_tensor_cores_oracle_selection():
    _sparse_sweep(_w(), use_oracle_selection=True)


def test_sparse_attention_tensor_cores_partial_chunk():
    _sparse_sweep(_w(N=1900, C=1024), use_oracle_selection=True)


def test_sparse_attention_cuda_cores_oracle_selection():
    _sparse_sweep(_w(dtype="f32", P=16, d=64, N=512, C=256, topk=(5, 1, 2)),
                  use_oracle_selection=True)


def test_sparse_attention_bf16_cuda_cores_flag():
    _sparse_sweep(_w(), use_oracle_selection=True, flags=B.PKV_FLAG_SIMT_ONLY)


def test_sparse_sweep_with_gpu_selection():
    _sparse_sweep(_w(N=3072, C=1024, topk=(4, 1, 2)), use_oracle_selection=False)


def test_sparse_with_all_pages_equals_dense_on_gpu():
    """K >= every candidate: the sparse kernels reproduce the dense ones."""
    w = _w(N=1024, C=512, keys="normal", topk=(64, 1, 2))
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.run()
        dense = ([to_numpy(x).copy() for x in sw.o], to_numpy(sw.gather()["dk"]).copy())
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            sel = torch.empty(((e - s) // w.P, w.Hkv, 67), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, 64, 1, 2, sel)
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, sel=sels[c])
        for a, b in zip(dense[0], [to_numpy(x) for x in sw.o]):
            np.testing.assert_array_equal(a, b)
        # The dense call may split a page's dK/dV over CTAs whose partial sums
        # meet by fp32 addition; the sparse call does not: the sums agree up to
        # the order of fp32 rounding.
        assert _rel(to_numpy(sw.gather()["dk"]), dense[1]) < 1e-5
    finally:
        sw.close()


# ---------------------------------------------------------------- local attention layers

@pytest.mark.parametrize("N,C,ns,nl", [(2048, 1024, 0, 2), (1900, 1024, 1, 2), (3000, 1024, 2, 5),
                                       (640, 256, 0, 1), (1024, 512, 0, 64)])
def test_page_local_lists_bit_exact(N, C, ns, nl):
    """pkv_page_local writes the oracle's local page lists and counts exactly
    (partial last query page, windows reaching page 0, windows wider than the
    sequence), and ignores the previous contents of the output."""
    w = _w(N=N, C=C, topk=None, local=(ns, nl))
    sw = ChunkSweep(w).load_inputs([])
    try:
        sw.reset()
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            k = torch.zeros((e - s, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
            B.pkv_append(sw.seq, k, k, e - s)
            n_qp = (e - s + w.P - 1) // w.P
            sel = torch.full((n_qp, w.Hkv, ns + nl), 5, dtype=torch.int32, device="cuda")
            cnt = torch.full((n_qp, w.Hkv), 77, dtype=torch.int32, device="cuda")
            B.pkv_page_local(sw.seq, s, e - s, ns, nl, sel, cnt)
            torch.cuda.synchronize()
            _, want = oracle.chunk_local_selection(s, e - s, w.Hkv, w.P, ns, nl)
            np.testing.assert_array_equal(sel.cpu().numpy(), want)
            np.testing.assert_array_equal(cnt.cpu().numpy(), (want >= 0).sum(-1))
        with pytest.raises(B.PkvError):
            B.pkv_page_local(sw.seq, 0, 128, 0, 0, sel)
        with pytest.raises(B.PkvError):
            B.pkv_page_local(sw.seq, 64, 128, 0, 2, sel)
        B.pkv_check(sw.pool)
    finally:
        sw.close()


@pytest.mark.parametrize("kw", [dict(local=(0, 2)), dict(local=(1, 2), N=1900),
                                dict(local=(0, 1), N=1536, C=512)])
def test_local_attention_tensor_cores(kw):
    base = dict(topk=None, keys="normal")
    base.update(kw)
    _sparse_sweep(_w(**base), use_oracle_selection=False)


@pytest.mark.parametrize("local", [None, (0, 2), (1, 3)])
def test_head_dim_64_sparse_and_local_tensor_cores(local):
    """Head dimension 64 through the tensor-core kernels with a selection: top-K
    from the GPU's own page selection, and local attention layers (the
    natively sparse models' page lists)."""
    if local is None:
        w = _w(d=64, N=2048, C=1024, Hq=8, Hkv=2)
    else:
        w = _w(d=64, N=2048, C=1024, Hq=8, Hkv=2, topk=None, keys="normal", local=local)
    _sparse_sweep(w, use_oracle_selection=False)


def test_local_attention_cuda_cores():
    _sparse_sweep(_w(dtype="f32", P=16, d=64, N=512, C=256, topk=None, local=(1, 3)),
                  use_oracle_selection=False)


@pytest.mark.parametrize("K", [1, 3])
def test_topk_error_against_dense_matches_oracle(K):
    """The sparse-vs-dense error the top-K budget study reports (relative
    Frobenius norm of O, dQ, dK, dV), measured on the GPU, equals the oracle's
    at a small size up to bf16 noise."""
    w = _w(N=2048, C=1024, topk=(K, 1, 2))
    qs, ks, vs, dos = _inputs(w)
    bt = synth.block_table(w)
    dense = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    sparse = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk)

    def flat(r):
        return (np.concatenate(r["o"]), np.concatenate(r["dq"]),
                oracle.logical_rows(r["dkpool"], bt, w.N, w.P),
                oracle.logical_rows(r["dvpool"], bt, w.N, w.P))

    e_ref = [_rel(a, b) for a, b in zip(flat(sparse), flat(dense))]
    sw = ChunkSweep(w).load_inputs()
    try:
        outs = []
        for sparse_run in (False, True):
            sw.reset()
            sels = []
            for c in range(w.n_chunks):
                s, e = w.chunk_range(c)
                B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
                sel = None
                if sparse_run:
                    sel = torch.empty(((e - s) // w.P, w.Hkv, K + 3), dtype=torch.int32, device="cuda")
                    B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, 1, 2, sel)
                sels.append(sel)
                B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
            for c in reversed(range(w.n_chunks)):
                sw.backward(c, sel=sels[c])
            g = sw.gather()
            outs.append((np.concatenate([to_numpy(x) for x in sw.o]),
                         np.concatenate([to_numpy(x) for x in sw.dq]),
                         to_numpy(g["dk"]), to_numpy(g["dv"])))
        B.pkv_check(sw.pool)
        e_gpu = [_rel(a, b) for a, b in zip(outs[1], outs[0])]
        assert min(e_ref) > 0.05, e_ref                 # the budget does cut attention
        for got, want in zip(e_gpu, e_ref):
            assert abs(got - want) <= 1e-2, (e_gpu, e_ref)
    finally:
        sw.close()


@pytest.mark.parametrize("key,n_q", [("qwen7b_local_256k", 9344), ("qwen7b_local_256k", 8192),
                                     ("gptoss_local_256k", 8192), ("qwen7b_dense_32k", 4096)])
def test_repeated_calls_are_bit_identical(key, n_q):
    """The forward, and the backward's dQ, have no atomics: calling them again
    on the same inputs must reproduce every bit. Local lists put 7 (GPT-OSS
    shape: 8) query heads in one forward CTA. 73 query pages is the case that
    once exposed a race there."""
    w = synth.workload(key, N=16384 + n_q, C=16384)
    s, e = w.chunk_range(1)
    n_qp = (e - s + w.P - 1) // w.P
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        for c in range(w.n_chunks):
            a, b = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], b - a)
        sel = None
        if w.local:
            sel = torch.empty((n_qp, w.Hkv, sum(w.local)), dtype=torch.int32, device="cuda")
            B.pkv_page_local(sw.seq, s, e - s, *w.local, sel)
        first = None
        for rep in range(12):
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[1], s, e - s, sw.o[1], sw.lse[1], sel)
            got = (sw.o[1].clone(), sw.lse[1].clone())
            if first is None:
                first = got
            else:
                assert torch.equal(got[0], first[0]) and torch.equal(got[1], first[1]), rep
        dq0 = None
        for rep in range(3):
            B.pkv_chunk_attn_bwd(sw.seq, sw.q[1], sw.o[1], sw.do[1], sw.lse[1], s, e - s, sw.dq[1], sel)
            if dq0 is None:
                dq0 = sw.dq[1].clone()
            else:
                assert torch.equal(sw.dq[1], dq0), rep
        B.pkv_check(sw.pool)
    finally:
        sw.close()
