"""GPU tests of the pinned-host page streamer (PINNED_HOST pools), through the C ABI.

The K/V pages and their fp32 gradient pages live in mapped pinned host memory;
per chunk the selected (or all) pages are staged into HBM slots on a side
stream, attention runs on the slots on the main stream, and the gradients are
written back. Results must match the oracle within the parity tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.sweep import to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _offloaded_sweep(w, n_slots, sparse: bool):
    K, ns, nl = w.topk
    n = w.n_chunks
    qs = [synth.chunk_q(w, c) for c in range(n)]
    ks = [synth.chunk_k(w, c) for c in range(n)]
    vs = [synth.chunk_v(w, c) for c in range(n)]
    dos = [synth.chunk_do(w, c) for c in range(n)]
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys,
                                      topk=w.topk if sparse else None)
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=n_slots)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        dq_, o_, lse_, sels = [], [], [], []
        dev = lambda x: to_device(x, "bf16")
        q = [dev(x) for x in qs]; k = [dev(x) for x in ks]; v = [dev(x) for x in vs]
        do = [dev(x) for x in dos]
        for c in range(n):
            s, e = w.chunk_range(c)
            B.pkv_append(seq, k[c], v[c], e - s, main)
            o_.append(torch.empty_like(q[c]))
            lse_.append(torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda"))
            dq_.append(torch.empty_like(q[c]))
            sel = None
            if sparse:
                sel = torch.empty(((e - s + w.P - 1) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32,
                                  device="cuda")
                B.pkv_page_topk(seq, q[c], s, e - s, K, ns, nl, sel, None, main)
            sels.append(sel)
            B.pkv_prefetch(seq, sel, 0 if sel is None else sel.numel(), B.PKV_STAGE_KV, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_fwd(seq, q[c], s, e - s, o_[c], lse_[c], sel, main)
        for c in reversed(range(n)):
            s, e = w.chunk_range(c)
            sel = sels[c]
            B.pkv_prefetch(seq, sel, 0 if sel is None else sel.numel(),
                           B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_bwd(seq, q[c], o_[c], do[c], lse_[c], s, e - s, dq_[c], sel, main)
            B.pkv_writeback_grads(seq, side)
        B.pkv_wait(seq, main, 5_000_000)            # bounded host wait, then GPU-side wait
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        kk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
        B.pkv_gather(seq, kk, None, dk, dv, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        np.testing.assert_array_equal(to_numpy(kk), np.concatenate(ks))
        o = np.concatenate([to_numpy(x) for x in o_])
        lse = np.concatenate([to_numpy(x) for x in lse_], axis=1)
        err = dict(
            o=float(np.abs(o - np.concatenate(ref["o"])).max()),
            lse=float(np.abs(lse - np.concatenate(ref["lse"], axis=1)).max()),
            dq=_rel(np.concatenate([to_numpy(x) for x in dq_]), np.concatenate(ref["dq"])),
            dk=_rel(to_numpy(dk), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)),
            dv=_rel(to_numpy(dv), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)),
        )
        assert err["o"] <= 1e-2 and err["lse"] <= 1e-2, err
        assert max(err["dq"], err["dk"], err["dv"]) <= 2e-2, err
        return err
    finally:
        B.pkv_pool_destroy(pool)


def _w(**kw):
    base = dict(N=3072, C=1024, P=128, Hq=4, Hkv=2, d=128, dtype="bf16", table="perm",
                keys="clustered", extra_pages=5, topk=(3, 1, 2), offload=True)
    base.update(kw)
    return synth.workload("qwen7b_sparse_1m_offload", **base)


def test_offloaded_sparse_sweep_matches_oracle():
    # 24 pages; a chunk stages only the union of its selections (at most 24 pages)
    _offloaded_sweep(_w(), n_slots=24, sparse=True)


def test_offloaded_dense_sweep_matches_oracle():
    w = _w(N=2048, keys="normal")
    _offloaded_sweep(w, n_slots=w.n_pages, sparse=False)


def test_staging_more_pages_than_slots_is_reported():
    w = _w(N=1024, C=1024)
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=3)
    try:
        seq = B.pkv_seq_create(pool)
        kv = to_device(synth.chunk_k(w, 0), "bf16")
        B.pkv_append(seq, kv, kv, w.N)
        B.pkv_prefetch(seq, None, 0, B.PKV_STAGE_KV, None)   # 8 pages into 3 slots
        with pytest.raises(B.PkvError) as e:
            B.pkv_check(pool)
        assert e.value.status == B.PKV_ERR_DEVICE_FAULT and "slots" in str(e.value)
        B.pkv_check(pool)                                   # the error word was cleared
        with pytest.raises(B.PkvError) as e:
            B.pkv_prefetch(seq, None, 0, 8, None)           # unknown staging flag
        assert e.value.status == B.PKV_ERR_INVALID
    finally:
        B.pkv_pool_destroy(pool)


def test_offload_calls_reject_device_pools():
    pool = B.pkv_pool_create(128, 1, 2, 128, B.PKV_BF16, 4)
    try:
        seq = B.pkv_seq_create(pool)
        for f in (lambda: B.pkv_prefetch(seq), lambda: B.pkv_writeback_grads(seq),
                  lambda: B.pkv_wait(seq)):
            with pytest.raises(B.PkvError) as e:
                f()
            assert e.value.status == B.PKV_ERR_INVALID
    finally:
        B.pkv_pool_destroy(pool)


def test_grad_accumulate_into_pinned_host_pages_then_prefetch():
    """pkv_grad_accumulate on a PINNED_HOST pool adds into the host gradient
    pages (bit-exact against the oracle's scatter-add), and a gradient prefetch
    issued on a side stream afterwards stages the sums (ordered by the
    sequence's event)."""
    w = synth.workload("qwen7b_sparse_256k", N=1024, C=512, Hq=4, Hkv=2, extra_pages=2,
                       topk=(2, 1, 2))
    bt = synth.block_table(w)
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            k = to_device(synth.chunk_k(w, c), "bf16")
            B.pkv_append(seq, k, k, e - s)
        ref = {t: np.zeros((w.n_phys, w.Hkv, w.P, w.d), np.float32) for t in ("dk", "dv")}
        for i, (r0, n) in enumerate([(0, w.N), (100, 300), (w.N - 1, 1)]):
            x = synth.draw_normal(w.seed, "misc", 200 + i, (n, w.Hkv, w.d))
            y = synth.draw_normal(w.seed, "misc", 300 + i, (n, w.Hkv, w.d))
            oracle.scatter_rows(ref["dk"], bt, r0, x, w.P, accumulate=True)
            oracle.scatter_rows(ref["dv"], bt, r0, y, w.P, accumulate=True)
            B.pkv_grad_accumulate(seq, r0, n, torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda())
        B.pkv_prefetch(seq, None, 0, B.PKV_STAGE_GRADS, side)
        B.pkv_wait(seq, torch.cuda.current_stream(), 0)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_numpy(dk), oracle.logical_rows(ref["dk"], bt, w.N, w.P))
        np.testing.assert_array_equal(to_numpy(dv), oracle.logical_rows(ref["dv"], bt, w.N, w.P))
        # the staged slots hold the same sums: write them back unchanged
        B.pkv_writeback_grads(seq, side)
        B.pkv_wait(seq, torch.cuda.current_stream(), 0)
        B.pkv_gather(seq, None, None, dk, dv, None)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_numpy(dk), oracle.logical_rows(ref["dk"], bt, w.N, w.P))
    finally:
        B.pkv_pool_destroy(pool)


def test_projections_overlapping_the_page_transfer_match_oracle():
    """The sparse-offload overlap ("Out of the Memory Barrier", gist.science/de
    §2.C: with sparse attention the transfer overlaps the key/value projections
    that follow): chunk c's selected pages stream in on a side stream while the
    main stream runs the next chunk's K/V projection, a bf16 cuBLAS GEMM
    x_{c+1} [wk | wv], whose output becomes chunk c+1's keys and values; in the
    backward, the chunk's query projection is recomputed (chunk-recurrent
    recomputation, gist.science/de §2.A) while its K/V and gradient pages
    stream in, and the recomputed queries feed the backward. Against the
    oracle on the same projections computed in fp64 and rounded to bf16 (the
    GEMM's own rounding may differ in the last bf16 place on a few elements).
    Selections equal the oracle's; O and LSE within 1e-2, dQ, dK, dV within
    2e-2 relative."""
    w = _w(N=3072, C=1024, keys="normal")
    K, ns, nl = w.topk
    hidden = 512
    n = w.n_chunks
    wts = synth.block_weights(w, hidden)
    xs = [synth.block_x(w, c, hidden) for c in range(n)]
    proj = lambda x, m: synth.round_bf16((x.astype(np.float64) @ m.astype(np.float64)).astype(np.float32))
    qs = [proj(x, wts["wq"]).reshape(-1, w.Hq, w.d) for x in xs]
    ks = [proj(x, wts["wk"]).reshape(-1, w.Hkv, w.d) for x in xs]
    vs = [proj(x, wts["wv"]).reshape(-1, w.Hkv, w.d) for x in xs]
    dos = [synth.chunk_do(w, c) for c in range(n)]
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk)

    dev = lambda x: to_device(x, "bf16")
    X = [dev(x) for x in xs]
    Wq, Wkv = dev(wts["wq"]), dev(np.concatenate([wts["wk"], wts["wv"]], axis=1))
    do = [dev(x) for x in dos]
    kvd = w.Hkv * w.d
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        o, lse, dq, sels = [], [], [], []
        kv_next = torch.matmul(X[0], Wkv)                      # chunk 0's K/V
        for c in range(n):
            s, e = w.chunk_range(c)
            kv = kv_next
            k_c = kv[:, :kvd].contiguous().view(e - s, w.Hkv, w.d)
            v_c = kv[:, kvd:].contiguous().view(e - s, w.Hkv, w.d)
            B.pkv_append(seq, k_c, v_c, e - s, main)
            q_c = torch.matmul(X[c], Wq).view(e - s, w.Hq, w.d)
            sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(seq, q_c, s, e - s, K, ns, nl, sel, None, main)
            sels.append(sel)
            B.pkv_prefetch(seq, sel, sel.numel(), B.PKV_STAGE_KV, side)
            if c + 1 < n:
                kv_next = torch.matmul(X[c + 1], Wkv)          # overlaps the transfer
            B.pkv_wait(seq, main, 0)
            o.append(torch.empty_like(q_c))
            lse.append(torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda"))
            dq.append(torch.empty_like(q_c))
            B.pkv_chunk_attn_fwd(seq, q_c, s, e - s, o[c], lse[c], sel, main)
        for c in reversed(range(n)):
            s, e = w.chunk_range(c)
            B.pkv_prefetch(seq, sels[c], sels[c].numel(), B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
            q_c = torch.matmul(X[c], Wq).view(e - s, w.Hq, w.d)    # recomputed, overlapping
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_bwd(seq, q_c, o[c], do[c], lse[c], s, e - s, dq[c], sels[c], main)
            B.pkv_writeback_grads(seq, side)
        B.pkv_wait(seq, main, 10_000_000)
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        for c in range(n):
            np.testing.assert_array_equal(sels[c].cpu().numpy(), ref["sel"][c])
            assert np.abs(to_numpy(o[c]) - ref["o"][c]).max() <= 1e-2, c
            assert np.abs(to_numpy(lse[c]) - ref["lse"][c]).max() <= 1e-2, c
            assert _rel(to_numpy(dq[c]), ref["dq"][c]) <= 2e-2, c
        assert _rel(to_numpy(dk), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)) <= 2e-2
        assert _rel(to_numpy(dv), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)) <= 2e-2
    finally:
        B.pkv_pool_destroy(pool)


def _unions(sels):
    return [np.unique(s[s >= 0]) for s in sels]


def test_slot_cache_with_evictions_matches_oracle_and_moves_fewer_pages():
    """The slot cache: fewer slots than pages, so pages (with dirty gradients
    in the backward) are evicted between chunks; no per-chunk write-back, one
    release at the end. Gradients, outputs and selections equal the oracle's;
    the K/V page-heads moved are fewer than staging every chunk's selection
    afresh, and every page staged with gradients was written back."""
    w = _w(N=4096, C=1024)
    K, ns, nl = w.topk
    n = w.n_chunks
    qs = [synth.chunk_q(w, c) for c in range(n)]
    ks = [synth.chunk_k(w, c) for c in range(n)]
    vs = [synth.chunk_v(w, c) for c in range(n)]
    dos = [synth.chunk_do(w, c) for c in range(n)]
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk)
    unions = _unions(ref["sel"])
    n_slots = max(len(u) for u in unions)
    assert n_slots < w.n_pages                       # evictions must happen
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=n_slots)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        dev = lambda x: to_device(x, "bf16")
        q = [dev(x) for x in qs]
        do = [dev(x) for x in dos]
        o, lse, dq, sels = [], [], [], []
        for c in range(n):
            s, e = w.chunk_range(c)
            B.pkv_append(seq, dev(ks[c]), dev(vs[c]), e - s, main)
            sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(seq, q[c], s, e - s, K, ns, nl, sel, None, main)
            sels.append(sel)
            o.append(torch.empty_like(q[c]))
            lse.append(torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda"))
            dq.append(torch.empty_like(q[c]))
            B.pkv_prefetch(seq, sel, sel.numel(), B.PKV_STAGE_KV, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_fwd(seq, q[c], s, e - s, o[c], lse[c], sel, main)
        for c in reversed(range(n)):
            s, e = w.chunk_range(c)
            B.pkv_prefetch(seq, sels[c], sels[c].numel(), B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_bwd(seq, q[c], o[c], do[c], lse[c], s, e - s, dq[c], sels[c], main)
        B.pkv_release_slots(seq, side)
        B.pkv_wait(seq, main, 10_000_000)
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        for c in range(n):
            np.testing.assert_array_equal(sels[c].cpu().numpy(), ref["sel"][c])
            assert np.abs(to_numpy(o[c]) - ref["o"][c]).max() <= 1e-2, c
            assert _rel(to_numpy(dq[c]), ref["dq"][c]) <= 2e-2, c
        assert _rel(to_numpy(dk), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)) <= 2e-2
        assert _rel(to_numpy(dv), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)) <= 2e-2
        st = B.pkv_stage_stats(seq)
        afresh = 2 * sum(len(u) for u in unions) * w.Hkv        # forward + backward
        graded = len(np.unique(np.concatenate(unions))) * w.Hkv
        assert st["kv_in"] < afresh, (st, afresh)
        # every page staged with gradients went back at least once; gradients
        # come in over the link only after a write-back (fresh pages are
        # recorded as zero and zero-filled in HBM)
        assert st["grads_out"] >= graded, (st, graded)
        assert st["grads_in"] <= st["grads_out"] - graded, (st, graded)
    finally:
        B.pkv_pool_destroy(pool)


def test_append_into_a_staged_partial_page_restages_it():
    """A page staged while partial is refreshed once an append completes it:
    the forward of the completed page matches the oracle."""
    w = _w(N=256, C=256, keys="normal", extra_pages=2)
    bt = synth.block_table(w)
    k, v, q = synth.chunk_k(w, 0), synth.chunk_v(w, 0), synth.chunk_q(w, 0)
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        dev = lambda x: to_device(np.ascontiguousarray(x), "bf16")
        pages = torch.tensor([0, 1], dtype=torch.int32, device="cuda")
        B.pkv_append(seq, dev(k[:200]), dev(v[:200]), 200, main)      # page 1 partial
        B.pkv_prefetch(seq, pages, 2, B.PKV_STAGE_KV, side)
        B.pkv_wait(seq, main, 0)
        B.pkv_append(seq, dev(k[200:]), dev(v[200:]), 56, main)       # completes page 1
        B.pkv_prefetch(seq, pages, 2, B.PKV_STAGE_KV, side)
        B.pkv_wait(seq, main, 0)
        qd = dev(q[128:])
        o = torch.empty_like(qd)
        lse = torch.empty((w.Hq, 128), dtype=torch.float32, device="cuda")
        B.pkv_chunk_attn_fwd(seq, qd, 128, 128, o, lse, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        o_ref, lse_ref = oracle.attention_forward(q[128:], k, v, 128)
        assert np.abs(to_numpy(o) - o_ref).max() <= 1e-2
        assert np.abs(to_numpy(lse) - lse_ref).max() <= 1e-2
    finally:
        B.pkv_pool_destroy(pool)


def _host_grads(pool, w):
    """numpy views of a PINNED_HOST pool's host gradient pages [n_phys, Hkv, P, d]."""
    import ctypes
    arr = B.pkv_pool_arrays(pool)
    shape = (w.n_phys, w.Hkv, w.P, w.d)
    n = int(np.prod(shape))
    return {t: np.ctypeslib.as_array((ctypes.c_float * n).from_address(arr[t])).reshape(shape)
            for t in ("dk", "dv")}


def test_zeroed_gradient_pages_are_recorded_not_written():
    """Gradient pages of a PINNED_HOST pool that are zero (fresh from an append,
    or after pkv_grad_zero) are recorded as zero in HBM and not written over the
    host link: with their host memory poisoned, pkv_gather reads zeros,
    pkv_grad_accumulate writes whole pages (bit-exact against the oracle's
    scatter-add onto zeros), staging fills slots with zeros without counting a
    transfer, and a write-back makes the host memory current -- in the slot
    cache and in whole-sequence staging."""
    w = synth.workload("qwen7b_sparse_256k", N=1024, C=512, Hq=4, Hkv=2, extra_pages=2,
                       topk=(2, 1, 2))
    bt = synth.block_table(w)
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    used = np.asarray(bt)[: w.n_pages]

    def gather():
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        return to_numpy(dk), to_numpy(dv)

    def sync():
        B.pkv_wait(seq, main, 5_000_000)
        torch.cuda.synchronize()
        B.pkv_check(pool)

    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            k = to_device(synth.chunk_k(w, c), "bf16")
            B.pkv_append(seq, k, k, e - s, main)
        torch.cuda.synchronize()
        host = _host_grads(pool, w)
        for t in host:
            host[t][...] = np.nan                     # nothing may read this memory as data
        dk, dv = gather()
        assert not dk.any() and not dv.any()
        assert np.isnan(host["dk"][used]).all()      # the appends wrote no zeros to the host

        # accumulation onto recorded pages writes them whole
        ref = {t: np.zeros((w.n_phys, w.Hkv, w.P, w.d), np.float32) for t in ("dk", "dv")}
        r0, n = 100, 300                              # pages 0..3, partially
        x = synth.draw_normal(w.seed, "misc", 400, (n, w.Hkv, w.d))
        y = synth.draw_normal(w.seed, "misc", 401, (n, w.Hkv, w.d))
        oracle.scatter_rows(ref["dk"], bt, r0, x, w.P, accumulate=True)
        oracle.scatter_rows(ref["dv"], bt, r0, y, w.P, accumulate=True)
        B.pkv_grad_accumulate(seq, r0, n, torch.from_numpy(x).cuda(), torch.from_numpy(y).cuda(), main)
        dk, dv = gather()
        np.testing.assert_array_equal(dk, oracle.logical_rows(ref["dk"], bt, w.N, w.P))
        np.testing.assert_array_equal(dv, oracle.logical_rows(ref["dv"], bt, w.N, w.P))
        np.testing.assert_array_equal(host["dk"][used[:4]], ref["dk"][used[:4]])
        assert np.isnan(host["dk"][used[4:]]).all()

        # slot cache: recorded pages are zero-filled, the others copied
        pages = torch.arange(w.n_pages, dtype=torch.int32, device="cuda")
        st0 = B.pkv_stage_stats(seq)
        B.pkv_prefetch(seq, pages, w.n_pages, B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
        B.pkv_writeback_grads(seq, side)
        sync()
        st1 = B.pkv_stage_stats(seq)
        assert st1["grads_in"] - st0["grads_in"] == 4 * w.Hkv
        assert st1["grads_out"] - st0["grads_out"] == w.n_pages * w.Hkv
        for t in host:                                # every host page is current now
            np.testing.assert_array_equal(host[t][used], ref[t][used])

        # zeroing while the gradients are staged zeroes the slots too
        B.pkv_grad_zero(seq, main)
        dk, dv = gather()
        assert not dk.any() and not dv.any()
        assert np.array_equal(host["dk"][used[:4]], ref["dk"][used[:4]])   # not written
        B.pkv_prefetch(seq, pages, w.n_pages, B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
        B.pkv_release_slots(seq, side)
        sync()
        assert not host["dk"][used].any() and not host["dv"][used].any()

        # whole-sequence staging by the copy engines
        B.pkv_grad_accumulate(seq, 0, w.N, torch.from_numpy(np.ones((w.N, w.Hkv, w.d), np.float32)).cuda(),
                              None, main)
        for zero_first in (False, True):
            if zero_first:                            # the cache is empty: host pages recorded
                B.pkv_grad_zero(seq, main)
            B.pkv_prefetch(seq, None, 0, B.PKV_STAGE_GRADS, side)   # copies stale host pages
            B.pkv_release_slots(seq, side)                           # writes the slots back
            sync()
            dk, dv = gather()
            assert (dk == (0.0 if zero_first else 1.0)).all() and not dv.any(), zero_first
            assert (host["dk"][used] == (0.0 if zero_first else 1.0)).all(), zero_first
    finally:
        B.pkv_pool_destroy(pool)
