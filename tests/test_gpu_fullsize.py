"""Full-size parity: the bench workloads, run exactly as bench.py runs them,
checked against the oracle on sampled outputs and on identities that hold at
any size; plus the bench's head layout (28 query heads, 4 KV heads, d 128,
page 128) in full at a size the oracle finishes.

Sampled: O, LSE and dQ of seeded query rows (the oracle computes each row
alone, over every key it sees). dK and dV of sampled pages for every KV head,
each against the oracle's sum over every query that sees the page (computed
in parallel by tests/oracle_pool.py):
  dense 32K: the final pool rows of a page of chunk 0, the pages on both
      sides of a chunk boundary, a page inside a later chunk and the last page;
  dense 128K, permuted table: the contribution of two whole chunks (the
      difference of the pool before and after each chunk's backward) to pages
      of chunk 0, on a chunk boundary and further on; these launches split
      each page's dK/dV over several CTAs that all add into the same rows;
  sparse 256K: every chunk's selection against the oracle (ties within 1e-5),
      then the final rows of pages that many query pages of many chunks
      selected, per KV head, over those selections;
  sparse 1M, pinned host: the sink page (selected by every query page), the
      most-selected candidate page and the chunk's first page, per KV head.
Identities: sum_j dK_j = 0 and sum_j dV_j = sum of dO over the group's heads
and queries, per KV head (rows of P sum to one; rows of dS sum to zero).
Tolerances as in the other parity tests: O/LSE max-abs 1e-2, dQ/dK/dV
relative Frobenius 2e-2 (per sampled page and KV head); identities 2e-2.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_device, to_numpy

from oracle_pool import OraclePool

pytestmark = pytest.mark.gpu
TIE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


@pytest.fixture(scope="module")
def opool():
    with OraclePool() as p:
        yield p


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _logical_kv(w):
    ks = np.concatenate([synth.chunk_k(w, c) for c in range(w.n_chunks)])
    vs = np.concatenate([synth.chunk_v(w, c) for c in range(w.n_chunks)])
    return ks, vs


def _check_rows(w, sw, K_all, V_all, c, heads, n_rows, allowed_pages=None):
    """O, LSE and dQ of sampled rows of chunk c against the oracle, row by row."""
    s, e = w.chunk_range(c)
    q = synth.chunk_q(w, c)
    do = synth.chunk_do(w, c)
    rng = np.random.default_rng(7 + c)
    rows = np.sort(rng.choice(e - s, size=n_rows, replace=False))
    o_gpu, lse_gpu, dq_gpu = to_numpy(sw.o[c]), to_numpy(sw.lse[c]), to_numpy(sw.dq[c])
    dq_ref, dq_got = [], []
    for h in heads:
        kv = h // w.g
        for r in rows:
            pos = s + int(r)
            k = K_all[: pos + 1, kv:kv + 1]
            v = V_all[: pos + 1, kv:kv + 1]
            allowed = None
            if allowed_pages is not None:
                # one query page (this row's), one KV head: its selected pages
                mask = np.zeros((1, 1, pos // w.P + 1), bool)
                mask[0, 0, allowed_pages[(int(r) // w.P, kv)]] = True
                allowed = mask
            qr = q[r:r + 1, h:h + 1]
            # the row's own query page is page 0 of this one-row "chunk": shift so
            # the mask lookup (q_pos - q_start) // P selects row 0 of the mask
            o, lse = oracle.attention_forward(qr, k, v, pos, w.P, allowed)
            dq, _, _ = oracle.attention_backward(qr, k, v, o, do[r:r + 1, h:h + 1], lse, pos, w.P, allowed)
            assert abs(o_gpu[r, h] - o[0, 0]).max() <= 1e-2, (c, h, r)
            assert abs(lse_gpu[h, r] - lse[0, 0]) <= 1e-2, (c, h, r)
            dq_ref.append(dq[0, 0])
            dq_got.append(dq_gpu[r, h])
    assert _rel(np.array(dq_got), np.array(dq_ref)) <= 2e-2


def _check_identities(w, g, dos_sum):
    dk, dv = to_numpy(g["dk"]), to_numpy(g["dv"])
    for kv in range(w.Hkv):
        sk = dk[:, kv].sum(0)
        assert np.linalg.norm(sk) <= 2e-2 * np.sqrt((dk[:, kv] ** 2).sum()), kv
        sv = dv[:, kv].sum(0)
        assert _rel(sv, dos_sum[kv]) <= 2e-2, kv


def _dos_sum(w):
    dos_sum = np.zeros((w.Hkv, w.d))
    for c in range(w.n_chunks):
        do = synth.chunk_do(w, c).astype(np.float64)
        for kv in range(w.Hkv):
            dos_sum[kv] += do[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))
    return dos_sum


def _page_rows(seq, w, pages, stream=None):
    """The gradient pool's dK/dV rows of the given logical pages, [P, Hkv, d] each."""
    out = {}
    for p in pages:
        dk = torch.empty((w.P, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather_rows(seq, p * w.P, w.P, None, None, dk, dv, stream)
        out[p] = (dk, dv)
    torch.cuda.synchronize()
    return {p: (to_numpy(a).astype(np.float64), to_numpy(b).astype(np.float64))
            for p, (a, b) in out.items()}


def _check_pages(got, want, what):
    """Per page and KV head: relative Frobenius <= 2e-2 for dK and dV."""
    for p in want:
        for kv in range(want[p][0].shape[1]):
            for t, name in ((0, "dk"), (1, "dv")):
                e = _rel(got[p][t][:, kv], want[p][t][:, kv])
                assert e <= 2e-2, (what, name, p, kv, e)


def test_dense_32k_full_size_sampled(opool):
    w = synth.workload("qwen7b_dense_32k")
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.run()
        B.pkv_check(sw.pool)
        g = sw.gather()
        K_all, V_all = _logical_kv(w)
        last = w.n_chunks - 1
        _check_rows(w, sw, K_all, V_all, last, heads=(0, 13, w.Hq - 1), n_rows=16)
        _check_rows(w, sw, K_all, V_all, 0, heads=(6, 20), n_rows=16)
        _check_identities(w, g, _dos_sum(w))
        # final rows: chunk 0's page 3 (every chunk adds into it), both sides of
        # the chunk 3 / chunk 4 boundary, a page inside chunk 6, the last page
        ppc = w.C // w.P
        pages = [3, 4 * ppc - 1, 4 * ppc, 6 * ppc + 8, w.n_pages - 1]
        want = opool.dense_page_grads(w, pages)
        dk, dv = to_numpy(g["dk"]), to_numpy(g["dv"])
        got = {p: (dk[p * w.P:(p + 1) * w.P], dv[p * w.P:(p + 1) * w.P]) for p in pages}
        _check_pages(got, want, "final")
    finally:
        sw.close()


def test_dense_128k_perm_full_size_sampled(opool):
    w = synth.workload("qwen7b_dense_128k_perm")
    ppc = w.C // w.P
    # chunk -> the pages whose contribution from that chunk is checked
    probe = {8: [3, ppc - 1, ppc, 8 * ppc - 1, 8 * ppc, 8 * ppc + 58],
             1: [3, ppc - 1, ppc, 2 * ppc - 1]}
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        for c in range(w.n_chunks):
            sw.forward(c)
        snaps = {}
        for c in reversed(range(w.n_chunks)):
            if c in probe:
                snaps[(c, "before")] = _page_rows(sw.seq, w, probe[c])
            sw.backward(c)
            if c in probe:
                snaps[(c, "after")] = _page_rows(sw.seq, w, probe[c])
        B.pkv_check(sw.pool)
        g = sw.gather()
        for c, pages in probe.items():
            got = {p: (snaps[(c, "after")][p][0] - snaps[(c, "before")][p][0],
                       snaps[(c, "after")][p][1] - snaps[(c, "before")][p][1]) for p in pages}
            want = opool.dense_page_grads(w, pages, chunks=[c])
            _check_pages(got, want, f"chunk {c}")
        K_all, V_all = _logical_kv(w)
        last = w.n_chunks - 1
        _check_rows(w, sw, K_all, V_all, last, heads=(0, 13, w.Hq - 1), n_rows=16)
        _check_rows(w, sw, K_all, V_all, 0, heads=(6, 20), n_rows=16)
        _check_identities(w, g, _dos_sum(w))
        # the last page's final rows: only the last page's own queries see it
        page = w.n_pages - 1
        want = opool.dense_page_grads(w, [page], chunks=[last], block=128)
        dk, dv = to_numpy(g["dk"]), to_numpy(g["dv"])
        _check_pages({page: (dk[page * w.P:], dv[page * w.P:])}, want, "final")
    finally:
        sw.close()


def _check_selection(sel_gpu, q, s, K_all, w, K, ns, nl):
    """The GPU's selection of every query page and KV head of a chunk against
    the oracle (a differing page must score within 1e-5 of the K-th score).
    Returns {(i, kv): the GPU's list}."""
    e = s + q.shape[0]
    lists, _ = oracle.chunk_selection(q, s, K_all[:e], w.P, K, ns, nl)
    qbar = oracle.query_page_means(q, w.P, w.Hkv)
    rep = oracle.page_representatives(K_all[:e], w.P)
    got_lists = {}
    for i in range(len(lists)):
        for kv in range(w.Hkv):
            got = [int(x) for x in sel_gpu[i, kv] if x >= 0]
            want = lists[i][kv]
            if got != want:
                qpg = s // w.P + i
                cand = np.arange(ns, qpg - nl + 1)
                kth = np.sort(rep[cand, kv] @ qbar[i, kv])[::-1][K - 1]
                for pg in set(got) ^ set(want):
                    assert abs(rep[pg, kv] @ qbar[i, kv] - kth) <= TIE, (s, i, kv, pg)
            got_lists[(i, kv)] = got
    return got_lists


def test_sparse_256k_full_size_sampled(opool):
    w = synth.workload("qwen7b_sparse_256k")
    K, ns, nl = w.topk
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sel)
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, sel=sels[c])
        B.pkv_check(sw.pool)
        g = sw.gather()
        K_all, V_all = _logical_kv(w)
        # every chunk's selection against the oracle
        lists = {}
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            lists[c] = _check_selection(sels[c].cpu().numpy(), synth.chunk_q(w, c), s, K_all, w,
                                        K, ns, nl)
        last = w.n_chunks - 1
        _check_rows(w, sw, K_all, V_all, last, heads=(0, 15, w.Hq - 1), n_rows=12,
                    allowed_pages=lists[last])
        _check_identities(w, g, _dos_sum(w))
        # sampled pages per KV head: among the pages of chunks 0 and 1 (not the
        # sink) that query pages of at least 3 chunks picked, the one picked
        # least often (bounding the oracle's work); the last page of chunk 15
        # (a chunk boundary); page 1500
        ppc = w.C // w.P
        count, chunks_of = {}, {}
        for c, lc in lists.items():
            for (i, kv), pl in lc.items():
                for p in pl:
                    count[(p, kv)] = count.get((p, kv), 0) + 1
                    chunks_of.setdefault((p, kv), set()).add(c)
        pages_by_kv = {}
        for kv in range(w.Hkv):
            early = [p for p in range(ns, 2 * ppc) if len(chunks_of.get((p, kv), ())) >= 3]
            assert early, kv
            p0 = min(early, key=lambda p: (count[(p, kv)], p))
            pages_by_kv[kv] = [p0, 16 * ppc - 1, 1500]
        want, n_tasks = opool.sparse_page_grads(
            w, lists, pages_by_kv, lambda p: (K_all[p * w.P:(p + 1) * w.P], V_all[p * w.P:(p + 1) * w.P]))
        dk, dv = to_numpy(g["dk"]), to_numpy(g["dv"])
        for (p, kv), (wk, wv) in want.items():
            rows = slice(p * w.P, (p + 1) * w.P)
            assert _rel(dk[rows, kv], wk) <= 2e-2, ("dk", p, kv)
            assert _rel(dv[rows, kv], wv) <= 2e-2, ("dv", p, kv)
    finally:
        sw.close()


def test_local_256k_full_size_sampled():
    """The local-attention workload as bench.py runs it: every chunk's page lists
    bit-exact, sampled rows of the first and last chunks over their local pages,
    dK/dV of one page in the middle (seen by its own and the next query page
    only) against the oracle, and the gradient identities."""
    w = synth.workload("qwen7b_local_256k")
    ns, nl = w.local
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            sel = torch.empty(((e - s) // w.P, w.Hkv, ns + nl), dtype=torch.int32, device="cuda")
            B.pkv_page_local(sw.seq, s, e - s, ns, nl, sel)
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, sel=sels[c])
        B.pkv_check(sw.pool)
        g = sw.gather()
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            _, want = oracle.chunk_local_selection(s, e - s, w.Hkv, w.P, ns, nl)
            np.testing.assert_array_equal(sels[c].cpu().numpy(), want)
        K_all, V_all = _logical_kv(w)
        for c in (0, w.n_chunks - 1):
            s, e = w.chunk_range(c)
            allowed = {(i, kv): oracle.local_pages(s // w.P + i, ns, nl)
                       for i in range((e - s) // w.P) for kv in range(w.Hkv)}
            _check_rows(w, sw, K_all, V_all, c, heads=(0, 15, w.Hq - 1), n_rows=12,
                        allowed_pages=allowed)
        # page p's keys are seen by query pages p .. p + nl - 1 only
        p = w.n_pages // 2 + 5
        q0, q1 = p * w.P, (p + nl) * w.P
        Q = np.concatenate([synth.chunk_q(w, c) for c in range(w.n_chunks)
                            if w.chunk_range(c)[1] > q0 and w.chunk_range(c)[0] < q1])
        DO = np.concatenate([synth.chunk_do(w, c) for c in range(w.n_chunks)
                             if w.chunk_range(c)[1] > q0 and w.chunk_range(c)[0] < q1])
        c_first = q0 // w.C
        off = q0 - c_first * w.C
        Q, DO = Q[off:off + (q1 - q0)], DO[off:off + (q1 - q0)]
        # no sink pages: these queries see pages p - nl + 1 .. p + nl - 1 only, so
        # the oracle runs on those keys, positions shifted to start at page b
        assert ns == 0
        b = p - nl + 1
        lists = [[[x - b for x in oracle.local_pages(p + i, ns, nl)]] * w.Hkv for i in range(nl)]
        allowed = oracle.page_allowed_from_lists(lists, p + nl - b)
        Kw, Vw = K_all[b * w.P:q1], V_all[b * w.P:q1]
        o, lse = oracle.attention_forward(Q, Kw, Vw, q0 - b * w.P, w.P, allowed)
        _, dk, dv = oracle.attention_backward(Q, Kw, Vw, o, DO, lse, q0 - b * w.P, w.P, allowed)
        rows = slice((p - b) * w.P, (p - b + 1) * w.P)
        grow = slice(p * w.P, (p + 1) * w.P)
        assert _rel(to_numpy(g["dk"])[grow], dk[rows]) <= 2e-2
        assert _rel(to_numpy(g["dv"])[grow], dv[rows]) <= 2e-2
        _check_identities(w, g, _dos_sum(w))
    finally:
        sw.close()


def test_sparse_1m_pinned_host_full_size_sampled(opool):
    """The 1M-token pinned-host workload as bench.py runs it: every K/V page and
    fp32 gradient page in mapped pinned host memory, the last chunk's selected
    pages staged into HBM slots on a side stream for its forward and backward,
    the gradients written back. Checked against the oracle: the selection of
    every query page (representatives from the seeded keys, ties within 1e-5);
    O, LSE and dQ of sampled rows, each computed by the oracle over that row's
    selected pages gathered into a compact key sequence (the row's own page
    last, so the causal mask falls where it does in the full sequence); and,
    over the whole written-back gradient pool, sum dK = 0 and sum dV = sum dO
    per KV head (the pool holds only this chunk's contribution)."""
    w = synth.workload("qwen7b_sparse_1m_offload")
    K, ns, nl = w.topk
    n = w.n_chunks
    c = n - 1
    s, e = w.chunk_range(c)
    ppc = w.C // w.P                                    # pages per chunk
    bt = synth.block_table(w)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        rep = np.zeros((w.n_pages, w.Hkv, w.d))
        for i in range(n):
            a, b_ = w.chunk_range(i)
            k_np = synth.chunk_k(w, i)
            rep[i * ppc:(i + 1) * ppc] = oracle.page_representatives(k_np, w.P)
            B.pkv_append(seq, to_device(k_np, "bf16"), to_device(synth.chunk_v(w, i), "bf16"),
                         b_ - a, main)
        q_np, do_np = synth.chunk_q(w, c), synth.chunk_do(w, c)
        q, do = to_device(q_np, "bf16"), to_device(do_np, "bf16")
        o, dq = torch.empty_like(q), torch.empty_like(q)
        lse = torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda")
        sel = torch.empty((w.C // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
        B.pkv_page_topk(seq, q, s, e - s, K, ns, nl, sel, None, main)
        B.pkv_prefetch(seq, sel, sel.numel(), B.PKV_STAGE_KV, side)
        B.pkv_wait(seq, main, 0)
        B.pkv_chunk_attn_fwd(seq, q, s, e - s, o, lse, sel, main)
        B.pkv_prefetch(seq, sel, sel.numel(), B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
        B.pkv_wait(seq, main, 0)
        B.pkv_chunk_attn_bwd(seq, q, o, do, lse, s, e - s, dq, sel, main)
        B.pkv_writeback_grads(seq, side)
        B.pkv_wait(seq, main, 60_000_000)
        torch.cuda.synchronize()
        B.pkv_check(pool)

        # selection of every query page and KV head
        sel_gpu = sel.cpu().numpy()
        qbar = oracle.query_page_means(q_np, w.P, w.Hkv)
        qp0 = s // w.P
        lists = {}
        for i in range(sel_gpu.shape[0]):
            for kv in range(w.Hkv):
                got = [int(x) for x in sel_gpu[i, kv] if x >= 0]
                want = oracle.select_pages(qbar[i, kv], rep[:, kv, :], qp0 + i, K, ns, nl)
                if got != want:
                    cand = np.arange(ns, qp0 + i - nl + 1)
                    kth = np.sort(rep[cand, kv] @ qbar[i, kv])[::-1][K - 1]
                    for pg in set(got) ^ set(want):
                        assert abs(rep[pg, kv] @ qbar[i, kv] - kth) <= 1e-5, (i, kv, pg)
                lists[(i, kv)] = got

        # sampled rows over their selected pages (compact key sequences)
        rng = np.random.default_rng(11)
        rows = np.sort(rng.choice(e - s, size=6, replace=False))
        heads = (0, 13, w.Hq - 1)
        need = sorted({pg for r in rows for h in heads for pg in lists[(int(r) // w.P, h // w.g)]})
        kv_rows = {}
        for ch in sorted({pg // ppc for pg in need}):
            kc, vc = synth.chunk_k(w, ch), synth.chunk_v(w, ch)
            for pg in need:
                if pg // ppc == ch:
                    o0 = (pg - ch * ppc) * w.P
                    kv_rows[pg] = (kc[o0:o0 + w.P], vc[o0:o0 + w.P])
        o_gpu, lse_gpu, dq_gpu = to_numpy(o), to_numpy(lse), to_numpy(dq)
        dq_ref, dq_got = [], []
        for h in heads:
            kv = h // w.g
            for r in rows:
                pages = lists[(int(r) // w.P, kv)]
                assert pages[-1] == qp0 + int(r) // w.P           # own page listed last
                kc = np.concatenate([kv_rows[pg][0][:, kv:kv + 1] for pg in pages])
                vc = np.concatenate([kv_rows[pg][1][:, kv:kv + 1] for pg in pages])
                pos = (len(pages) - 1) * w.P + int(r) % w.P       # compact position
                qr, dor = q_np[r:r + 1, h:h + 1], do_np[r:r + 1, h:h + 1]
                o_r, lse_r = oracle.attention_forward(qr, kc[:pos + 1], vc[:pos + 1], pos)
                dq_r, _, _ = oracle.attention_backward(qr, kc[:pos + 1], vc[:pos + 1], o_r, dor,
                                                       lse_r, pos)
                assert abs(o_gpu[r, h] - o_r[0, 0]).max() <= 1e-2, (h, r)
                assert abs(lse_gpu[h, r] - lse_r[0, 0]) <= 1e-2, (h, r)
                dq_ref.append(dq_r[0, 0])
                dq_got.append(dq_gpu[r, h])
        assert _rel(np.array(dq_got), np.array(dq_ref)) <= 2e-2

        # gradient-pool identities over the whole written-back pool
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None, main)
        torch.cuda.synchronize()
        # sampled pages per KV head against the oracle over this chunk's
        # selections: the sink page (every query page lists it), the candidate
        # page the most query pages picked, and the chunk's first page
        pages_by_kv = {}
        for kv in range(w.Hkv):
            cnt = {}
            for i in range(sel_gpu.shape[0]):
                for pg in lists[(i, kv)]:
                    if ns <= pg < qp0:
                        cnt[pg] = cnt.get(pg, 0) + 1
            top = max(cnt, key=lambda pg: (cnt[pg], -pg))
            pages_by_kv[kv] = [0, top, qp0]
        @functools.lru_cache(maxsize=1)
        def kv_chunk(ch):
            return synth.chunk_k(w, ch), synth.chunk_v(w, ch)

        def page_kv(pg):                          # pages are asked for in ascending order
            kc, vc = kv_chunk(pg // ppc)
            o0 = (pg % ppc) * w.P
            return kc[o0:o0 + w.P], vc[o0:o0 + w.P]

        want, _ = opool.sparse_page_grads(w, {c: lists}, pages_by_kv, page_kv)
        for (pg, kv), (wk, wv) in want.items():
            rows = slice(pg * w.P, (pg + 1) * w.P)
            assert _rel(dk[rows, kv].double().cpu().numpy(), wk) <= 2e-2, ("dk", pg, kv)
            assert _rel(dv[rows, kv].double().cpu().numpy(), wv) <= 2e-2, ("dv", pg, kv)
        sk = dk.double().sum(0).cpu().numpy()
        sv = dv.double().sum(0).cpu().numpy()
        nk = torch.sqrt((dk.double() ** 2).sum(0).sum(-1)).cpu().numpy()
        do64 = do_np.astype(np.float64)
        for kv in range(w.Hkv):
            assert np.linalg.norm(sk[kv]) <= 2e-2 * nk[kv], kv
            assert _rel(sv[kv], do64[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))) <= 2e-2, kv
    finally:
        B.pkv_pool_destroy(pool)


def _gpu_sweep_outputs(sw):
    g = sw.gather()
    return dict(o=[to_numpy(x) for x in sw.o], lse=[to_numpy(x) for x in sw.lse],
                dq=[to_numpy(x) for x in sw.dq], dk=to_numpy(g["dk"]), dv=to_numpy(g["dv"]))


def _compare_all(w, got, ref):
    for c in range(w.n_chunks):
        assert np.abs(got["o"][c] - ref["o"][c]).max() <= 1e-2, ("o", c)
        assert np.abs(got["lse"][c] - ref["lse"][c]).max() <= 1e-2, ("lse", c)
        assert _rel(got["dq"][c], ref["dq"][c]) <= 2e-2, ("dq", c)
    for kv in range(w.Hkv):
        assert _rel(got["dk"][:, kv], ref["dk"][:, kv]) <= 2e-2, ("dk", kv)
        assert _rel(got["dv"][:, kv], ref["dv"][:, kv]) <= 2e-2, ("dv", kv)


def test_bench_head_layout_dense_8k_every_output(opool):
    """28 query heads / 4 KV heads, d 128, page 128, chunks of 4096 as in the
    dense bench workload, at 8192 tokens (two chunks, permuted pages): O, LSE,
    dQ, dK, dV of every position against the oracle, element by element."""
    w = synth.workload("qwen7b_dense_32k", N=8192, table="perm", extra_pages=5)
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.run()
        B.pkv_check(sw.pool)
        got = _gpu_sweep_outputs(sw)
    finally:
        sw.close()
    _compare_all(w, got, opool.dense_full(w))


def test_bench_head_layout_sparse_16k_every_output(opool):
    """The page-sparse bench workload's layout and selection (top-64 + 1 sink +
    2 local, clustered keys, chunks of 8192, permuted pages) at 16384 tokens:
    the selections against the oracle, then O, LSE, dQ, dK, dV of every
    position against the oracle over those selections."""
    w = synth.workload("qwen7b_sparse_256k", N=16384)
    K, ns, nl = w.topk
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
            sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
            B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sel)
            sels.append(sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c, sel=sels[c])
        B.pkv_check(sw.pool)
        got = _gpu_sweep_outputs(sw)
        K_all, V_all = _logical_kv(w)
        lists = {c: _check_selection(sels[c].cpu().numpy(), synth.chunk_q(w, c),
                                     w.chunk_range(c)[0], K_all, w, K, ns, nl)
                 for c in range(w.n_chunks)}
    finally:
        sw.close()
    _compare_all(w, got, opool.sparse_full(
        w, lists, lambda p: (K_all[p * w.P:(p + 1) * w.P], V_all[p * w.P:(p + 1) * w.P])))


def test_sparse_chunk_of_320_query_pages_every_output(opool):
    """One chunk of 40960 tokens (320 query pages, more than 256) through the
    page-sparse tensor-core kernels: selections against the oracle, then O,
    LSE, dQ, dK, dV of every position against the oracle over them."""
    w = synth.workload("qwen7b_sparse_256k", N=40960, C=40960, Hq=2, Hkv=1, topk=(4, 1, 2))
    K, ns, nl = w.topk
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        s, e = w.chunk_range(0)
        B.pkv_append(sw.seq, sw.k[0], sw.v[0], e - s)
        sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32, device="cuda")
        B.pkv_page_topk(sw.seq, sw.q[0], s, e - s, K, ns, nl, sel)
        B.pkv_chunk_attn_fwd(sw.seq, sw.q[0], s, e - s, sw.o[0], sw.lse[0], sel)
        sw.backward(0, sel=sel)
        B.pkv_check(sw.pool)
        got = _gpu_sweep_outputs(sw)
        K_all, V_all = _logical_kv(w)
        lists = {0: _check_selection(sel.cpu().numpy(), synth.chunk_q(w, 0), 0, K_all, w, K, ns, nl)}
    finally:
        sw.close()
    _compare_all(w, got, opool.sparse_full(
        w, lists, lambda p: (K_all[p * w.P:(p + 1) * w.P], V_all[p * w.P:(p + 1) * w.P])))
