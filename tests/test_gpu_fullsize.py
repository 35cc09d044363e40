"""Full-size parity: the bench workloads, run exactly as bench.py runs them,
checked against the oracle on sampled outputs and on identities that hold at
any size.

Sampled: O, LSE and dQ of seeded query rows (the oracle computes each row
alone, over every key it sees); dK and dV of the last page (seen only by the
last page's queries). Sparse: the selection of every query page of the last
chunk (ties within 1e-5 allowed), and rows over the selected pages. Identities:
sum_j dK_j = 0 and sum_j dV_j = sum of dO over the group's heads and queries,
per KV head (rows of P sum to one; rows of dS sum to zero), for dense and
sparse alike. Tolerances as in the other parity tests: O/LSE max-abs 1e-2,
dQ/dK/dV relative Frobenius 2e-2; identities relative 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


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


@pytest.mark.parametrize("name", ["qwen7b_dense_32k", "qwen7b_dense_128k_perm"])
def test_dense_full_size_sampled(name):
    w = synth.workload(name)
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.run()
        B.pkv_check(sw.pool)
        g = sw.gather()
        K_all, V_all = _logical_kv(w)
        last = w.n_chunks - 1
        _check_rows(w, sw, K_all, V_all, last, heads=(0, 13, w.Hq - 1), n_rows=16)
        _check_rows(w, sw, K_all, V_all, 0, heads=(6, 20), n_rows=16)
        dos_sum = np.zeros((w.Hkv, w.d))
        for c in range(w.n_chunks):
            do = synth.chunk_do(w, c).astype(np.float64)
            for kv in range(w.Hkv):
                dos_sum[kv] += do[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))
        _check_identities(w, g, dos_sum)
        # the last page: only the last page's own queries see it
        page = w.n_pages - 1
        p0 = page * w.P
        dk_gpu, dv_gpu = to_numpy(g["dk"]), to_numpy(g["dv"])
        s, e = w.chunk_range(last)
        q = synth.chunk_q(w, last)[p0 - s:]
        do = synth.chunk_do(w, last)[p0 - s:]
        o, lse = oracle.attention_forward(q, K_all, V_all, p0)
        _, dk, dv = oracle.attention_backward(q, K_all, V_all, o, do, lse, p0)
        assert _rel(dk_gpu[p0:], dk[p0:]) <= 2e-2
        assert _rel(dv_gpu[p0:], dv[p0:]) <= 2e-2
    finally:
        sw.close()


def test_sparse_256k_full_size_sampled():
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
        last = w.n_chunks - 1
        s, e = w.chunk_range(last)
        q = synth.chunk_q(w, last)
        sel_gpu = sels[last].cpu().numpy()
        # selection of every query page of the last chunk vs the oracle (tie rule 1e-5)
        lists, _ = oracle.chunk_selection(q, s, K_all[:e], w.P, K, ns, nl)
        qbar = oracle.query_page_means(q, w.P, w.Hkv)
        rep = oracle.page_representatives(K_all[:e], w.P)
        allowed = {}
        for i in range(len(lists)):
            for kv in range(w.Hkv):
                got = [int(x) for x in sel_gpu[i, kv] if x >= 0]
                want = lists[i][kv]
                if got != want:
                    qpg = s // w.P + i
                    cand = np.arange(ns, qpg - nl + 1)
                    kth = np.sort(rep[cand, kv] @ qbar[i, kv])[::-1][K - 1]
                    for pg in set(got) ^ set(want):
                        assert abs(rep[pg, kv] @ qbar[i, kv] - kth) <= 1e-5, (i, kv, pg)
                allowed[(i, kv)] = got          # the pages the GPU attended to
        _check_rows(w, sw, K_all, V_all, last, heads=(0, 15, w.Hq - 1), n_rows=12,
                    allowed_pages=allowed)
        dos_sum = np.zeros((w.Hkv, w.d))
        for c in range(w.n_chunks):
            do = synth.chunk_do(w, c).astype(np.float64)
            for kv in range(w.Hkv):
                dos_sum[kv] += do[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))
        _check_identities(w, g, dos_sum)
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
        dos_sum = np.zeros((w.Hkv, w.d))
        for c in range(w.n_chunks):
            do = synth.chunk_do(w, c).astype(np.float64)
            for kv in range(w.Hkv):
                dos_sum[kv] += do[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))
        _check_identities(w, g, dos_sum)
    finally:
        sw.close()


def test_sparse_1m_pinned_host_full_size_sampled():
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
        sk = dk.double().sum(0).cpu().numpy()
        sv = dv.double().sum(0).cpu().numpy()
        nk = torch.sqrt((dk.double() ** 2).sum(0).sum(-1)).cpu().numpy()
        do64 = do_np.astype(np.float64)
        for kv in range(w.Hkv):
            assert np.linalg.norm(sk[kv]) <= 2e-2 * nk[kv], kv
            assert _rel(sv[kv], do64[:, kv * w.g:(kv + 1) * w.g].sum((0, 1))) <= 2e-2, kv
    finally:
        B.pkv_pool_destroy(pool)
