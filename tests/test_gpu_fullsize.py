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
from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_numpy

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
