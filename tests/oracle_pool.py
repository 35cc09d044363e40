"""The fp64 oracle at the bench workloads' sizes, spread over worker processes.

Test infrastructure. At 32K-1M tokens one exact oracle value (the dK/dV of
one page, say) depends on every query that sees the page, each with its whole
softmax row, so a single numpy process would need minutes. Here the work is
split over query rows, chunks and KV heads and handed to worker processes
started with "spawn" (never forked from a process that may already hold a
CUDA context), each running single-threaded BLAS. Every worker calls only
``oracle`` functions on inputs it regenerates from the seeded generators in
``synth``; no value comes from the CUDA path.

Two exact restatements keep the work small; both follow from the definition
of causal attention that the oracle writes out:

* dK/dV of the keys of one page p: P_ij, D_i and dS_ij need only the row's
  LSE and O (from the oracle's own forward over the row's whole key range)
  and the page's own keys. So the oracle's backward is called on the page's
  P keys alone, with the query positions shifted by -p*P (key positions
  restart at 0); its dK/dV are the page's rows, its dQ is discarded.
* A page-sparse row sees its selected pages only, and the causal mask acts
  only inside its own page, the last of its list. So the row's attention is
  dense causal attention over the selected pages' keys laid end to end, with
  the row at its place in the last page.
"""
from __future__ import annotations

import functools
import multiprocessing as mp
import os
import shutil
import tempfile

import numpy as np

import oracle
from paged_kv_chunk_chunked_gb300 import synth

_THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


@functools.lru_cache(maxsize=None)
def _kv_chunk(w: synth.Workload, c: int):
    return synth.chunk_k(w, c), synth.chunk_v(w, c)


@functools.lru_cache(maxsize=2)
def _q_do_chunk(w: synth.Workload, c: int):
    return synth.chunk_q(w, c), synth.chunk_do(w, c)


def _keys(w: synth.Workload, kv: int, L: int):
    """K, V of one KV head for positions 0..L-1, [L, 1, d] float32."""
    ks, vs = [], []
    for c in range(w.n_chunks):
        s, e = w.chunk_range(c)
        if s >= L:
            break
        k, v = _kv_chunk(w, c)
        ks.append(k[: L - s, kv:kv + 1])
        vs.append(v[: L - s, kv:kv + 1])
    return np.concatenate(ks), np.concatenate(vs)


def _dense_rows_task(args):
    """Chunk c, KV head kv, chunk rows [r0, r1), dense causal attention.

    Returns the rows' O and LSE (the group's g query heads); with want_dq
    also their dQ and the dK/dV rows of every key 0..s+r1-1 contributed by
    these queries; and, for each listed page, that page's dK/dV rows."""
    w, c, kv, r0, r1, pages, want_dq = args
    s, _ = w.chunk_range(c)
    g = w.g
    q_all, do_all = _q_do_chunk(w, c)
    q = q_all[r0:r1, kv * g:(kv + 1) * g]
    do = do_all[r0:r1, kv * g:(kv + 1) * g]
    L = s + r1
    K, V = _keys(w, kv, L)
    o, lse = oracle.attention_forward(q, K, V, s + r0)
    dq = dk_all = dv_all = None
    if want_dq:
        dq, dk_all, dv_all = oracle.attention_backward(q, K, V, o, do, lse, s + r0)
        dk_all, dv_all = dk_all[:, 0], dv_all[:, 0]
    out = {}
    for p in pages:
        a = p * w.P
        if a >= L:
            continue
        b = min(L, a + w.P)
        _, dk, dv = oracle.attention_backward(q, K[a:b], V[a:b], o, do, lse, s + r0 - a)
        out[p] = (dk[:, 0], dv[:, 0])
    return (c, kv, r0, r1, o, lse, dq, dk_all, dv_all, out)


@functools.lru_cache(maxsize=2)
def _page_store(path: str):
    """(page -> row index, K pages, V pages) saved by OraclePool._share_pages;
    the page arrays are memory-mapped [n, P, Hkv, d] float32."""
    idx = np.load(os.path.join(path, "idx.npy"))
    K = np.load(os.path.join(path, "k.npy"), mmap_mode="r")
    V = np.load(os.path.join(path, "v.npy"), mmap_mode="r")
    return {int(p): r for r, p in enumerate(idx)}, K, V


def _sparse_qpage_task(args):
    """One query page (page i of chunk c; its rows q, do [n, g, d]) and KV head
    kv over its selected pages ``sel`` (ascending, own page last). Returns the
    rows' O, LSE, dQ and the dK/dV rows of each listed page that the selection
    holds."""
    w, c, i, kv, sel, pages, q, do, store = args
    P = w.P
    row, Ks, Vs = _page_store(store)
    Kc = np.concatenate([Ks[row[pg], :, kv:kv + 1] for pg in sel])
    Vc = np.concatenate([Vs[row[pg], :, kv:kv + 1] for pg in sel])
    own = (len(sel) - 1) * P                      # compact position of the row block
    o, lse = oracle.attention_forward(q, Kc, Vc, own)
    dq, _, _ = oracle.attention_backward(q, Kc, Vc, o, do, lse, own)
    out = {}
    for p in pages:
        if p in sel:
            a = sel.index(p) * P
            _, dk, dv = oracle.attention_backward(q, Kc[a:a + P], Vc[a:a + P], o, do, lse, own - a)
            out[p] = (dk[:, 0], dv[:, 0])
    return (c, i, kv, o, lse, dq, out)


def _each(it, n, timeout_s):
    """The n results of an imap_unordered iterator (chunk size 1); a worker
    that does not answer within timeout_s (a pool that cannot start its
    workers, say) fails the caller instead of hanging it."""
    for _ in range(n):
        yield it.next(timeout_s)


class OraclePool:
    """A spawn-started process pool of single-threaded oracle workers."""

    timeout_s = 1800

    def __init__(self, processes: int = 0):
        n = processes or max(1, min(32, os.cpu_count() or 1))
        saved = {k: os.environ.get(k) for k in _THREAD_VARS}
        for k in _THREAD_VARS:
            os.environ[k] = "1"                 # inherited by the spawned workers
        try:
            self.pool = mp.get_context("spawn").Pool(n)
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v
        self.n = n

    def close(self):
        self.pool.close()
        self.pool.join()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.pool.terminate()
        self.pool.join()

    def dense_page_grads(self, w, pages, chunks=None, kvs=None, block=512):
        """dK, dV of the listed pages from the queries of the given chunks
        (default: every chunk), dense causal. Returns {page: (dk, dv)}, each
        [P, Hkv, d] fp64, with zeros for KV heads not in kvs."""
        chunks = range(w.n_chunks) if chunks is None else chunks
        kvs = range(w.Hkv) if kvs is None else kvs
        tasks = []
        for c in chunks:
            s, e = w.chunk_range(c)
            for kv in kvs:
                for r0 in range(0, e - s, block):
                    r1 = min(e - s, r0 + block)
                    if s + r1 - 1 < min(pages) * w.P:
                        continue
                    tasks.append((w, c, kv, r0, r1, list(pages), False))
        acc = {p: (np.zeros((w.P, w.Hkv, w.d)), np.zeros((w.P, w.Hkv, w.d))) for p in pages}
        for (_, kv, _, _, _, _, _, _, _, out) in _each(self.pool.imap_unordered(
                _dense_rows_task, tasks), len(tasks), self.timeout_s):
            for p, (dk, dv) in out.items():
                acc[p][0][: dk.shape[0], kv] += dk
                acc[p][1][: dv.shape[0], kv] += dv
        return acc

    def dense_full(self, w, block=512):
        """The whole chunk-recurrent sweep, dense: per-chunk O [n, Hq, d],
        LSE [Hq, n], dQ [n, Hq, d], and the final dK, dV [N, Hkv, d] in
        logical order (every chunk's contribution summed)."""
        o = [np.zeros((e - s, w.Hq, w.d)) for s, e in map(w.chunk_range, range(w.n_chunks))]
        lse = [np.zeros((w.Hq, x.shape[0])) for x in o]
        dq = [np.zeros_like(x) for x in o]
        dk = np.zeros((w.N, w.Hkv, w.d))
        dv = np.zeros_like(dk)
        tasks = [(w, c, kv, r0, min(o[c].shape[0], r0 + block), [], True)
                 for c in range(w.n_chunks) for kv in range(w.Hkv)
                 for r0 in range(0, o[c].shape[0], block)]
        g = w.g
        for (c, kv, r0, r1, o_, l_, dq_, dk_, dv_, _) in _each(self.pool.imap_unordered(
                _dense_rows_task, tasks), len(tasks), self.timeout_s):
            o[c][r0:r1, kv * g:(kv + 1) * g] = o_
            lse[c][kv * g:(kv + 1) * g, r0:r1] = l_
            dq[c][r0:r1, kv * g:(kv + 1) * g] = dq_
            dk[: dk_.shape[0], kv] += dk_
            dv[: dv_.shape[0], kv] += dv_
        return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)

    def _share_pages(self, w, lists, page_kv):
        """Writes the K/V pages that the selections list to memory-mapped files
        for the workers. page_kv(p) -> (k, v), each [P, Hkv, d]."""
        need = sorted({p for lc in lists.values() for sel in lc.values() for p in sel})
        path = tempfile.mkdtemp(prefix="oracle_pages_")
        np.save(os.path.join(path, "idx.npy"), np.array(need, np.int64))
        K = np.lib.format.open_memmap(os.path.join(path, "k.npy"), "w+", np.float32,
                                      (len(need), w.P, w.Hkv, w.d))
        V = np.lib.format.open_memmap(os.path.join(path, "v.npy"), "w+", np.float32,
                                      (len(need), w.P, w.Hkv, w.d))
        for r, p in enumerate(need):
            K[r], V[r] = page_kv(p)
        K.flush(); V.flush()
        del K, V
        return path

    def _sparse_tasks(self, w, lists, want_of, page_kv):
        path = self._share_pages(w, lists, page_kv)
        tasks = []
        g, P = w.g, w.P
        for c in sorted(lists):
            s, e = w.chunk_range(c)
            q_all, do_all = synth.chunk_q(w, c), synth.chunk_do(w, c)
            for (i, kv), sel in sorted(lists[c].items()):
                want = want_of(kv, sel)
                if want:
                    r0, r1 = i * P, min(e - s, (i + 1) * P)
                    tasks.append((w, c, i, kv, list(sel), want,
                                  np.ascontiguousarray(q_all[r0:r1, kv * g:(kv + 1) * g]),
                                  np.ascontiguousarray(do_all[r0:r1, kv * g:(kv + 1) * g]), path))
        return tasks, path

    def sparse_page_grads(self, w, lists, pages_by_kv, page_kv):
        """dK, dV of pages over page-sparse attention. lists[c][(i, kv)] is the
        ascending selection of query page i of chunk c for KV head kv (checked
        against the oracle's selection by the caller); pages_by_kv[kv] lists
        the pages wanted for that head; page_kv(p) gives a page's K and V
        [P, Hkv, d]. Returns ({(page, kv): (dk, dv)}, number of query pages
        involved), each [P, d] fp64, summed over every query page that
        selected the page."""
        tasks, path = self._sparse_tasks(
            w, lists, lambda kv, sel: [p for p in pages_by_kv.get(kv, ()) if p in sel], page_kv)
        acc = {(p, kv): (np.zeros((w.P, w.d)), np.zeros((w.P, w.d)))
               for kv, ps in pages_by_kv.items() for p in ps}
        try:
            for (_, _, kv, _, _, _, out) in _each(self.pool.imap_unordered(
                    _sparse_qpage_task, tasks), len(tasks), self.timeout_s):
                for p, (dk, dv) in out.items():
                    acc[(p, kv)][0][: dk.shape[0]] += dk
                    acc[(p, kv)][1][: dv.shape[0]] += dv
        finally:
            shutil.rmtree(path, ignore_errors=True)
        return acc, len(tasks)

    def sparse_full(self, w, lists, page_kv):
        """The whole page-sparse sweep given every chunk's selections
        (lists[c][(i, kv)], checked against the oracle's by the caller):
        per-chunk O, LSE, dQ and the final dK, dV [N, Hkv, d] summed over
        every query page that selected each page."""
        o = [np.zeros((e - s, w.Hq, w.d)) for s, e in map(w.chunk_range, range(w.n_chunks))]
        lse = [np.zeros((w.Hq, x.shape[0])) for x in o]
        dq = [np.zeros_like(x) for x in o]
        dk = np.zeros((w.N, w.Hkv, w.d))
        dv = np.zeros_like(dk)
        tasks, path = self._sparse_tasks(w, lists, lambda kv, sel: list(sel), page_kv)
        g, P = w.g, w.P
        try:
            for (c, i, kv, o_, l_, dq_, out) in _each(self.pool.imap_unordered(
                    _sparse_qpage_task, tasks), len(tasks), self.timeout_s):
                r0, r1 = i * P, i * P + o_.shape[0]
                o[c][r0:r1, kv * g:(kv + 1) * g] = o_
                lse[c][kv * g:(kv + 1) * g, r0:r1] = l_
                dq[c][r0:r1, kv * g:(kv + 1) * g] = dq_
                for p, (a, b) in out.items():
                    dk[p * P: p * P + a.shape[0], kv] += a
                    dv[p * P: p * P + b.shape[0], kv] += b
        finally:
            shutil.rmtree(path, ignore_errors=True)
        return dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
