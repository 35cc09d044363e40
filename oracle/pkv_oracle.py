"""CPU oracle for paged chunk attention (fp64, numpy) -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import or run this module. The library and its Python binding never do;
they share no code with it. Inputs come from the seeded generators in
``paged_kv_chunk_chunked_gb300.synth`` (passed in as arrays), never from the CUDA
path.

What it computes, with the passage each function follows. The source is
"Out of the Memory Barrier: A Highly Memory Efficient Training System for LLMs
with Million-Token Contexts" (OOMB), read from five web summaries of it:

* Chunk-recurrent processing: the sequence is split into chunks processed one
  after another; every chunk's queries attend to all earlier keys plus the
  chunk's own (gist.science/de §2.A; gist.science/ja §2.1; sciencestack.ai
  abstract and Fig. 1 caption).
* Paged KV cache *and* paged KV gradients: keys/values live in fixed-size pages
  reached through a block table; dK/dV are accumulated in place into gradient
  pages (gist.science/de §2.B "Paged Memory Management"; gist.science/fr
  "Résumé technique" §2.B; sciencestack.ai Fig. 3 caption).
* The kernels compute exact causal softmax attention on the visible keys (the
  pages name FlashAttention as the dense baseline, gist.science/de §4), so the
  forward and backward here are that plain definition written out.
* Page-level sparse attention: a representative vector per page, the top-K
  pages per query page (gist.science/de §2.D; gist.science/nl "Pagina-niveau
  Sparse Attention"; sciencestack.ai Fig. 5 caption).

Readings where the pages are silent (each is listed with its reason in the
repository's design notes):
  R1 softmax scale s = 1/sqrt(d);  R2 LSE is the natural log of the sum of
  exp of the *scaled* logits;  R3 query head h reads KV head floor(h/g);
  R4 backward runs chunks in reverse;  R6 representative = fp32 mean key of a
  page, page query = mean over the query page's tokens and the g heads of a
  KV group;  R7 one selection per (query page, KV head);  R8 sink = pages
  [0, n_sink), local = the n_local pages ending at the query page, candidates =
  every page in between;  R13 score ties go to the lower page index;
  R16 local attention layers are page-granular: the query page, the n_local - 1
  pages before it and the sink pages.

Every function here is pinned by tests in ``tests/test_oracle_*.py`` against
something other than itself (library attention, finite differences, closed
forms, invariants, brute force):
  attention_forward / attention_backward / full_causal_attention -- torch SDPA
      and autograd in fp64, finite differences, closed forms, shift invariance,
      sum_j dK_j = 0 and sum_j dV_j = sum_i dO_i, a hand-worked example;
  chunk_recurrent_step, logical_rows, scatter_rows -- equal one-shot attention
      over random shapes and permuted tables; scatter-add equals contiguous sums;
  page_representatives, query_page_means, select_pages, chunk_selection --
      constructed means, brute-force ranking, ties, a planted page, K >= every
      candidate equals dense;
  local_pages, chunk_local_selection -- closed-form counts, the set definition,
      K = 0 selection, blockwise library attention for one local page;
  attention_block -- torch autograd of the same block in fp64.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

F64 = np.float64


# --------------------------------------------------------------------------- paging

def softmax_scale(d: int) -> float:
    """R1: the scale applied to q.k before the softmax."""
    return 1.0 / math.sqrt(d)


def logical_rows(pool: np.ndarray, block_table: np.ndarray, length: int,
                 page_size: int) -> np.ndarray:
    """Keys (or values, or grads) of positions 0..length-1 in logical order.

    pool is [n_phys, Hkv, P, d]; position j lives in physical page
    block_table[j // P], row j % P (paged KV cache, gist.science/de §2.B)."""
    j = np.arange(length)
    return pool[np.asarray(block_table)[j // page_size], :, j % page_size, :]


def scatter_rows(pool: np.ndarray, block_table: np.ndarray, start: int,
                 rows: np.ndarray, page_size: int, accumulate: bool = False) -> None:
    """Write (or add) rows [n, Hkv, d] for positions start..start+n-1 into pages."""
    j = start + np.arange(rows.shape[0])
    pp = np.asarray(block_table)[j // page_size]
    if accumulate:
        np.add.at(pool, (pp, slice(None), j % page_size, slice(None)), rows)
    else:
        pool[pp, :, j % page_size, :] = rows


# --------------------------------------------------------------------------- dense attention

def _visible_mask(q_pos: np.ndarray, L: int, page_size: int,
                  page_allowed: Optional[np.ndarray], kv: int,
                  q_start: int) -> np.ndarray:
    """[n, L] bool: key j visible to query i.

    Causal: j <= i. With page_allowed ([n_qp, Hkv, n_pages] bool, query pages
    counted from q_start), key j is also required to lie in a page selected for
    the query's page and this KV head."""
    key_pos = np.arange(L)
    mask = key_pos[None, :] <= q_pos[:, None]
    if page_allowed is not None:
        qp = (q_pos - q_start) // page_size
        mask &= page_allowed[qp, kv][:, key_pos // page_size]
    return mask


def attention_forward(q: np.ndarray, k: np.ndarray, v: np.ndarray, q_start: int,
                      page_size: int = 1, page_allowed: Optional[np.ndarray] = None,
                      block: int = 512):
    """Causal GQA attention of one query chunk against keys 0..L-1.

    q [n, Hq, d] holds queries at global positions q_start..q_start+n-1;
    k, v [L, Hkv, d] are all keys/values in logical order. For query i and
    head h (KV head floor(h/g), R3):
        S_ij  = s * q_i . k_j            for visible j (j <= i, R1)
        LSE_i = m_i + ln sum_j exp(S_ij - m_i),  m_i = max_j S_ij   (R2)
        O_i   = sum_j exp(S_ij - LSE_i) v_j
    Returns O [n, Hq, d] and LSE [Hq, n], fp64. ``block`` only bounds memory."""
    q = np.asarray(q, F64); k = np.asarray(k, F64); v = np.asarray(v, F64)
    n, Hq, d = q.shape
    L, Hkv, _ = k.shape
    g = Hq // Hkv
    s = softmax_scale(d)
    o = np.zeros((n, Hq, d), F64)
    lse = np.zeros((Hq, n), F64)
    for h in range(Hq):
        kv = h // g
        for r0 in range(0, n, block):
            r1 = min(n, r0 + block)
            q_pos = q_start + np.arange(r0, r1)
            S = s * (q[r0:r1, h, :] @ k[:, kv, :].T)
            S = np.where(_visible_mask(q_pos, L, page_size, page_allowed, kv, q_start),
                         S, -np.inf)
            m = S.max(axis=1)
            l = m + np.log(np.exp(S - m[:, None]).sum(axis=1))
            Pm = np.exp(S - l[:, None])
            o[r0:r1, h, :] = Pm @ v[:, kv, :]
            lse[h, r0:r1] = l
    return o, lse


def attention_backward(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray,
                       do: np.ndarray, lse: np.ndarray, q_start: int,
                       page_size: int = 1, page_allowed: Optional[np.ndarray] = None,
                       block: int = 512):
    """Gradients of L = sum(O * dO) for the chunk of ``attention_forward``.

    The backward recomputes P from the saved LSE instead of storing it
    (activation recomputation, gist.science/de §2.A):
        D_i   = sum_d dO_i * O_i
        P_ij  = exp(S_ij - LSE_i)
        dV_j += sum_{h in group, i} P_ij dO_i
        dP_ij = dO_i . v_j
        dS_ij = P_ij (dP_ij - D_i)
        dQ_i  = s sum_j dS_ij k_j
        dK_j += s sum_{h in group, i} dS_ij q_i
    Returns dQ [n, Hq, d] and this chunk's dK, dV [L, Hkv, d], fp64."""
    q = np.asarray(q, F64); k = np.asarray(k, F64); v = np.asarray(v, F64)
    o = np.asarray(o, F64); do = np.asarray(do, F64); lse = np.asarray(lse, F64)
    n, Hq, d = q.shape
    L, Hkv, _ = k.shape
    g = Hq // Hkv
    s = softmax_scale(d)
    D = (do * o).sum(axis=2)                       # [n, Hq]
    dq = np.zeros((n, Hq, d), F64)
    dk = np.zeros((L, Hkv, d), F64)
    dv = np.zeros((L, Hkv, d), F64)
    for h in range(Hq):
        kv = h // g
        for r0 in range(0, n, block):
            r1 = min(n, r0 + block)
            q_pos = q_start + np.arange(r0, r1)
            mask = _visible_mask(q_pos, L, page_size, page_allowed, kv, q_start)
            S = s * (q[r0:r1, h, :] @ k[:, kv, :].T)
            Pm = np.where(mask, np.exp(S - lse[h, r0:r1, None]), 0.0)
            dv[:, kv, :] += Pm.T @ do[r0:r1, h, :]
            dP = do[r0:r1, h, :] @ v[:, kv, :].T
            dS = Pm * (dP - D[r0:r1, h, None])
            dq[r0:r1, h, :] = s * (dS @ k[:, kv, :])
            dk[:, kv, :] += s * (dS.T @ q[r0:r1, h, :])
    return dq, dk, dv


def full_causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray):
    """Whole-sequence causal attention with no paging and no chunks.

    Materialises the full [N, N] logit matrix per head. Used to pin the paged,
    chunk-recurrent path: both must agree (chunk recurrence is exact)."""
    q = np.asarray(q, F64); k = np.asarray(k, F64); v = np.asarray(v, F64)
    N, Hq, d = q.shape
    g = Hq // k.shape[1]
    s = softmax_scale(d)
    o = np.zeros_like(q)
    lse = np.zeros((Hq, N), F64)
    tri = np.tril(np.ones((N, N), bool))
    for h in range(Hq):
        S = np.where(tri, s * q[:, h, :] @ k[:, h // g, :].T, -np.inf)
        m = S.max(axis=1, keepdims=True)
        e = np.exp(S - m)
        z = e.sum(axis=1, keepdims=True)
        o[:, h, :] = (e / z) @ v[:, h // g, :]
        lse[h] = (m + np.log(z))[:, 0]
    return o, lse


# --------------------------------------------------------------------------- attention block

def attention_block(x: np.ndarray, wq: np.ndarray, wk: np.ndarray, wv: np.ndarray,
                    wo: np.ndarray, dy: np.ndarray, n_q_heads: int, n_kv_heads: int):
    """One attention block over the whole sequence, forward and backward.

    y = x + A wo with A = causal GQA attention(x wq, x wk, x wv) (heads laid
    out [.., H, d] in the projection outputs); the loss is sum(y * dy). This is
    the layer that chunk-recurrent training processes chunk by chunk while
    recomputing activations (gist.science/de §2.A; sciencestack.ai Fig. 1
    caption); chunking and recomputation do not change it, so the whole-sequence
    definition is the reference. Returns y and the gradients of x, wq, wk, wv,
    wo (fp64)."""
    x = np.asarray(x, F64); dy = np.asarray(dy, F64)
    wq, wk, wv, wo = (np.asarray(t, F64) for t in (wq, wk, wv, wo))
    N = x.shape[0]
    d = wq.shape[1] // n_q_heads
    q = (x @ wq).reshape(N, n_q_heads, d)
    k = (x @ wk).reshape(N, n_kv_heads, d)
    v = (x @ wv).reshape(N, n_kv_heads, d)
    o, lse = attention_forward(q, k, v, 0)
    a = o.reshape(N, n_q_heads * d)
    y = x + a @ wo
    da = dy @ wo.T
    dwo = a.T @ dy
    dq, dk, dv = attention_backward(q, k, v, o, da.reshape(N, n_q_heads, d), lse, 0)
    dq, dk, dv = (t.reshape(N, -1) for t in (dq, dk, dv))
    dx = dy + dq @ wq.T + dk @ wk.T + dv @ wv.T
    return y, dict(x=dx, wq=x.T @ dq, wk=x.T @ dk, wv=x.T @ dv, wo=dwo)


# --------------------------------------------------------------------------- page selection

def page_representatives(k_logical: np.ndarray, page_size: int) -> np.ndarray:
    """R6: representative of logical page p and KV head h = mean of its stored keys.

    k_logical [L, Hkv, d] -> [ceil(L/P), Hkv, d]; a partial last page averages
    only the rows it holds."""
    k = np.asarray(k_logical, F64)
    L, Hkv, d = k.shape
    n_pg = (L + page_size - 1) // page_size
    rep = np.zeros((n_pg, Hkv, d), F64)
    for p in range(n_pg):
        rep[p] = k[p * page_size: min(L, (p + 1) * page_size)].mean(axis=0)
    return rep


def query_page_means(q_chunk: np.ndarray, page_size: int, n_kv_heads: int) -> np.ndarray:
    """R6: mean query of each query page and KV group.

    q_chunk [n, Hq, d] -> [ceil(n/P), Hkv, d]: the mean over the page's tokens
    and over the g query heads that read KV head h."""
    q = np.asarray(q_chunk, F64)
    n, Hq, d = q.shape
    g = Hq // n_kv_heads
    n_qp = (n + page_size - 1) // page_size
    out = np.zeros((n_qp, n_kv_heads, d), F64)
    for qp in range(n_qp):
        blk = q[qp * page_size: min(n, (qp + 1) * page_size)]
        for h in range(n_kv_heads):
            out[qp, h] = blk[:, h * g:(h + 1) * g, :].mean(axis=(0, 1))
    return out


def select_pages(qbar: np.ndarray, rep: np.ndarray, qp: int, K: int, n_sink: int,
                 n_local: int) -> list:
    """Visible pages of global query page qp for one KV head (R7, R8, R13).

    qbar [d] is the page query, rep [n_pages>=qp+1, d] the representatives.
    Candidates are pages n_sink .. qp-n_local; each scores qbar . rep[p]
    (unscaled: a positive scale does not change the order). The K best by
    (score descending, page index ascending) are kept, together with the sink
    pages [0, n_sink) and the local pages qp-n_local+1 .. qp. Returns the set
    sorted ascending."""
    keep = set(range(0, min(n_sink, qp + 1)))
    keep |= set(range(max(0, qp - n_local + 1), qp + 1))
    cand = np.arange(n_sink, qp - n_local + 1)
    if cand.size:
        score = np.asarray(rep, F64)[cand] @ np.asarray(qbar, F64)
        order = np.lexsort((cand, -score))          # primary: -score; ties: page index
        keep |= set(int(p) for p in cand[order[:K]])
    return sorted(keep)


def chunk_selection(q_chunk: np.ndarray, q_start: int, k_logical: np.ndarray,
                    page_size: int, K: int, n_sink: int, n_local: int):
    """Selected pages for every query page of a chunk and every KV head.

    Returns (lists, padded): lists[qp][h] is the sorted page list of the chunk's
    query page qp; padded is int32 [n_qp, Hkv, K+n_sink+n_local] with -1 after
    the list. Representatives come from all keys up to the end of the chunk."""
    n, Hq, d = q_chunk.shape
    Hkv = k_logical.shape[1]
    if q_start % page_size:
        raise ValueError("chunks start on page boundaries")
    qbar = query_page_means(q_chunk, page_size, Hkv)
    rep = page_representatives(k_logical[: q_start + n], page_size)
    qp0 = q_start // page_size
    kmax = K + n_sink + n_local
    lists, padded = [], np.full((qbar.shape[0], Hkv, kmax), -1, np.int32)
    for i in range(qbar.shape[0]):
        row = []
        for h in range(Hkv):
            sel = select_pages(qbar[i, h], rep[:, h, :], qp0 + i, K, n_sink, n_local)
            padded[i, h, :len(sel)] = sel
            row.append(sel)
        lists.append(row)
    return lists, padded


def local_pages(qp: int, n_sink: int, n_local: int) -> list:
    """Visible pages of global query page qp in a local attention layer.

    The pages use local attention layers, not a scorer, for natively sparse
    models (gist.science/nl "Pagina-niveau Sparse Attention"). Read at page
    granularity (R16): the query page itself (causal inside), the n_local - 1
    pages before it, and the sink pages [0, n_sink); sorted ascending."""
    keep = set(range(0, min(n_sink, qp + 1)))
    keep |= set(range(max(0, qp - n_local + 1), qp + 1))
    return sorted(keep)


def chunk_local_selection(q_start: int, n_q: int, n_kv_heads: int, page_size: int,
                          n_sink: int, n_local: int):
    """local_pages for every query page of a chunk, the same list for every KV
    head. Returns (lists, padded) as chunk_selection does, padded being int32
    [n_qp, Hkv, n_sink + n_local]."""
    if q_start % page_size:
        raise ValueError("chunks start on page boundaries")
    n_qp = (n_q + page_size - 1) // page_size
    qp0 = q_start // page_size
    padded = np.full((n_qp, n_kv_heads, n_sink + n_local), -1, np.int32)
    lists = []
    for i in range(n_qp):
        sel = local_pages(qp0 + i, n_sink, n_local)
        padded[i, :, :len(sel)] = sel
        lists.append([sel] * n_kv_heads)
    return lists, padded


def page_allowed_from_lists(lists: Sequence, n_pages: int) -> np.ndarray:
    """[n_qp, Hkv, n_pages] bool mask from per-(query page, KV head) page lists."""
    n_qp, Hkv = len(lists), len(lists[0])
    out = np.zeros((n_qp, Hkv, n_pages), bool)
    for i in range(n_qp):
        for h in range(Hkv):
            out[i, h, lists[i][h]] = True
    return out


# --------------------------------------------------------------------------- chunk recurrence

def chunk_recurrent_step(qs, ks, vs, dos, block_table, page_size: int, n_phys: int,
                         topk: Optional[tuple] = None, local: Optional[tuple] = None):
    """One training step of one attention layer, chunk by chunk (gist.science/de §2.A).

    qs/ks/vs/dos are lists of per-chunk arrays. Forward: for c = 0, 1, ...
    append chunk c's K/V into the paged pools, then attend its queries to every
    key so far. Backward (R4: reverse chunk order): recompute from the saved
    O/LSE, write dQ and add dK/dV into the paged gradient pools in place.
    With ``topk`` = (K, n_sink, n_local) each chunk attends only to the pages
    selected for its query pages; with ``local`` = (n_sink, n_local) only to
    its local pages (local_pages). Returns a dict of per-chunk outputs and the
    final pools (physical layout [n_phys, Hkv, P, d])."""
    Hkv, d = ks[0].shape[1], ks[0].shape[2]
    P = page_size
    kpool = np.zeros((n_phys, Hkv, P, d), F64)
    vpool = np.zeros_like(kpool)
    dkpool = np.zeros_like(kpool)
    dvpool = np.zeros_like(kpool)
    starts = np.cumsum([0] + [x.shape[0] for x in qs])
    outs, lses, masks, sels = [], [], [], []
    for c in range(len(qs)):
        st = int(starts[c])
        scatter_rows(kpool, block_table, st, np.asarray(ks[c], F64), P)
        scatter_rows(vpool, block_table, st, np.asarray(vs[c], F64), P)
        L = st + qs[c].shape[0]
        k_log = logical_rows(kpool, block_table, L, P)
        v_log = logical_rows(vpool, block_table, L, P)
        allowed = None
        if topk is not None:
            lists, padded = chunk_selection(qs[c], st, k_log, P, *topk)
            allowed = page_allowed_from_lists(lists, (L + P - 1) // P)
            sels.append(padded)
        elif local is not None:
            lists, padded = chunk_local_selection(st, qs[c].shape[0], Hkv, P, *local)
            allowed = page_allowed_from_lists(lists, (L + P - 1) // P)
            sels.append(padded)
        o, lse = attention_forward(qs[c], k_log, v_log, st, P, allowed)
        outs.append(o); lses.append(lse); masks.append(allowed)
    dqs = [None] * len(qs)
    for c in reversed(range(len(qs))):
        st = int(starts[c])
        L = st + qs[c].shape[0]
        k_log = logical_rows(kpool, block_table, L, P)
        v_log = logical_rows(vpool, block_table, L, P)
        dq, dk, dv = attention_backward(qs[c], k_log, v_log, outs[c], dos[c], lses[c], st,
                                        P, masks[c])
        dqs[c] = dq
        scatter_rows(dkpool, block_table, 0, dk, P, accumulate=True)
        scatter_rows(dvpool, block_table, 0, dv, P, accumulate=True)
    return dict(o=outs, lse=lses, dq=dqs, kpool=kpool, vpool=vpool, dkpool=dkpool,
                dvpool=dvpool, sel=sels)
