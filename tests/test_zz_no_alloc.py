"""pkv_chunk_attn_bwd_noalloc against the oracle, through the C ABI.

Who needs it: a caller that cannot let the library allocate device memory
while the backward runs. Examples are a trainer under a fixed memory budget,
a framework whose caching allocator owns all device memory (a cudaMalloc
behind its back can fail or fragment it), code that must not synchronize the
device (cudaMalloc and cudaFree can), and loops that forbid allocation after
start-up. The variant keeps its per-row scratch in one fixed array of the
library's device image instead of a cudaMalloc'd buffer.

Checked here: dQ and the accumulated dK/dV pages equal the oracle's
chunk-recurrent backward (relative Frobenius 2e-2 for bf16, 1e-4 for fp32),
on two backward sweeps in a row (the array keeps the previous call's
contents); with a page selection made by pkv_page_topk; and on a pinned-host
pool, where the gradient write-back runs on a side stream right after the
call and must wait for it (the call marks the sequence as used, as
pkv_chunk_attn_bwd does).

The file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
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

# The parity tolerances used throughout the GPU tests (relative Frobenius).
REL_TOL = {"bf16": 2e-2, "f32": 1e-4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def _oracle(w):
    n = w.n_chunks
    qs = [synth.chunk_q(w, c) for c in range(n)]
    ks = [synth.chunk_k(w, c) for c in range(n)]
    vs = [synth.chunk_v(w, c) for c in range(n)]
    dos = [synth.chunk_do(w, c) for c in range(n)]
    bt = synth.block_table(w)
    ref = oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys, topk=w.topk)
    return ref, bt


CASES = {
    # tensor-core kernels: bf16, page 128, d 128, 7:1 grouping, permuted block table
    "bf16_tensor_cores": synth.workload("qwen7b_dense_32k", N=768, C=256, Hq=14, Hkv=2,
                                        table="perm", extra_pages=2),
    # CUDA-core kernels: fp32, page 16, d 64
    "f32_cuda_cores": synth.workload("tiny_dense_f32"),
    # page-sparse: the selection comes from pkv_page_topk
    "bf16_sparse_topk": synth.workload("qwen7b_sparse_256k", N=2048, C=1024, Hq=4, Hkv=2,
                                       extra_pages=3, topk=(3, 1, 2)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_backward_matches_oracle(case):
    w = CASES[case]
    ref, bt = _oracle(w)
    tol = REL_TOL[w.dtype]
    dk_ref = oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)
    dv_ref = oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        sels = []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            sel = None
            if w.topk is not None:
                B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
                K, ns, nl = w.topk
                sel = torch.empty(((e - s + w.P - 1) // w.P, w.Hkv, K + ns + nl),
                                  dtype=torch.int32, device="cuda")
                B.pkv_page_topk(sw.seq, sw.q[c], s, e - s, K, ns, nl, sel)
                # clustered keys leave no score ties: the selection is the oracle's
                np.testing.assert_array_equal(sel.cpu().numpy(), ref["sel"][c])
                B.pkv_chunk_attn_fwd(sw.seq, sw.q[c], s, e - s, sw.o[c], sw.lse[c], sel)
            else:
                sw.forward(c)
            sels.append(sel)
        for call in range(2):                       # two sweeps in a row share the array
            B.pkv_grad_zero(sw.seq)
            dq = [torch.full_like(x, float("nan")) for x in sw.dq]
            for c in reversed(range(w.n_chunks)):
                s, e = w.chunk_range(c)
                B.pkv_chunk_attn_bwd_noalloc(sw.seq, sw.q[c], sw.o[c], sw.do[c], sw.lse[c], s,
                                             e - s, dq[c], sels[c])
            got = sw.gather()
            B.pkv_check(sw.pool)
            for c in range(w.n_chunks):
                assert _rel(to_numpy(dq[c]), ref["dq"][c]) <= tol, (call, c)
            assert _rel(to_numpy(got["dk"]), dk_ref) <= tol, call
            assert _rel(to_numpy(got["dv"]), dv_ref) <= tol, call
    finally:
        sw.close()


def test_noalloc_backward_on_pinned_host_pool_orders_the_writeback():
    """Pinned-host pool: per chunk in reverse, stage K/V and gradient pages on a
    side stream, run the no-allocation backward on the main stream, and queue
    the gradient write-back on the side stream at once (no host wait between).
    The written-back host gradient pages must equal the oracle's."""
    w = synth.workload("qwen7b_sparse_1m_offload", N=3072, C=1024, Hq=4, Hkv=2,
                       extra_pages=5, topk=(3, 1, 2))
    ref, bt = _oracle(w)
    K, ns, nl = w.topk
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    try:
        seq = B.pkv_seq_create(pool)
        B.pkv_set_block_table(seq, bt)
        dev = lambda x: to_device(x, "bf16")
        q = [dev(synth.chunk_q(w, c)) for c in range(w.n_chunks)]
        do = [dev(synth.chunk_do(w, c)) for c in range(w.n_chunks)]
        o, lse, dq, sels = [], [], [], []
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(seq, dev(synth.chunk_k(w, c)), dev(synth.chunk_v(w, c)), e - s, main)
            sel = torch.empty(((e - s) // w.P, w.Hkv, K + ns + nl), dtype=torch.int32,
                              device="cuda")
            B.pkv_page_topk(seq, q[c], s, e - s, K, ns, nl, sel, None, main)
            sels.append(sel)
            o.append(torch.empty_like(q[c]))
            lse.append(torch.empty((w.Hq, e - s), dtype=torch.float32, device="cuda"))
            dq.append(torch.empty_like(q[c]))
            B.pkv_prefetch(seq, sel, sel.numel(), B.PKV_STAGE_KV, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_fwd(seq, q[c], s, e - s, o[c], lse[c], sel, main)
        for c in reversed(range(w.n_chunks)):
            s, e = w.chunk_range(c)
            B.pkv_prefetch(seq, sels[c], sels[c].numel(), B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
            B.pkv_wait(seq, main, 0)
            B.pkv_chunk_attn_bwd_noalloc(seq, q[c], o[c], do[c], lse[c], s, e - s, dq[c],
                                         sels[c], main)
            B.pkv_writeback_grads(seq, side)
        B.pkv_wait(seq, main, 10_000_000)
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        B.pkv_gather(seq, None, None, dk, dv, None, main)
        torch.cuda.synchronize()
        B.pkv_check(pool)
        for c in range(w.n_chunks):
            np.testing.assert_array_equal(sels[c].cpu().numpy(), ref["sel"][c])
            assert _rel(to_numpy(dq[c]), ref["dq"][c]) <= 2e-2, c
        assert _rel(to_numpy(dk), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)) <= 2e-2
        assert _rel(to_numpy(dv), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)) <= 2e-2
    finally:
        B.pkv_pool_destroy(pool)


def test_noalloc_rejects_chunks_beyond_the_fixed_scratch():
    # 256 query heads x 1040 queries = 266240 floats > 262144: rejected before any launch.
    pool = B.pkv_pool_create(16, 1, 256, 64, B.PKV_F32, 80)
    try:
        seq = B.pkv_seq_create(pool)
        kv = torch.zeros((1040, 1, 64), dtype=torch.float32, device="cuda")
        B.pkv_append(seq, kv, kv, 1040)
        q = torch.zeros((1040, 256, 64), dtype=torch.float32, device="cuda")
        lse = torch.zeros((256, 1040), dtype=torch.float32, device="cuda")
        with pytest.raises(B.PkvError) as e:
            B.pkv_chunk_attn_bwd_noalloc(seq, q, q, q, lse, 0, 1040, q)
        assert e.value.status == B.PKV_ERR_INVALID
        assert "exceeds the fixed scratch" in str(e.value)
        torch.cuda.synchronize()
        B.pkv_check(pool)
    finally:
        B.pkv_pool_destroy(pool)


def test_noalloc_scan_fallback_equals_the_mask_path_bit_for_bit():
    """With a selection, the dK/dV kernel reads each page's query tiles from
    per-(page, KV head) query-page masks; when those masks do not fit the fixed
    scratch the no-allocation backward lets the kernel scan the selection
    instead. Both give the same tile lists in the same order, and every
    (page, KV head) block of the pool gets one addition per call, so dQ, dK
    and dV must match pkv_chunk_attn_bwd (the oracle-checked mask path) bit
    for bit. Sizes: 28 query heads x 9344 queries (73 query pages) after 16384
    earlier tokens, local lists of 2 pages: D and the page list fit the
    262144 floats (261834), D, list and masks do not (265051)."""
    w = synth.workload("qwen7b_local_256k", N=16384 + 9344, C=16384)
    s, e = w.chunk_range(1)
    n_q, n_qp, n_key_pages, kmax = e - s, (e - s + w.P - 1) // w.P, (e + w.P - 1) // w.P, 2
    n_d = w.Hq * n_q
    n_list = 1 + min(n_key_pages, n_qp * w.Hkv * kmax)
    n_mask = 1 + 2 * n_key_pages * w.Hkv * ((n_qp + 63) // 64)
    assert n_d + n_list <= 262144 < n_d + n_list + n_mask
    outs = []
    for noalloc in (False, True):
        sw = ChunkSweep(w).load_inputs()
        try:
            sw.reset()
            for c in range(w.n_chunks):
                a, b = w.chunk_range(c)
                B.pkv_append(sw.seq, sw.k[c], sw.v[c], b - a)
            sel = torch.empty((n_qp, w.Hkv, kmax), dtype=torch.int32, device="cuda")
            B.pkv_page_local(sw.seq, s, n_q, 0, 2, sel)
            B.pkv_chunk_attn_fwd(sw.seq, sw.q[1], s, n_q, sw.o[1], sw.lse[1], sel)
            B.pkv_grad_zero(sw.seq)
            bwd = B.pkv_chunk_attn_bwd_noalloc if noalloc else B.pkv_chunk_attn_bwd
            bwd(sw.seq, sw.q[1], sw.o[1], sw.do[1], sw.lse[1], s, n_q, sw.dq[1], sel)
            g = sw.gather()
            B.pkv_check(sw.pool)
            outs.append((sw.dq[1].cpu(), g["dk"].cpu(), g["dv"].cpu()))
        finally:
            sw.close()
    for x, y in zip(outs[0], outs[1]):
        assert torch.equal(x, y)
    assert float(outs[0][1].abs().sum()) > 0.0                      # gradients were added
