"""GPU parity: libpkv (through its C ABI) against the CPU oracle, element by element.

Tolerances (stated for this path): O and LSE max-abs <= 1e-2 with bf16 inputs,
1e-4 with fp32; dQ, dK, dV relative Frobenius <= 2e-2 (bf16), 1e-4 (fp32).
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

TOL = {"bf16": (1e-2, 2e-2), "f32": (1e-4, 1e-4)}


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
    return oracle.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys), bt


def _sweep_vs_oracle(w, flags=0):
    sw = ChunkSweep(w, flags=flags).load_inputs()
    try:
        sw.run()
        B.pkv_check(sw.pool)
        g = sw.gather()
        ref, bt = _oracle(w)
        tol_abs, tol_rel = TOL[w.dtype]
        o = np.concatenate([to_numpy(x) for x in sw.o])
        lse = np.concatenate([to_numpy(x) for x in sw.lse], axis=1)
        dq = np.concatenate([to_numpy(x) for x in sw.dq])
        err = dict(
            o=float(np.abs(o - np.concatenate(ref["o"])).max()),
            lse=float(np.abs(lse - np.concatenate(ref["lse"], axis=1)).max()),
            dq=_rel(dq, np.concatenate(ref["dq"])),
            dk=_rel(to_numpy(g["dk"]), oracle.logical_rows(ref["dkpool"], bt, w.N, w.P)),
            dv=_rel(to_numpy(g["dv"]), oracle.logical_rows(ref["dvpool"], bt, w.N, w.P)),
        )
        assert err["o"] <= tol_abs and err["lse"] <= tol_abs, err
        assert err["dq"] <= tol_rel and err["dk"] <= tol_rel and err["dv"] <= tol_rel, err
        # the pool holds exactly the appended keys/values, in logical order
        np.testing.assert_array_equal(to_numpy(g["k"]), oracle.logical_rows(ref["kpool"], bt, w.N, w.P))
        np.testing.assert_array_equal(to_numpy(g["v"]), oracle.logical_rows(ref["vpool"], bt, w.N, w.P))
        rep_ref = oracle.page_representatives(oracle.logical_rows(ref["kpool"], bt, w.N, w.P), w.P)
        np.testing.assert_allclose(to_numpy(g["rep"]), rep_ref, rtol=0, atol=1e-5)
        return err, sw
    finally:
        sw.close()


def test_tiny_dense_f32():
    _sweep_vs_oracle(synth.workload("tiny_dense_f32"))


def test_tiny_dense_f32_partial_last_page_and_perm():
    _sweep_vs_oracle(synth.workload("tiny_dense_f32", N=200, table="perm", extra_pages=3))


def test_small_dense_bf16_page16_cuda_cores():
    _sweep_vs_oracle(synth.workload("tiny_dense_f32", dtype="bf16", Hq=4, Hkv=2, N=320, C=96,
                                    table="perm", extra_pages=2, name="bf16_p16"))


@pytest.mark.parametrize("N,C,Hq,Hkv", [(768, 256, 4, 2), (1024, 512, 7, 1), (700, 256, 4, 2)])
def test_dense_bf16_page128_tensor_cores(N, C, Hq, Hkv):
    w = synth.workload("qwen7b_dense_32k", N=N, C=C, Hq=Hq, Hkv=Hkv, table="perm",
                       extra_pages=3, name=f"bf16_p128_{N}_{C}")
    _sweep_vs_oracle(w)


@pytest.mark.parametrize("N,C,Hq,Hkv", [(768, 256, 8, 1), (700, 256, 4, 2), (1024, 512, 16, 2)])
def test_dense_bf16_page128_head_dim_64_tensor_cores(N, C, Hq, Hkv):
    """Head dimension 64 (the natively sparse models' geometry) on the
    tensor-core kernels: several tiles, a ragged last chunk, 8:1 and 2:1 groups."""
    w = synth.workload("qwen7b_dense_32k", N=N, C=C, Hq=Hq, Hkv=Hkv, d=64, table="perm",
                       extra_pages=3, name=f"bf16_p128_d64_{N}_{C}")
    _sweep_vs_oracle(w)


def test_dense_bf16_page128_cuda_cores_flag():
    w = synth.workload("qwen7b_dense_32k", N=512, C=256, Hq=4, Hkv=2, name="bf16_p128_simt")
    _sweep_vs_oracle(w, flags=B.PKV_FLAG_SIMT_ONLY)


def test_permuted_block_table_gives_identical_results():
    base = dict(N=640, C=256, Hq=4, Hkv=2, extra_pages=4)
    outs = []
    for table in ("identity", "perm"):
        w = synth.workload("qwen7b_dense_32k", table=table, **base)
        sw = ChunkSweep(w).load_inputs()
        sw.run()
        g = sw.gather()
        outs.append(([to_numpy(x) for x in sw.o], [to_numpy(x) for x in sw.lse], to_numpy(g["dv"])))
        sw.close()
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("key,N", [("tiny_dense_f32", 250), ("qwen7b_dense_128k_perm", 16384 + 200),
                                   ("qwen7b_dense_32k", 32768)])
def test_grad_accumulate_bit_exact(key, N):
    """pkv_grad_accumulate against the oracle's paged scatter-add, bit for bit:
    ragged row ranges (page-crossing, partial last page, one row, NULL dv or dk)
    on identity and permuted block tables, and the whole 32K sequence in the
    launch the benchmark times. Fresh pages start at zero gradient, so the
    oracle starts from a zero float32 pool and repeats the same additions."""
    w = synth.workload(key, N=N)
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        for c in range(w.n_chunks):
            s, e = w.chunk_range(c)
            B.pkv_append(sw.seq, sw.k[c], sw.v[c], e - s)
        P = w.P
        ops = [(0, N, True, True), (37, 3 * P, True, False), (2 * P - 1, 2, True, True),
               (N - 1, 1, False, True), (P, N - P - 3, True, True)]
        pool = {t: np.zeros((w.n_phys, w.Hkv, P, w.d), np.float32) for t in ("dk", "dv")}
        bt = synth.block_table(w)
        for i, (r0, n, with_dk, with_dv) in enumerate(ops):
            dev = {}
            for j, t in enumerate(("dk", "dv")):
                if (with_dk, with_dv)[j]:
                    x = synth.draw_normal(w.seed, "misc", 100 + 2 * i + j, (n, w.Hkv, w.d))
                    oracle.scatter_rows(pool[t], bt, r0, x, P, accumulate=True)
                    dev[t] = torch.from_numpy(x).cuda()
            B.pkv_grad_accumulate(sw.seq, r0, n, dev.get("dk"), dev.get("dv"))
        torch.cuda.synchronize()
        B.pkv_check(sw.pool)
        g = sw.gather()
        for t in ("dk", "dv"):
            np.testing.assert_array_equal(to_numpy(g[t]), oracle.logical_rows(pool[t], bt, N, P))
    finally:
        sw.close()


def test_grad_accumulate_rejects_bad_ranges_and_alignment():
    w = synth.workload("tiny_dense_f32")
    sw = ChunkSweep(w).load_inputs([0])
    try:
        sw.reset()
        B.pkv_append(sw.seq, sw.k[0], sw.v[0], w.C)
        x = torch.zeros((w.C + 1, w.Hkv, w.d), device="cuda")
        for r0, n, buf in [(-1, 4, x), (0, w.C + 1, x), (w.C, 1, x), (0, 4, x.view(-1)[1:])]:
            with pytest.raises(B.PkvError) as e:
                B.pkv_grad_accumulate(sw.seq, r0, n, buf, None)
            assert e.value.status == B.PKV_ERR_INVALID
        B.pkv_grad_accumulate(sw.seq, w.C, 0, x, x)        # empty range: nothing to do
        B.pkv_check(sw.pool)
    finally:
        sw.close()


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
def test_umma_selftest(mode):
    g = torch.Generator().manual_seed(mode)
    a = torch.randn((64, 128) if mode == 2 else (128, 64), generator=g).to(torch.bfloat16)
    b = torch.randn((128, 64) if mode == 0 else (64, 128), generator=g).to(torch.bfloat16)
    d = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    B.pkv_selftest_umma(mode, a.cuda(), b.cuda(), d)
    af, bf = a.double(), b.double()
    ref = af @ bf.T if mode == 0 else (af.T @ bf if mode == 2 else af @ bf)
    np.testing.assert_allclose(d.cpu().double().numpy(), ref.numpy(), rtol=1e-5, atol=1e-4)


def test_host_buffer_sweep_matches_device_sweep():
    """ChunkSweep.run_from_host (inputs and results in pinned host memory,
    copies on side streams overlapped with the kernels) gives the device
    sweep's results: dQ bit for bit, dK/dV up to the order of the gradient
    additions."""
    w = synth.workload("qwen7b_dense_32k", N=1024, C=256, Hq=4, Hkv=2, table="perm", extra_pages=2,
                       name="host_sweep")
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.run()
        ref = sw.gather()
        ref_dq = [to_numpy(x) for x in sw.dq]
        host = {name: [t.cpu().pin_memory() for t in lst]
                for name, lst in (("q", sw.q), ("k", sw.k), ("v", sw.v), ("do", sw.do))}
        for lst in (sw.q, sw.k, sw.v, sw.do, sw.dq):      # the copies must bring the data back
            for t in lst:
                t.zero_()
        dk = torch.empty((w.N, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        dv = torch.empty_like(dk)
        out = {"dq": [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in sw.dq],
               "dk": torch.empty(dk.shape, dtype=torch.float32).pin_memory(),
               "dv": torch.empty(dk.shape, dtype=torch.float32).pin_memory()}
        sw.run_from_host(host, out, dk, dv, torch.cuda.Stream(), torch.cuda.Stream())
        torch.cuda.synchronize()
        B.pkv_check(sw.pool)
        for a, b in zip(out["dq"], ref_dq):
            np.testing.assert_array_equal(a.float().numpy(), b)
        assert _rel(out["dk"].numpy(), to_numpy(ref["dk"])) < 1e-6
        assert _rel(out["dv"].numpy(), to_numpy(ref["dv"])) < 1e-6
    finally:
        sw.close()


def test_bounded_wait_gives_up_reports_and_leaves_the_device_usable():
    """Every kernel wait is bounded. Self-test mode 4 issues no MMA, so its wait
    for the MMA can never succeed: it must give up after its bound (~4 s),
    record the timeout in the error word, free its tensor memory and return.
    The next launch on the same context then works normally."""
    import time
    a = torch.zeros((128, 64), dtype=torch.bfloat16, device="cuda")
    b = torch.zeros((64, 128), dtype=torch.bfloat16, device="cuda")
    d = torch.empty((128, 128), dtype=torch.float32, device="cuda")
    t0 = time.time()
    with pytest.raises(B.PkvError) as e:
        B.pkv_selftest_umma(4, a, b, d)
    assert e.value.status == B.PKV_ERR_DEVICE_FAULT and "device error 1" in str(e.value)
    assert time.time() - t0 < 60
    g = torch.Generator().manual_seed(0)
    a = torch.randn((128, 64), generator=g).to(torch.bfloat16)
    b = torch.randn((128, 64), generator=g).to(torch.bfloat16)
    B.pkv_selftest_umma(0, a.cuda(), b.cuda(), d)
    np.testing.assert_allclose(d.cpu().double().numpy(), (a.double() @ b.double().T).numpy(),
                               rtol=1e-5, atol=1e-4)


def test_host_wait_with_a_deadline_times_out_then_completes():
    """pkv_wait with a deadline polls the staging event and returns
    PKV_ERR_TIMEOUT instead of blocking; without one it orders the streams."""
    w = synth.workload("qwen7b_dense_32k", N=8192, C=8192, Hq=4, Hkv=2, name="wait_deadline")
    pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, B.PKV_BF16, w.n_phys,
                             residency=B.PKV_RES_PINNED_HOST, n_device_slots=w.n_pages)
    try:
        seq = B.pkv_seq_create(pool)
        kv = to_device(synth.chunk_k(w, 0), "bf16")
        B.pkv_append(seq, kv, kv, w.N)
        torch.cuda.synchronize()
        side = torch.cuda.Stream()
        B.pkv_prefetch(seq, None, 0, B.PKV_STAGE_KV | B.PKV_STAGE_GRADS, side)
        with pytest.raises(B.PkvError) as e:
            B.pkv_wait(seq, None, 1)                 # 1 us: the copies take far longer
        assert e.value.status == B.PKV_ERR_TIMEOUT
        B.pkv_wait(seq, None, 0)
        torch.cuda.synchronize()
        B.pkv_check(pool)
    finally:
        B.pkv_pool_destroy(pool)
