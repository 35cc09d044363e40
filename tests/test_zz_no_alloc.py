"""pkv_chunk_attn_bwd_noalloc against pkv_chunk_attn_bwd, through the C ABI.

The no-allocation variant exists for callers that cannot let the library
allocate device memory when the backward runs: a fixed memory budget, an
allocator that owns all device memory, code that must not synchronize the
device, or a loop that forbids allocation after start-up. It keeps its
per-row scratch in one fixed array of the library's device image instead of a
cudaMalloc'd buffer. Its results must equal the allocating entry point's, call
after call (the array keeps the previous call's contents).

The file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import numpy as np
import pytest
import torch

from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.sweep import ChunkSweep, to_numpy

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


CASES = {
    # tensor-core kernels: bf16, page 128, d 128, permuted block table
    "bf16_tensor_cores": synth.workload("qwen7b_dense_32k", N=768, C=256, Hq=4, Hkv=2,
                                        table="perm", extra_pages=2),
    # CUDA-core kernels: fp32, page 16, d 64
    "f32_cuda_cores": synth.workload("tiny_dense_f32"),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_noalloc_backward_matches_allocating_backward(case):
    w = CASES[case]
    sw = ChunkSweep(w).load_inputs()
    try:
        sw.reset()
        for c in range(w.n_chunks):
            sw.forward(c)
        for c in reversed(range(w.n_chunks)):
            sw.backward(c)
        ref = sw.gather()
        dq_ref = [to_numpy(x) for x in sw.dq]
        dk_ref, dv_ref = to_numpy(ref["dk"]), to_numpy(ref["dv"])
        for call in range(2):                       # two calls in a row share the array
            B.pkv_grad_zero(sw.seq)
            dq = [torch.full_like(x, float("nan")) for x in sw.dq]
            for c in reversed(range(w.n_chunks)):
                s, e = w.chunk_range(c)
                B.pkv_chunk_attn_bwd_noalloc(sw.seq, sw.q[c], sw.o[c], sw.do[c], sw.lse[c], s,
                                             e - s, dq[c])
            got = sw.gather()
            B.pkv_check(sw.pool)
            tol = REL_TOL[w.dtype]
            for c in range(w.n_chunks):
                assert _rel(to_numpy(dq[c]), dq_ref[c]) <= tol, (call, c)
            assert _rel(to_numpy(got["dk"]), dk_ref) <= tol, call
            assert _rel(to_numpy(got["dv"]), dv_ref) <= tol, call
    finally:
        sw.close()


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
