"""GPU parity of chunk-recurrent training of one attention block against the
whole-sequence oracle (oracle.attention_block), through the library's C ABI.

The block is trained chunk by chunk with activation recomputation and the
KV cache and its gradients in pages; chunking and recomputation are exact, so
the outputs y and the gradients of x, wq, wk, wv, wo must equal the
whole-sequence block's. Tolerances (relative Frobenius): 1e-4 for fp32
workloads, 2e-2 for bf16 ones, as for dQ/dK/dV in the other parity tests: the
block adds bf16 projections whose inputs are rounded once (2^-9 relative).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build
from paged_kv_chunk_chunked_gb300 import synth
from paged_kv_chunk_chunked_gb300.layer import ChunkRecurrentBlock
from paged_kv_chunk_chunked_gb300.sweep import to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pkv_build.build()
    B.lib()
    torch.cuda.set_device(0)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("key,kw,hidden,tol", [
    ("tiny_dense_f32", {}, 64, 1e-4),
    ("tiny_dense_f32", dict(N=200), 48, 1e-4),                       # partial last page and chunk
    ("qwen7b_dense_32k", dict(N=1152, C=256, Hq=4, Hkv=2), 256, 2e-2),
    ("qwen7b_dense_128k_perm", dict(N=1024, C=512, Hq=7, Hkv=1, extra_pages=3), 192, 2e-2),
])
def test_chunk_recurrent_block_matches_whole_sequence(key, kw, hidden, tol):
    w = synth.workload(key, **kw)
    n = w.n_chunks
    xs = [synth.block_x(w, c, hidden) for c in range(n)]
    dys = [synth.block_dy(w, c, hidden) for c in range(n)]
    W = synth.block_weights(w, hidden)
    y_ref, g_ref = oracle.attention_block(np.concatenate(xs), W["wq"], W["wk"], W["wv"],
                                          W["wo"], np.concatenate(dys), w.Hq, w.Hkv)
    blk = ChunkRecurrentBlock(w, hidden)
    try:
        xd = [to_device(x, w.dtype) for x in xs]
        dyd = [to_device(x, w.dtype) for x in dys]
        ys = blk.forward(xd)
        dxs, g = blk.backward(xd, dyd)
        torch.cuda.synchronize()
        B.pkv_check(blk.pool)
        err = {"y": _rel(np.concatenate([to_numpy(y) for y in ys]), y_ref),
               "x": _rel(np.concatenate([to_numpy(d) for d in dxs]), g_ref["x"])}
        for name in ("wq", "wk", "wv", "wo"):
            err[name] = _rel(to_numpy(g[name]), g_ref[name])
        assert max(err.values()) <= tol, err
    finally:
        blk.close()


def test_block_twice_gives_the_same_result():
    """The pool is reset between steps: a second step reproduces the first (a
    gradient pool that kept the first step's sums would double dK/dV). Up to
    the order of the dK/dV kernel's fp32 reductions, which bf16 rounding of dK
    before the K projection turns into ~1e-5 relative differences in wk's
    gradient."""
    w = synth.workload("qwen7b_dense_32k", N=768, C=256, Hq=4, Hkv=2)
    hidden = 128
    xd = [to_device(synth.block_x(w, c, hidden), w.dtype) for c in range(w.n_chunks)]
    dyd = [to_device(synth.block_dy(w, c, hidden), w.dtype) for c in range(w.n_chunks)]
    blk = ChunkRecurrentBlock(w, hidden)
    try:
        out = []
        for _ in range(2):
            blk.forward(xd)
            dxs, g = blk.backward(xd, dyd)
            out.append((torch.cat(dxs).float().cpu().numpy(), g["wk"].cpu().numpy()))
        assert _rel(out[1][0], out[0][0]) < 1e-4 and _rel(out[1][1], out[0][1]) < 1e-4
    finally:
        blk.close()
