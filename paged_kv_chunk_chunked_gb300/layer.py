"""Chunk-recurrent training of one attention block on the paged KV cache.

The block is y = x + A wo, A = causal GQA attention(x wq, x wk, x wv), with
random weights (no data or trained model is involved). "Out of the Memory
Barrier" trains a layer chunk by chunk and recomputes activations in the
backward pass, so activation memory does not grow with the context; the KV
cache and its gradients live in pages and grow instead (gist.science/de §2.A
and §2.B; sciencestack.ai Fig. 1 and Fig. 3 captions). Here:

* forward, chunks in order: project the chunk, append its K/V to the paged
  cache (``pkv_append``), attend (``pkv_chunk_attn_fwd``), output projection
  and residual. Nothing per chunk is kept.
* backward, chunks in reverse: recompute the chunk's Q and its attention
  output and LSE (``pkv_chunk_attn_fwd`` again, over the full cache: the
  kernel sees keys up to each query only), dA = dy wo^T,
  ``pkv_chunk_attn_bwd`` (dQ written; dK/dV added into the paged gradient
  pool), then the chunk's own dK/dV rows, final because every later chunk's
  backward has run, are read out (``pkv_gather_rows``) and go back through
  the K/V projections.

No rotary embedding or normalisation: the block exercises the path's KV-side
memory and compute, not a particular model. The projections are plain torch
matmuls (cuBLAS); every attention step runs in the library's kernels.
"""
from __future__ import annotations

import torch

from . import binding as B
from . import synth
from .sweep import to_device


class ChunkRecurrentBlock:
    """One attention block of workload ``w`` (heads, page size, chunk length,
    dtype) with hidden size ``hidden`` and the seeded weights of
    ``synth.block_weights``; a paged pool holding one sequence of w.N tokens."""

    def __init__(self, w: synth.Workload, hidden: int, flags: int = 0):
        self.w, self.hidden = w, hidden
        self.dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
        self.weights = {n: to_device(a, w.dtype) for n, a in synth.block_weights(w, hidden).items()}
        pdt = B.PKV_BF16 if w.dtype == "bf16" else B.PKV_F32
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        self.pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, pdt, w.n_phys, flags=flags)
        torch.cuda.synchronize()
        self.pool_device_bytes = free0 - torch.cuda.mem_get_info()[0]   # K, V, dK, dV pages, reps
        self.seq = B.pkv_seq_create(self.pool)
        C = w.C
        self.o = torch.empty((C, w.Hq, w.d), dtype=self.dt, device="cuda")
        self._lse = torch.empty(w.Hq * C, dtype=torch.float32, device="cuda")
        self.dq = torch.empty((C, w.Hq, w.d), dtype=self.dt, device="cuda")
        self.dk = torch.empty((C, w.Hkv, w.d), dtype=torch.float32, device="cuda")
        self.dv = torch.empty_like(self.dk)

    def _lse_of(self, n: int) -> torch.Tensor:
        """[Hq, n] float32, contiguous (a partial last chunk has n < C)."""
        return self._lse[: self.w.Hq * n].view(self.w.Hq, n)

    def _reset(self):
        B.pkv_seq_reset(self.seq)
        if self.w.table == "perm":
            B.pkv_set_block_table(self.seq, synth.block_table(self.w))

    def forward(self, xs: list) -> list:
        """Chunks in order, on the current stream; returns every chunk's output y."""
        w, W = self.w, self.weights
        stream = torch.cuda.current_stream()
        self._reset()
        ys = []
        for c, x in enumerate(xs):
            s, e = w.chunk_range(c)
            n = e - s
            q = (x @ W["wq"]).view(n, w.Hq, w.d)
            k = (x @ W["wk"]).view(n, w.Hkv, w.d)
            v = (x @ W["wv"]).view(n, w.Hkv, w.d)
            B.pkv_append(self.seq, k, v, n, stream)
            B.pkv_chunk_attn_fwd(self.seq, q, s, n, self.o[:n], self._lse_of(n), None, stream)
            ys.append(x + self.o[:n].view(n, -1) @ W["wo"])
        return ys

    def backward(self, xs: list, dys: list):
        """Chunks in reverse, on the current stream, after ``forward`` of the same
        inputs. Returns every chunk's input gradient and the weight gradients
        (float32)."""
        w, W = self.w, self.weights
        stream = torch.cuda.current_stream()
        g = {n: torch.zeros(t.shape, dtype=torch.float32, device="cuda") for n, t in W.items()}
        dxs = [None] * len(xs)
        for c in reversed(range(len(xs))):
            s, e = w.chunk_range(c)
            n = e - s
            x, dy = xs[c], dys[c]
            q = (x @ W["wq"]).view(n, w.Hq, w.d)                      # recomputed
            o, lse, dq = self.o[:n], self._lse_of(n), self.dq[:n]
            B.pkv_chunk_attn_fwd(self.seq, q, s, n, o, lse, None, stream)   # recomputed
            a = o.view(n, -1)
            da = (dy @ W["wo"].t()).view(n, w.Hq, w.d)
            g["wo"] += (a.t() @ dy).float()
            B.pkv_chunk_attn_bwd(self.seq, q, o, da, lse, s, n, dq, None, stream)
            # rows s..e-1 of dK/dV are final: no earlier chunk's queries see them
            B.pkv_gather_rows(self.seq, s, n, None, None, self.dk[:n], self.dv[:n], stream)
            dqf = dq.view(n, -1)
            dkf = self.dk[:n].view(n, -1).to(self.dt)
            dvf = self.dv[:n].view(n, -1).to(self.dt)
            dxs[c] = dy + dqf @ W["wq"].t() + dkf @ W["wk"].t() + dvf @ W["wv"].t()
            xt = x.t()
            g["wq"] += (xt @ dqf).float()
            g["wk"] += (xt @ dkf).float()
            g["wv"] += (xt @ dvf).float()
        return dxs, g

    def close(self):
        if self.pool:
            B.pkv_pool_destroy(self.pool)
            self.pool = 0
