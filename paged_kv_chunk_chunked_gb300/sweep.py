"""Chunk-recurrent sweep of one attention layer through libpkv.

Drives the library the way a chunk-recurrent trainer would ("Out of the Memory
Barrier", gist.science/de §2.A): forward over chunks 0, 1, ... (append the
chunk's K/V into the paged pool, attend its queries to every key so far),
then backward over the chunks in reverse (dQ out, dK/dV added in place into
the paged gradient pool). PyTorch only supplies device memory and the stream;
every step runs in libpkv's kernels.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

from . import binding as B
from . import synth


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """float32 numpy array (bf16-exact for bf16) -> contiguous device tensor."""
    if dtype == "bf16":
        t = torch.from_numpy(synth.bf16_bits(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(device).contiguous()


def to_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


@dataclass
class ChunkSweep:
    """A paged pool + one sequence holding a workload's layer, with per-chunk buffers."""
    w: synth.Workload
    flags: int = 0
    device: str = "cuda"
    pool: int = 0
    seq: int = 0
    q: list = field(default_factory=list)
    k: list = field(default_factory=list)
    v: list = field(default_factory=list)
    do: list = field(default_factory=list)
    o: list = field(default_factory=list)
    lse: list = field(default_factory=list)
    dq: list = field(default_factory=list)
    sel: list = field(default_factory=list)

    def __post_init__(self):
        w = self.w
        dt = B.PKV_BF16 if w.dtype == "bf16" else B.PKV_F32
        self.pool = B.pkv_pool_create(w.P, w.Hkv, w.Hq, w.d, dt, w.n_phys, flags=self.flags)
        self.seq = B.pkv_seq_create(self.pool)
        self.tdtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32

    def load_inputs(self, chunks=None):
        """Uploads the seeded per-chunk Q, K, V, dO and allocates outputs."""
        w = self.w
        chunks = range(w.n_chunks) if chunks is None else chunks
        for c in chunks:
            s, e = w.chunk_range(c)
            self.q.append(to_device(synth.chunk_q(w, c), w.dtype, self.device))
            self.k.append(to_device(synth.chunk_k(w, c), w.dtype, self.device))
            self.v.append(to_device(synth.chunk_v(w, c), w.dtype, self.device))
            self.do.append(to_device(synth.chunk_do(w, c), w.dtype, self.device))
            self.o.append(torch.empty((e - s, w.Hq, w.d), dtype=self.tdtype, device=self.device))
            self.lse.append(torch.empty((w.Hq, e - s), dtype=torch.float32, device=self.device))
            self.dq.append(torch.empty((e - s, w.Hq, w.d), dtype=self.tdtype, device=self.device))
        return self

    def reset(self):
        """Empties the sequence (pages back to the free list) and re-applies the block table."""
        B.pkv_seq_reset(self.seq)
        if self.w.table == "perm":
            B.pkv_set_block_table(self.seq, synth.block_table(self.w))

    def forward(self, c: int, stream=None, sel=None):
        w = self.w
        s, e = w.chunk_range(c)
        B.pkv_append(self.seq, self.k[c], self.v[c], e - s, stream)
        B.pkv_chunk_attn_fwd(self.seq, self.q[c], s, e - s, self.o[c], self.lse[c], sel, stream)

    def backward(self, c: int, stream=None, sel=None):
        """Backward of chunk c (dQ written, dK/dV added into the gradient pages)."""
        w = self.w
        s, e = w.chunk_range(c)
        B.pkv_chunk_attn_bwd(self.seq, self.q[c], self.o[c], self.do[c], self.lse[c], s, e - s,
                             self.dq[c], sel, stream)

    def run(self, stream=None):
        """Full forward sweep, then the backward sweep over chunks in reverse.

        The backward of chunk c runs with every chunk's keys in the pool; by
        causality its queries see keys up to the chunk's own end only."""
        w = self.w
        self.reset()
        for c in range(w.n_chunks):
            self.forward(c, stream)
        for c in reversed(range(w.n_chunks)):
            self.backward(c, stream)

    def gather(self):
        """Logical-order K, V, dK, dV [N, Hkv, d] and representatives [n_pages, Hkv, d]."""
        w = self.w
        L = B.pkv_seq_length(self.seq)
        n_pg = (L + w.P - 1) // w.P
        k = torch.empty((L, w.Hkv, w.d), dtype=self.tdtype, device=self.device)
        v = torch.empty_like(k)
        dk = torch.empty((L, w.Hkv, w.d), dtype=torch.float32, device=self.device)
        dv = torch.empty_like(dk)
        rep = torch.empty((n_pg, w.Hkv, w.d), dtype=torch.float32, device=self.device)
        B.pkv_gather(self.seq, k, v, dk, dv, rep)
        torch.cuda.synchronize()
        return dict(k=k, v=v, dk=dk, dv=dv, rep=rep)

    def close(self):
        if self.pool:
            B.pkv_pool_destroy(self.pool)
            self.pool = 0
            self.seq = 0
