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

    def run_from_host(self, host: dict, out: dict, dk: torch.Tensor, dv: torch.Tensor,
                      h2d_stream, d2h_stream):
        """One layer sweep whose inputs start and whose results end in pinned
        host memory: host["q"|"k"|"v"|"do"][c] -> device, then out["dq"][c],
        out["dk"], out["dv"] <- device (dk, dv: device [N, Hkv, d] fp32 staging).

        The copies run on two side streams, overlapped with the kernels on the
        current stream: chunk c's forward waits only for chunk c's Q, K, V; dO
        arrives (last chunk first) while the forward runs; chunk c's dQ and
        the dK/dV rows of chunk c's keys (final once chunk c's own backward has
        run: no earlier chunk sees them) go back while the backward of chunk
        c - 1 runs. Only the first chunk's inputs and chunk 0's results are
        exposed."""
        w = self.w
        n = w.n_chunks
        comp = torch.cuda.current_stream()
        fwd_ready = [torch.cuda.Event() for _ in range(n)]
        bwd_ready = [torch.cuda.Event() for _ in range(n)]
        dq_done = [torch.cuda.Event() for _ in range(n)]
        h2d_stream.wait_stream(comp)              # the previous user of the buffers is done
        with torch.cuda.stream(h2d_stream):
            for c in range(n):
                for dst, src in ((self.q[c], host["q"][c]), (self.k[c], host["k"][c]),
                                 (self.v[c], host["v"][c])):
                    dst.copy_(src, non_blocking=True)
                fwd_ready[c].record(h2d_stream)
            for c in reversed(range(n)):
                self.do[c].copy_(host["do"][c], non_blocking=True)
                bwd_ready[c].record(h2d_stream)
        self.reset()
        for c in range(n):
            comp.wait_event(fwd_ready[c])
            self.forward(c, comp)
        for c in reversed(range(n)):
            s, e = w.chunk_range(c)
            comp.wait_event(bwd_ready[c])
            self.backward(c, comp)
            B.pkv_gather_rows(self.seq, s, e - s, None, None, dk[s:e], dv[s:e], comp)
            dq_done[c].record(comp)
            d2h_stream.wait_event(dq_done[c])
            with torch.cuda.stream(d2h_stream):
                out["dq"][c].copy_(self.dq[c], non_blocking=True)
                out["dk"][s:e].copy_(dk[s:e], non_blocking=True)
                out["dv"][s:e].copy_(dv[s:e], non_blocking=True)
        comp.wait_stream(d2h_stream)

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
