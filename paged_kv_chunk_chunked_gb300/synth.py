"""Seeded synthetic inputs for paged chunk attention.

This module is the one thing the oracle tests and the CUDA path share. It draws
random tensors and block-table permutations and nothing else: it holds none of
the attention, paging or page-selection arithmetic.

Draws use numpy's counter-based Philox generator keyed by (workload seed,
tensor id, chunk index), so any chunk can be regenerated on its own and in any
order. Values are drawn in fp32 and, for bf16 workloads, rounded to bf16 with
round-to-nearest-even; the float32 arrays returned here already hold the
rounded values, so the oracle (which widens them to fp64) and the kernels (which
read the bf16 bit patterns) see the same numbers.

Workloads follow the shapes named in "Out of the Memory Barrier" for
Qwen2.5-7B (28 query heads, 4 KV heads, head dim 128): the pages train that
model on one GPU (gist.science/de §4; sciencestack.ai abstract). Page size,
chunk sizes and distributions are fixed by the workload table below; the pages
do not state them.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "draw_normal", "round_bf16",
    "bf16_bits", "chunk_q", "chunk_k", "chunk_v", "chunk_do", "block_table",
]

# Tensor ids for the Philox key; changing one changes every draw of that tensor.
_TENSOR_ID = {"q": 1, "k": 2, "v": 3, "do": 4, "mu": 5, "perm": 6, "misc": 7, "qmu": 8,
              "wq": 9, "wk": 10, "wv": 11, "wo": 12, "x": 13, "dy": 14}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: sequence/chunk/page geometry, heads, dtype, inputs."""
    name: str
    N: int                 # context length in tokens
    C: int                 # chunk length in tokens
    P: int                 # page size in tokens
    Hq: int                # query heads
    Hkv: int               # KV heads (Hq % Hkv == 0, grouped consecutively)
    d: int                 # head dimension
    dtype: str             # "f32" or "bf16": storage type of Q/K/V/O/dO/dQ
    seed: int
    table: str = "identity"    # "identity" or "perm" (seeded permutation of physical pages)
    keys: str = "normal"       # "normal": K ~ N(0,1); "clustered": page centre N(0,2^2) + N(0,1)
    queries: str = "normal"    # "normal": Q ~ N(0,1); "coherent": (query page, KV group) centre N(0,1) + N(0,1)
    topk: Optional[tuple] = None   # (K, n_sink, n_local) for the page-sparse variant
    local: Optional[tuple] = None  # (n_sink, n_local) for a local attention layer
    offload: bool = False          # pools in pinned host memory, pages streamed to HBM
    extra_pages: int = 0           # physical pages beyond the sequence's need

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def n_chunks(self) -> int:
        return (self.N + self.C - 1) // self.C

    @property
    def n_pages(self) -> int:
        return (self.N + self.P - 1) // self.P

    @property
    def n_phys(self) -> int:
        return self.n_pages + self.extra_pages

    def chunk_range(self, c: int) -> tuple[int, int]:
        s = c * self.C
        return s, min(self.N, s + self.C)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Seeds are 1234 + the workload's index in this table.
WORKLOADS = {
    # Tiny dense fp32: 2 q heads / 1 KV head, d 64, page 16, 256 tokens in 4 chunks of 64.
    "tiny_dense_f32": Workload("tiny_dense_f32", N=256, C=64, P=16, Hq=2, Hkv=1, d=64,
                               dtype="f32", seed=1235),
    # Qwen2.5-7B attention shape, dense, 32K context in chunks of 4096.
    "qwen7b_dense_32k": Workload("qwen7b_dense_32k", N=32768, C=4096, P=128, Hq=28, Hkv=4,
                                 d=128, dtype="bf16", seed=1236),
    # Same shape, 128K context in chunks of 8192, permuted block table.
    "qwen7b_dense_128k_perm": Workload("qwen7b_dense_128k_perm", N=131072, C=8192, P=128,
                                       Hq=28, Hkv=4, d=128, dtype="bf16", seed=1237,
                                       table="perm"),
    # Page-sparse, 256K context, clustered keys, top-64 + 1 sink + 2 local pages.
    "qwen7b_sparse_256k": Workload("qwen7b_sparse_256k", N=262144, C=8192, P=128, Hq=28,
                                   Hkv=4, d=128, dtype="bf16", seed=1238, table="perm",
                                   keys="clustered", topk=(64, 1, 2)),
    # Page-sparse at 1M context with all pages in pinned host memory.
    "qwen7b_sparse_1m_offload": Workload("qwen7b_sparse_1m_offload", N=1048576, C=8192,
                                         P=128, Hq=28, Hkv=4, d=128, dtype="bf16",
                                         seed=1239, table="perm", keys="clustered",
                                         topk=(64, 1, 2), offload=True),
    # Local attention layer (natively sparse models): each query page sees its
    # own page and the one before it, no sink; 256K context, Qwen2.5-7B shape.
    "qwen7b_local_256k": Workload("qwen7b_local_256k", N=262144, C=8192, P=128, Hq=28, Hkv=4,
                                  d=128, dtype="bf16", seed=1240, table="perm", local=(0, 2)),
    # The same local layer with head dimension 64 and 64 query / 8 KV heads:
    # the attention geometry of the published GPT-OSS models, the natively
    # sparse family the pages name (the pages give no shapes for it).
    "gptoss_local_256k": Workload("gptoss_local_256k", N=262144, C=8192, P=128, Hq=64, Hkv=8,
                                  d=64, dtype="bf16", seed=1241, table="perm", local=(0, 2)),
}


def workload(key: str, **overrides) -> Workload:
    """The named workload, optionally with fields replaced (e.g. a smaller N)."""
    w = WORKLOADS[key]
    return replace(w, **overrides) if overrides else w


def _rng(seed: int, tensor: str, chunk: int) -> np.random.Generator:
    key = np.array([seed, (_TENSOR_ID[tensor] << 40) | chunk], dtype=np.uint64)
    return np.random.Generator(np.random.Philox(key=key))


def draw_normal(seed: int, tensor: str, chunk: int, shape, std: float = 1.0) -> np.ndarray:
    """float32 N(0, std^2) draws from the (seed, tensor, chunk) Philox stream."""
    x = _rng(seed, tensor, chunk).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32.

    Inputs must be finite (the generators never produce NaN or Inf)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + bias) & np.uint32(0xFFFF0000)).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns of float32 values that are already bf16-exact."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if np.any(b & np.uint32(0xFFFF)):
        raise ValueError("bf16_bits: values are not bf16-representable; call round_bf16 first")
    return (b >> np.uint32(16)).astype(np.uint16)


def _finish(w: Workload, x: np.ndarray) -> np.ndarray:
    return round_bf16(x) if w.dtype == "bf16" else x


def chunk_q(w: Workload, c: int) -> np.ndarray:
    """Queries of chunk c, [n, Hq, d] float32 (bf16-exact for bf16 workloads)."""
    s, e = w.chunk_range(c)
    eps = draw_normal(w.seed, "q", c, (e - s, w.Hq, w.d))
    if w.queries == "normal":
        return _finish(w, eps)
    if w.queries != "coherent":
        raise ValueError(w.queries)
    # "coherent": the tokens of a query page and the g heads of a KV group share
    # a centre ~ N(0, I) (queries of neighbouring tokens point the same way).
    n_pg = (e - s + w.P - 1) // w.P
    mu = draw_normal(w.seed, "qmu", c, (n_pg, w.Hkv, w.d))
    page_of_token = np.arange(e - s) // w.P
    head_group = np.arange(w.Hq) // w.g
    return _finish(w, mu[page_of_token][:, head_group] + eps)


def chunk_k(w: Workload, c: int) -> np.ndarray:
    """Keys of chunk c, [n, Hkv, d].

    "clustered": every (page, KV head) draws a centre ~ N(0, 2^2 I) and each
    token adds noise ~ N(0, I), so pages differ in how well they match a query."""
    s, e = w.chunk_range(c)
    if w.keys == "normal":
        return _finish(w, draw_normal(w.seed, "k", c, (e - s, w.Hkv, w.d)))
    if w.keys != "clustered":
        raise ValueError(w.keys)
    if s % w.P:
        raise ValueError("clustered keys need chunks that start on a page boundary")
    n_pg = (e - s + w.P - 1) // w.P
    mu = draw_normal(w.seed, "mu", c, (n_pg, w.Hkv, w.d), std=2.0)
    eps = draw_normal(w.seed, "k", c, (e - s, w.Hkv, w.d))
    page_of_token = np.arange(e - s) // w.P
    return _finish(w, mu[page_of_token] + eps)


def chunk_v(w: Workload, c: int) -> np.ndarray:
    s, e = w.chunk_range(c)
    return _finish(w, draw_normal(w.seed, "v", c, (e - s, w.Hkv, w.d)))


def chunk_do(w: Workload, c: int) -> np.ndarray:
    """Upstream gradient dL/dO of chunk c, [n, Hq, d]."""
    s, e = w.chunk_range(c)
    return _finish(w, draw_normal(w.seed, "do", c, (e - s, w.Hq, w.d)))


def block_weights(w: Workload, hidden: int) -> dict:
    """Random projection weights of one attention block, N(0, 1/hidden) (wo:
    N(0, 1/(Hq d))): wq [hidden, Hq d], wk and wv [hidden, Hkv d], wo [Hq d, hidden]."""
    shapes = {"wq": (hidden, w.Hq * w.d), "wk": (hidden, w.Hkv * w.d),
              "wv": (hidden, w.Hkv * w.d), "wo": (w.Hq * w.d, hidden)}
    return {n: _finish(w, draw_normal(w.seed, n, 0, sh, std=float(sh[0]) ** -0.5))
            for n, sh in shapes.items()}


def block_x(w: Workload, c: int, hidden: int) -> np.ndarray:
    """Input of the attention block for chunk c, [n, hidden], N(0, 1)."""
    s, e = w.chunk_range(c)
    return _finish(w, draw_normal(w.seed, "x", c, (e - s, hidden)))


def block_dy(w: Workload, c: int, hidden: int) -> np.ndarray:
    """Upstream gradient of the block's output for chunk c, [n, hidden], N(0, 1)."""
    s, e = w.chunk_range(c)
    return _finish(w, draw_normal(w.seed, "dy", c, (e - s, hidden)))


def block_table(w: Workload) -> np.ndarray:
    """int32 [n_pages]: physical page of each logical page.

    "identity" maps page p to p; "perm" takes the first n_pages entries of a
    seeded permutation of all n_phys physical pages."""
    if w.table == "identity":
        return np.arange(w.n_pages, dtype=np.int32)
    if w.table != "perm":
        raise ValueError(w.table)
    perm = _rng(w.seed, "perm", 0).permutation(w.n_phys)
    return perm[: w.n_pages].astype(np.int32)
