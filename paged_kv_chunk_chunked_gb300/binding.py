"""ctypes binding of libpkv (include/pkv.h): argument marshalling only.

Every function here has the name of the C entry point it calls and passes
plain pointers (ints, or anything with ``data_ptr()`` such as a torch tensor)
and sizes through. All compute runs in the library's CUDA kernels; there is no
fallback: ``lib()`` raises if libpkv.so is missing or does not load.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_OOM, PKV_ERR_CUDA = 0, 1, 2, 3
PKV_ERR_TIMEOUT, PKV_ERR_DEVICE_FAULT, PKV_ERR_UNSUPPORTED = 4, 5, 6
STATUS_NAMES = {0: "PKV_OK", 1: "PKV_ERR_INVALID", 2: "PKV_ERR_OOM", 3: "PKV_ERR_CUDA",
                4: "PKV_ERR_TIMEOUT", 5: "PKV_ERR_DEVICE_FAULT", 6: "PKV_ERR_UNSUPPORTED"}
PKV_BF16, PKV_F32 = 0, 1
PKV_RES_DEVICE, PKV_RES_PINNED_HOST, PKV_RES_META = 0, 1, 2
PKV_FLAG_SIMT_ONLY = 1
PKV_STAGE_KV, PKV_STAGE_GRADS = 1, 2


class PkvError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class pkv_pool_desc(ctypes.Structure):
    _fields_ = [("page_size", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("residency", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int64), ("n_device_slots", ctypes.c_int64),
                ("flags", ctypes.c_uint32), ("reserved", ctypes.c_int32)]


class pkv_sel(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("kmax", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("n_qp", ctypes.c_int64)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_ST = ctypes.c_int
# name -> (restype, argtypes)
_SIGS = {
    "pkv_last_error": (ctypes.c_char_p, []),
    "pkv_check": (_ST, [_P]),
    "pkv_pool_create": (_ST, [ctypes.POINTER(pkv_pool_desc), ctypes.POINTER(_P)]),
    "pkv_pool_destroy": (None, [_P]),
    "pkv_pool_free_pages": (_ST, [_P, ctypes.POINTER(_I64)]),
    "pkv_pool_arrays": (_ST, [_P] + [ctypes.POINTER(_P)] * 5),
    "pkv_seq_create": (_ST, [_P, ctypes.POINTER(_P)]),
    "pkv_seq_free": (None, [_P]),
    "pkv_seq_reset": (_ST, [_P]),
    "pkv_seq_length": (_ST, [_P, ctypes.POINTER(_I64)]),
    "pkv_seq_reserve": (_ST, [_P, _I64]),
    "pkv_get_block_table": (_ST, [_P, _P, _I64, ctypes.POINTER(_I64)]),
    "pkv_set_block_table": (_ST, [_P, _P, _I64]),
    "pkv_append": (_ST, [_P, _P, _P, _I64, _P]),
    "pkv_chunk_attn_fwd": (_ST, [_P, _P, _I64, _I64, _P, _P, ctypes.POINTER(pkv_sel), _P]),
    "pkv_chunk_attn_bwd": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _P, ctypes.POINTER(pkv_sel), _P]),
    "pkv_chunk_attn_bwd_noalloc": (_ST, [_P, _P, _P, _P, _P, _I64, _I64, _P,
                                         ctypes.POINTER(pkv_sel), _P]),
    "pkv_grad_zero": (_ST, [_P, _P]),
    "pkv_gather": (_ST, [_P, _P, _P, _P, _P, _P, _P]),
    "pkv_gather_rows": (_ST, [_P, _I64, _I64, _P, _P, _P, _P, _P]),
    "pkv_grad_accumulate": (_ST, [_P, _I64, _I64, _P, _P, _P]),
    "pkv_page_local": (_ST, [_P, _I64, _I64, _I32, _I32, _P, _P, _P]),
    "pkv_page_topk": (_ST, [_P, _P, _I64, _I64, _I32, _I32, _I32, _P, _P, _P]),
    "pkv_prefetch": (_ST, [_P, _P, _I64, _I32, _P]),
    "pkv_writeback_grads": (_ST, [_P, _P]),
    "pkv_release_slots": (_ST, [_P, _P]),
    "pkv_stage_stats": (_ST, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
    "pkv_wait": (_ST, [_P, _P, _I64]),
    "pkv_selftest_umma": (_ST, [_I32, _P, _P, _P, _I32, _I32]),
    "pkv_profile_enable": (_ST, [_I32]),
    "pkv_profile_collect": (_ST, [_I32, _P, _P, _P, ctypes.POINTER(_I32)]),
}
EXPORTED = tuple(_SIGS)

_lib: Optional[ctypes.CDLL] = None


def lib() -> ctypes.CDLL:
    """Loads libpkv.so (built by ``paged_kv_chunk_chunked_gb300.build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run __graft_entry__.build() first "
                              "(the CUDA library is required; there is no CPU path)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def ptr(x) -> Optional[int]:
    """Address of a tensor-like (``data_ptr()``), an int, or None. Every array
    the library reads or writes is dense in the layout its header states, so a
    strided view is refused here instead of being read as if it were dense."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "is_contiguous") and not x.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(x.shape)} with strides {x.stride()} is not "
                         "contiguous; pass .contiguous()")
    return x.data_ptr()


def stream_ptr(stream) -> Optional[int]:
    if stream is None:
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int):
    if status != PKV_OK:
        raise PkvError(status, lib().pkv_last_error().decode())


def _sel(sel) -> Optional[pkv_sel]:
    """(pages tensor [n_qp, Hkv, kmax]) -> pkv_sel by reference, or None for dense."""
    if sel is None:
        return None
    s = pkv_sel()
    s.pages = ptr(sel)
    s.kmax = int(sel.shape[-1])
    s.n_qp = int(sel.shape[0])
    return ctypes.byref(s)


# ---------------------------------------------------------------- one function per entry point

def pkv_last_error() -> str:
    return lib().pkv_last_error().decode()


def pkv_check(pool) -> None:
    _check(lib().pkv_check(pool))


def pkv_pool_create(page_size, n_kv_heads, n_q_heads, head_dim, dtype=PKV_BF16,
                    num_phys_pages=1, residency=PKV_RES_DEVICE, n_device_slots=0, flags=0) -> int:
    d = pkv_pool_desc(page_size, n_kv_heads, n_q_heads, head_dim, dtype, residency,
                      num_phys_pages, n_device_slots, flags, 0)
    out = _P()
    _check(lib().pkv_pool_create(ctypes.byref(d), ctypes.byref(out)))
    return out.value


def pkv_pool_destroy(pool) -> None:
    lib().pkv_pool_destroy(pool)


def pkv_pool_free_pages(pool) -> int:
    n = _I64()
    _check(lib().pkv_pool_free_pages(pool, ctypes.byref(n)))
    return n.value


def pkv_pool_arrays(pool) -> dict:
    vals = [_P() for _ in range(5)]
    _check(lib().pkv_pool_arrays(pool, *[ctypes.byref(v) for v in vals]))
    return dict(zip(("k", "v", "dk", "dv", "rep"), (v.value for v in vals)))


def pkv_seq_create(pool) -> int:
    out = _P()
    _check(lib().pkv_seq_create(pool, ctypes.byref(out)))
    return out.value


def pkv_seq_free(seq) -> None:
    lib().pkv_seq_free(seq)


def pkv_seq_reset(seq) -> None:
    _check(lib().pkv_seq_reset(seq))


def pkv_seq_length(seq) -> int:
    n = _I64()
    _check(lib().pkv_seq_length(seq, ctypes.byref(n)))
    return n.value


def pkv_seq_reserve(seq, n_tok) -> None:
    _check(lib().pkv_seq_reserve(seq, n_tok))


def pkv_get_block_table(seq) -> list:
    n = _I64()
    _check(lib().pkv_get_block_table(seq, None, 0, ctypes.byref(n)))
    buf = (ctypes.c_int32 * max(1, n.value))()
    _check(lib().pkv_get_block_table(seq, ctypes.cast(buf, _P), n.value, ctypes.byref(n)))
    return list(buf[: n.value])


def pkv_set_block_table(seq, bt) -> None:
    arr = (ctypes.c_int32 * max(1, len(bt)))(*[int(x) for x in bt])
    _check(lib().pkv_set_block_table(seq, ctypes.cast(arr, _P), len(bt)))


def pkv_append(seq, k, v, n_tok, stream=None) -> None:
    _check(lib().pkv_append(seq, ptr(k), ptr(v), n_tok, stream_ptr(stream)))


def pkv_chunk_attn_fwd(seq, q, q_start, n_q, o, lse, sel=None, stream=None) -> None:
    _check(lib().pkv_chunk_attn_fwd(seq, ptr(q), q_start, n_q, ptr(o), ptr(lse), _sel(sel),
                                    stream_ptr(stream)))


def pkv_chunk_attn_bwd(seq, q, o, dout, lse, q_start, n_q, dq, sel=None, stream=None) -> None:
    _check(lib().pkv_chunk_attn_bwd(seq, ptr(q), ptr(o), ptr(dout), ptr(lse), q_start, n_q,
                                    ptr(dq), _sel(sel), stream_ptr(stream)))


def pkv_chunk_attn_bwd_noalloc(seq, q, o, dout, lse, q_start, n_q, dq, sel=None,
                               stream=None) -> None:
    """Same as pkv_chunk_attn_bwd, with the library's fixed device scratch instead
    of an allocation (for callers that cannot allocate at call time)."""
    _check(lib().pkv_chunk_attn_bwd_noalloc(seq, ptr(q), ptr(o), ptr(dout), ptr(lse), q_start,
                                            n_q, ptr(dq), _sel(sel), stream_ptr(stream)))


def pkv_grad_zero(seq, stream=None) -> None:
    _check(lib().pkv_grad_zero(seq, stream_ptr(stream)))


def pkv_grad_accumulate(seq, row0, n_rows, dk=None, dv=None, stream=None) -> None:
    _check(lib().pkv_grad_accumulate(seq, row0, n_rows, ptr(dk), ptr(dv), stream_ptr(stream)))


def pkv_gather(seq, k=None, v=None, dk=None, dv=None, rep=None, stream=None) -> None:
    _check(lib().pkv_gather(seq, ptr(k), ptr(v), ptr(dk), ptr(dv), ptr(rep), stream_ptr(stream)))


def pkv_gather_rows(seq, row0, n_rows, k=None, v=None, dk=None, dv=None, stream=None) -> None:
    _check(lib().pkv_gather_rows(seq, row0, n_rows, ptr(k), ptr(v), ptr(dk), ptr(dv),
                                 stream_ptr(stream)))


def pkv_page_topk(seq, q, q_start, n_q, k, n_sink, n_local, pages_out, counts_out=None,
                  stream=None) -> None:
    _check(lib().pkv_page_topk(seq, ptr(q), q_start, n_q, k, n_sink, n_local, ptr(pages_out),
                               ptr(counts_out), stream_ptr(stream)))


def pkv_page_local(seq, q_start, n_q, n_sink, n_local, pages_out, counts_out=None,
                   stream=None) -> None:
    _check(lib().pkv_page_local(seq, q_start, n_q, n_sink, n_local, ptr(pages_out),
                                ptr(counts_out), stream_ptr(stream)))


def pkv_prefetch(seq, logical_pages=None, n=0, what=3, side=None) -> None:
    """what: PKV_STAGE_KV (1) | PKV_STAGE_GRADS (2)."""
    _check(lib().pkv_prefetch(seq, ptr(logical_pages), n, what, stream_ptr(side)))


def pkv_writeback_grads(seq, side=None) -> None:
    _check(lib().pkv_writeback_grads(seq, stream_ptr(side)))


def pkv_release_slots(seq, side=None) -> None:
    _check(lib().pkv_release_slots(seq, stream_ptr(side)))


def pkv_stage_stats(seq) -> dict:
    """Page-heads moved by the sequence's staging so far."""
    kv, gi, go = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    _check(lib().pkv_stage_stats(seq, ctypes.byref(kv), ctypes.byref(gi), ctypes.byref(go)))
    return {"kv_in": kv.value, "grads_in": gi.value, "grads_out": go.value}


def pkv_wait(seq, main=None, timeout_us=10_000_000) -> None:
    _check(lib().pkv_wait(seq, stream_ptr(main), timeout_us))


def pkv_profile_enable(on: bool) -> None:
    _check(lib().pkv_profile_enable(1 if on else 0))


def pkv_profile_collect(max_kernels: int = 64) -> dict:
    """{kernel name: (launches, total device ms)} since profiling was enabled."""
    names = ctypes.create_string_buffer(64 * max_kernels)
    ms = (ctypes.c_double * max_kernels)()
    cnt = (ctypes.c_int64 * max_kernels)()
    n = _I32()
    _check(lib().pkv_profile_collect(max_kernels, ctypes.cast(names, _P), ctypes.cast(ms, _P),
                                     ctypes.cast(cnt, _P), ctypes.byref(n)))
    out = {}
    for k in range(min(n.value, max_kernels)):
        name = names.raw[64 * k: 64 * k + 64].split(b"\0", 1)[0].decode()
        out[name] = (int(cnt[k]), float(ms[k]))
    return out


def pkv_selftest_umma(mode, a, b, d, lbo=0, sbo=0) -> None:
    _check(lib().pkv_selftest_umma(mode, ptr(a), ptr(b), ptr(d), lbo, sbo))
