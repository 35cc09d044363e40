"""CPU-only checks of the C-ABI library: it builds, loads, exports every symbol
include/pkv.h declares, and its host logic (page free list, block tables,
argument validation, error messages) behaves as documented. Nothing here
launches a kernel: the pools are metadata-only (PKV_RES_META)."""
import ctypes
import os
import re

import pytest

from paged_kv_chunk_chunked_gb300 import binding as B
from paged_kv_chunk_chunked_gb300 import build as pkv_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "pkv.h")


@pytest.fixture(scope="module")
def lib():
    pkv_build.build()
    return B.lib()


def _declared():
    txt = open(HEADER).read()
    return set(re.findall(r"^\s*(?:pkv_status|void|const char\s*\*)\s*(pkv_\w+)\s*\(", txt, re.M))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 20
    for n in names:
        assert hasattr(lib, n), n
    assert names == set(B.EXPORTED), names ^ set(B.EXPORTED)


def _meta_pool(pages=10, P=16):
    return B.pkv_pool_create(P, 1, 2, 64, B.PKV_F32, pages, residency=B.PKV_RES_META)


def test_reserve_and_free_list(lib):
    pool = _meta_pool()
    seq = B.pkv_seq_create(pool)
    assert B.pkv_pool_free_pages(pool) == 10
    B.pkv_seq_reserve(seq, 40)                 # ceil(40/16) = 3 pages, taken in order
    assert B.pkv_get_block_table(seq) == [0, 1, 2]
    assert B.pkv_pool_free_pages(pool) == 7
    with pytest.raises(B.PkvError) as e:
        B.pkv_seq_reserve(seq, 16 * 11)         # would need 8 more pages, 7 free
    assert e.value.status == B.PKV_ERR_OOM and "exhausted" in str(e.value)
    assert B.pkv_get_block_table(seq) == [0, 1, 2] and B.pkv_pool_free_pages(pool) == 7
    seq2 = B.pkv_seq_create(pool)
    B.pkv_seq_reserve(seq2, 17)
    assert B.pkv_get_block_table(seq2) == [3, 4]
    B.pkv_seq_reset(seq)
    assert B.pkv_pool_free_pages(pool) == 8
    seq3 = B.pkv_seq_create(pool)
    B.pkv_seq_reserve(seq3, 48)                # the freed pages come back first, in order
    assert B.pkv_get_block_table(seq3) == [0, 1, 2]
    B.pkv_seq_free(seq2)
    assert B.pkv_pool_free_pages(pool) == 7
    B.pkv_pool_destroy(pool)                   # frees remaining sequences too


def test_set_block_table_validation(lib):
    pool = _meta_pool()
    seq = B.pkv_seq_create(pool)
    B.pkv_set_block_table(seq, [7, 2, 9])
    assert B.pkv_get_block_table(seq) == [7, 2, 9]
    assert B.pkv_pool_free_pages(pool) == 7
    B.pkv_seq_reserve(seq, 40)                 # pre-assigned pages cover the first 48 tokens
    assert B.pkv_get_block_table(seq) == [7, 2, 9]
    B.pkv_seq_reserve(seq, 100)                # 100 tokens -> 7 pages: 4 new ones from the free list
    assert B.pkv_get_block_table(seq)[:3] == [7, 2, 9] and len(B.pkv_get_block_table(seq)) == 7
    other = B.pkv_seq_create(pool)
    for bad, why in (([10], "out of range"), ([-1], "out of range"), ([3, 3], "twice"),
                     ([7], "not free")):
        with pytest.raises(B.PkvError) as e:
            B.pkv_set_block_table(other, bad)
        assert e.value.status == B.PKV_ERR_INVALID and why in str(e.value), (bad, str(e.value))
    assert B.pkv_get_block_table(other) == []
    with pytest.raises(B.PkvError):
        B.pkv_set_block_table(seq, [0])         # sequence not empty
    B.pkv_pool_destroy(pool)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), B.PKV_ERR_UNSUPPORTED),
    (dict(page_size=0), B.PKV_ERR_INVALID),
    (dict(page_size=12), B.PKV_ERR_INVALID),
    (dict(n_q_heads=3), B.PKV_ERR_INVALID),
    (dict(num_phys_pages=0), B.PKV_ERR_INVALID),
    (dict(dtype=7), B.PKV_ERR_INVALID),
])
def test_pool_desc_validation(lib, kw, status):
    args = dict(page_size=16, n_kv_heads=2, n_q_heads=4, head_dim=64, dtype=B.PKV_F32,
                num_phys_pages=4, residency=B.PKV_RES_META)
    args.update(kw)
    with pytest.raises(B.PkvError) as e:
        B.pkv_pool_create(**args)
    assert e.value.status == status
    assert B.pkv_last_error()


def test_compute_calls_reject_meta_pools_and_bad_chunks(lib):
    pool = _meta_pool()
    seq = B.pkv_seq_create(pool)
    with pytest.raises(B.PkvError) as e:
        B.pkv_append(seq, 1, 1, 16)
    assert e.value.status == B.PKV_ERR_INVALID
    with pytest.raises(B.PkvError) as e:
        B.pkv_chunk_attn_fwd(seq, 16, 0, 16, 16, 16)
    assert e.value.status == B.PKV_ERR_INVALID
    with pytest.raises(B.PkvError):
        B.pkv_seq_reserve(seq, -1)
    with pytest.raises(B.PkvError) as e:
        B.pkv_gather_rows(seq, 0, 16, dk=16)
    assert e.value.status == B.PKV_ERR_INVALID
    with pytest.raises(B.PkvError) as e:
        B.pkv_grad_accumulate(seq, 0, 16, dk=16)
    assert e.value.status == B.PKV_ERR_INVALID
    with pytest.raises(B.PkvError) as e:
        B.pkv_page_local(seq, 0, 16, 0, 2, 16)
    assert e.value.status == B.PKV_ERR_INVALID
    assert B.pkv_seq_length(seq) == 0
    B.pkv_pool_destroy(pool)


def test_strided_tensors_are_refused_before_the_call(lib):
    import torch
    pool = _meta_pool()
    seq = B.pkv_seq_create(pool)
    with pytest.raises(ValueError):
        B.pkv_gather_rows(seq, 0, 16, dk=torch.zeros(8, 4).t())
    with pytest.raises(ValueError):
        B.pkv_grad_accumulate(seq, 0, 4, dk=torch.zeros(4, 8)[:, ::2])
    B.pkv_pool_destroy(pool)


def test_null_arguments(lib):
    assert lib.pkv_pool_create(None, None) == B.PKV_ERR_INVALID
    assert lib.pkv_seq_create(None, None) == B.PKV_ERR_INVALID
    assert lib.pkv_check(None) == B.PKV_ERR_INVALID
    lib.pkv_pool_destroy(None)                 # NULL-safe
    lib.pkv_seq_free(None)
    n = ctypes.c_int64()
    assert lib.pkv_pool_free_pages(None, ctypes.byref(n)) == B.PKV_ERR_INVALID
