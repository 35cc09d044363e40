"""Pins for the dense oracle: each test ties it to something other than itself.

- library attention (torch scaled_dot_product_attention in fp64, and autograd
  through it) for O and dQ/dK/dV;
- central finite differences of L = sum(O * dO) for the backward;
- closed forms (zero queries, equal values, single key, the hand-worked
  three-token example in tests/golden/hand_example.json);
- invariants (shift invariance, sum_j dK_j = 0, sum_j dV_j = sum_i dO_i);
- paging and chunk recurrence: chunked, paged processing (identity or
  permuted block table) equals one-shot full-sequence attention.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc
from paged_kv_chunk_chunked_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, q_start=0):
    """torch's causal attention in fp64 with consecutive GQA grouping (h -> h // g)."""
    n, Hq, d = q.shape
    L, Hkv, _ = k.shape
    g = Hq // Hkv
    tq = torch.tensor(q, dtype=torch.float64).permute(1, 0, 2)[None]
    tk = torch.tensor(k, dtype=torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    tv = torch.tensor(v, dtype=torch.float64).repeat_interleave(g, dim=1).permute(1, 0, 2)[None]
    # query i sits at global position q_start + i; key j at position j
    mask = torch.arange(L)[None, :] <= (q_start + torch.arange(n))[:, None]
    return tq, tk, tv, mask


def test_forward_matches_library_attention():
    n, Hq, Hkv, d = 37, 6, 2, 16
    q, k, v = _rand((n, Hq, d), 1), _rand((n, Hkv, d), 2), _rand((n, Hkv, d), 3)
    o, lse = orc.attention_forward(q, k, v, 0)
    tq, tk, tv, mask = _sdpa(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_forward_chunk_offset_matches_library_attention():
    # a chunk of 20 queries starting at position 30 against 50 keys
    L, n, Hq, Hkv, d = 50, 20, 4, 1, 8
    k, v = _rand((L, Hkv, d), 4), _rand((L, Hkv, d), 5)
    q = _rand((n, Hq, d), 6)
    o, _ = orc.attention_forward(q, k, v, 30)
    tq, tk, tv, mask = _sdpa(q, k, v, q_start=30)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_backward_matches_library_autograd():
    L, n, Hq, Hkv, d = 45, 15, 6, 3, 8
    k, v = _rand((L, Hkv, d), 7), _rand((L, Hkv, d), 8)
    q, do = _rand((n, Hq, d), 9), _rand((n, Hq, d), 10)
    q_start = L - n
    o, lse = orc.attention_forward(q, k, v, q_start)
    dq, dk, dv = orc.attention_backward(q, k, v, o, do, lse, q_start)
    tq = torch.tensor(q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(k, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(v, dtype=torch.float64, requires_grad=True)
    g = Hq // Hkv
    mask = torch.arange(L)[None, :] <= (q_start + torch.arange(n))[:, None]
    out = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(g, 1).permute(1, 0, 2)[None],
        tv.repeat_interleave(g, 1).permute(1, 0, 2)[None], attn_mask=mask)
    (out[0].permute(1, 0, 2) * torch.tensor(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)


def test_backward_finite_differences():
    L, n, Hq, Hkv, d = 12, 8, 4, 2, 5
    k, v = _rand((L, Hkv, d), 11), _rand((L, Hkv, d), 12)
    q, do = _rand((n, Hq, d), 13), _rand((n, Hq, d), 14)
    q_start = L - n

    def loss(q_, k_, v_):
        o_, _ = orc.attention_forward(q_, k_, v_, q_start)
        return float((o_ * do).sum())

    o, lse = orc.attention_forward(q, k, v, q_start)
    dq, dk, dv = orc.attention_backward(q, k, v, o, do, lse, q_start)
    eps = 1e-6
    rng = np.random.default_rng(0)
    for name, x, gx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(s)) for s in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - gx[idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, gx[idx])


def test_closed_form_zero_queries():
    # q = 0: every visible key gets the same weight, O_i = mean_{j<=i} v_j, LSE_i = ln(i+1)
    L, Hq, Hkv, d = 20, 4, 2, 6
    q = np.zeros((L, Hq, d))
    k, v = _rand((L, Hkv, d), 15), _rand((L, Hkv, d), 16)
    o, lse = orc.attention_forward(q, k, v, 0)
    for i in range(L):
        for h in range(Hq):
            np.testing.assert_allclose(o[i, h], v[: i + 1, h // 2].mean(0), atol=1e-13)
            assert abs(lse[h, i] - math.log(i + 1)) < 1e-13


def test_closed_form_equal_values_and_single_key():
    L, Hq, Hkv, d = 10, 2, 1, 4
    q, k = _rand((L, Hq, d), 17), _rand((L, Hkv, d), 18)
    v = np.broadcast_to(np.arange(1.0, d + 1), (L, Hkv, d)).copy()
    o, lse = orc.attention_forward(q, k, v, 0)
    np.testing.assert_allclose(o, np.broadcast_to(v[:1], o.shape[:1] + (1, d)).repeat(Hq, 1),
                               atol=1e-13)
    # the first query sees exactly one key: O_0 = v_0 and LSE_0 = S_00
    for h in range(Hq):
        assert abs(lse[h, 0] - q[0, h] @ k[0, 0] / math.sqrt(d)) < 1e-13


def test_shift_invariance():
    # k_j -> k_j + c for every j: logits shift by s q_i.c, so O is unchanged
    # and LSE_i moves by exactly s q_i.c
    L, Hq, Hkv, d = 24, 2, 1, 8
    q, k, v = _rand((L, Hq, d), 19), _rand((L, Hkv, d), 20), _rand((L, Hkv, d), 21)
    c = _rand((d,), 22)
    o1, l1 = orc.attention_forward(q, k, v, 0)
    o2, l2 = orc.attention_forward(q, k + c, v, 0)
    np.testing.assert_allclose(o1, o2, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, (q @ c).T / math.sqrt(d), atol=1e-12)


def test_backward_invariants():
    # sum_j dS_ij = 0 for every row, so sum_j dK_j = 0; sum_j P_ij = 1, so
    # sum_j dV_j = sum over the group's heads and queries of dO_i
    L, n, Hq, Hkv, d = 40, 16, 6, 2, 8
    k, v = _rand((L, Hkv, d), 23), _rand((L, Hkv, d), 24)
    q, do = _rand((n, Hq, d), 25), _rand((n, Hq, d), 26)
    o, lse = orc.attention_forward(q, k, v, L - n)
    _, dk, dv = orc.attention_backward(q, k, v, o, do, lse, L - n)
    np.testing.assert_allclose(dk.sum(0), 0, atol=1e-12)
    for h in range(Hkv):
        np.testing.assert_allclose(dv[:, h].sum(0), do[:, 3 * h:3 * h + 3].sum((0, 1)),
                                   atol=1e-12)


def _golden_value(x):
    names = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4),
             "3ln3/8": 3 * math.log(3) / 8, "-ln3/4": -math.log(3) / 4,
             "ln2/2": math.log(2) / 2}
    if isinstance(x, list):
        return [_golden_value(e) for e in x]
    return names[x] if isinstance(x, str) else float(x)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    arr = {key: np.array(_golden_value(g[key]))
           for key in ("q", "k", "v", "do", "o", "lse", "dq", "dk", "dv")}
    q, k, v, do = (arr[x][:, None, :] for x in ("q", "k", "v", "do"))
    o, lse = orc.attention_forward(q, k, v, 0)
    np.testing.assert_allclose(o[:, 0], arr["o"], atol=1e-14)
    np.testing.assert_allclose(lse[0], arr["lse"], atol=1e-14)
    dq, dk, dv = orc.attention_backward(q, k, v, o, do, lse, 0)
    np.testing.assert_allclose(dq[:, 0], arr["dq"], atol=1e-14)
    np.testing.assert_allclose(dk[:, 0], arr["dk"], atol=1e-14)
    np.testing.assert_allclose(dv[:, 0], arr["dv"], atol=1e-14)


def test_full_matrix_path_matches_library():
    N, Hq, Hkv, d = 33, 4, 2, 8
    q, k, v = _rand((N, Hq, d), 27), _rand((N, Hkv, d), 28), _rand((N, Hkv, d), 29)
    o, lse = orc.full_causal_attention(q, k, v)
    tq, tk, tv, mask = _sdpa(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask)
    np.testing.assert_allclose(o, ref[0].permute(1, 0, 2).numpy(), atol=1e-12)
    o2, lse2 = orc.attention_forward(q, k, v, 0)
    np.testing.assert_allclose(lse, lse2, atol=1e-12)


def _tiny_inputs(w):
    qs = [synth.chunk_q(w, c) for c in range(w.n_chunks)]
    ks = [synth.chunk_k(w, c) for c in range(w.n_chunks)]
    vs = [synth.chunk_v(w, c) for c in range(w.n_chunks)]
    dos = [synth.chunk_do(w, c) for c in range(w.n_chunks)]
    return qs, ks, vs, dos


@pytest.mark.parametrize("table", ["identity", "perm"])
def test_chunk_recurrent_paged_equals_one_shot(table):
    """Chunked paged fwd/bwd (4 chunks of 64, pages of 16) == one-shot full causal."""
    w = synth.workload("tiny_dense_f32", table=table, extra_pages=5)
    qs, ks, vs, dos = _tiny_inputs(w)
    bt = synth.block_table(w)
    res = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    Q, K, V, dO = (np.concatenate(x) for x in (qs, ks, vs, dos))
    o, lse = orc.full_causal_attention(Q, K, V)
    np.testing.assert_allclose(np.concatenate(res["o"]), o, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(res["lse"], axis=1), lse, atol=1e-12)
    # full backward through library autograd on the whole sequence
    tq = torch.tensor(Q, dtype=torch.float64, requires_grad=True)
    tk = torch.tensor(K, dtype=torch.float64, requires_grad=True)
    tv = torch.tensor(V, dtype=torch.float64, requires_grad=True)
    out = torch.nn.functional.scaled_dot_product_attention(
        tq.permute(1, 0, 2)[None], tk.repeat_interleave(w.g, 1).permute(1, 0, 2)[None],
        tv.repeat_interleave(w.g, 1).permute(1, 0, 2)[None], is_causal=True)
    (out[0].permute(1, 0, 2) * torch.tensor(dO, dtype=torch.float64)).sum().backward()
    np.testing.assert_allclose(np.concatenate(res["dq"]), tq.grad.numpy(), atol=1e-11)
    dk = orc.logical_rows(res["dkpool"], bt, w.N, w.P)
    dv = orc.logical_rows(res["dvpool"], bt, w.N, w.P)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-11)
    # pages not owned by the sequence stay untouched
    unused = np.setdiff1d(np.arange(w.n_phys), bt)
    assert unused.size == 5 and not res["kpool"][unused].any() and not res["dkpool"][unused].any()


def test_partial_last_page_paged_equals_one_shot():
    """N=200 with P=16: the last page holds 8 rows; chunks of 64, 64, 64, 8."""
    w = synth.workload("tiny_dense_f32", N=200, table="perm", extra_pages=3)
    qs, ks, vs, dos = _tiny_inputs(w)
    bt = synth.block_table(w)
    res = orc.chunk_recurrent_step(qs, ks, vs, dos, bt, w.P, w.n_phys)
    Q, K, V = (np.concatenate(x) for x in (qs, ks, vs))
    o, lse = orc.full_causal_attention(Q, K, V)
    np.testing.assert_allclose(np.concatenate(res["o"]), o, atol=1e-12)
    np.testing.assert_allclose(np.concatenate(res["lse"], axis=1), lse, atol=1e-12)


def test_synth_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.005859375, 1.0078125, -2.0009765625], np.float32)
    r = synth.round_bf16(x)
    # 1 + 2^-8 is halfway between 1 and 1 + 2^-7 -> ties to even (1.0);
    # 1 + 3*2^-9 rounds up to 1 + 2^-7; -2 - 2^-10 rounds to -2
    np.testing.assert_array_equal(r, np.array([1.0, 1.0, 1.0078125, 1.0078125, -2.0], np.float32))
    t = torch.tensor(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(r, t)


def test_paged_gradient_accumulation_equals_contiguous_sums():
    """scatter_rows(accumulate=True) through a permuted block table, read back in
    logical order, equals the same additions on a contiguous [N, Hkv, d] array;
    rows outside every range and physical pages outside the table stay zero.
    In float32 each element takes exactly one rounded addition per call."""
    P, Hkv, d, n_pages, extra = 16, 2, 8, 10, 3
    N = n_pages * P - 5                                   # partial last page
    bt = np.random.default_rng(7).permutation(n_pages + extra)[:n_pages].astype(np.int32)
    pool = np.zeros((n_pages + extra, Hkv, P, d), np.float32)
    flat = np.zeros((N, Hkv, d), np.float32)
    for i, (r0, n) in enumerate([(0, N), (37, 60), (3 * P - 1, 2), (N - 1, 1), (20, 90)]):
        delta = np.random.default_rng(100 + i).standard_normal((n, Hkv, d)).astype(np.float32)
        orc.scatter_rows(pool, bt, r0, delta, P, accumulate=True)
        flat[r0:r0 + n] = flat[r0:r0 + n] + delta
    np.testing.assert_array_equal(orc.logical_rows(pool, bt, N, P), flat)
    unused = np.setdiff1d(np.arange(n_pages + extra), bt)
    assert not pool[unused].any()
    assert not pool[bt[-1], :, P - 5:].any()             # rows beyond the sequence
    assert pool.dtype == np.float32


def test_attention_block_matches_library_autograd():
    """The whole-sequence attention block (projections, causal GQA attention,
    output projection, residual) and all five gradients against torch autograd
    in fp64 through scaled_dot_product_attention."""
    N, hidden, Hq, Hkv, d = 48, 24, 4, 2, 8
    rng = np.random.default_rng(11)
    x = rng.standard_normal((N, hidden))
    ws = [rng.standard_normal(s) / 4 for s in ((hidden, Hq * d), (hidden, Hkv * d),
                                               (hidden, Hkv * d), (Hq * d, hidden))]
    dy = rng.standard_normal((N, hidden))
    y, grads = orc.attention_block(x, *ws, dy, Hq, Hkv)
    tx = torch.tensor(x, requires_grad=True)
    tw = [torch.tensor(w, requires_grad=True) for w in ws]
    q = (tx @ tw[0]).view(N, Hq, d).permute(1, 0, 2)
    k = (tx @ tw[1]).view(N, Hkv, d).repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    v = (tx @ tw[2]).view(N, Hkv, d).repeat_interleave(Hq // Hkv, dim=1).permute(1, 0, 2)
    a = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    ty = tx + a.permute(1, 0, 2).reshape(N, Hq * d) @ tw[3]
    (ty * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(y, ty.detach().numpy(), atol=1e-12)
    for name, t in zip(("x", "wq", "wk", "wv", "wo"), [tx] + tw):
        np.testing.assert_allclose(grads[name], t.grad.numpy(), atol=1e-10, err_msg=name)
