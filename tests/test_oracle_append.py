"""Pins of the oracle's draft-KV append.

"Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token
Context", §3: each draft forward writes its own token's K and V into the
draft cache that the next forward re-reads; App. A "The windowing change":
the row goes to the slot the ring rule (or the page table) gives.  The pool
layout is [num_slots][H_kv][D]: the K (or V) row of KV head g for slot s
starts at element (s * H_kv + g) * D.

The expected pools are built here by numpy fancy-index assignment, an
operation independent of the oracle's C loop, on pools whose every element
is distinct, so that a wrong head stride, a swapped K/V source, a per-token
offset error or a write outside the target slots changes some element.
CPU only.
"""
import numpy as np
import pytest

import oracle


def _distinct_pool(num_slots, H_kv, D, base):
    """A pool whose elements are pairwise distinct 16-bit patterns."""
    n = num_slots * H_kv * D
    assert base + n <= 0x10000
    return (np.arange(n, dtype=np.int64) + base).astype(np.uint16).reshape(num_slots, H_kv, D)


@pytest.mark.parametrize("H_kv,D,n", [(2, 8, 5), (3, 16, 7), (1, 4, 1), (4, 8, 12)])
def test_append_writes_each_row_to_its_slot(H_kv, D, n):
    rng = np.random.default_rng(100 * H_kv + D + n)
    num_slots = 40
    k_pool = _distinct_pool(num_slots, H_kv, D, 0)
    v_pool = _distinct_pool(num_slots, H_kv, D, 0x8000)
    k_new = rng.integers(0, 0x10000, size=(n, H_kv, D)).astype(np.uint16)
    v_new = rng.integers(0, 0x10000, size=(n, H_kv, D)).astype(np.uint16)
    assert not np.array_equal(k_new, v_new)
    slots = rng.permutation(num_slots)[:n].astype(np.int32)

    exp_k, exp_v = k_pool.copy(), v_pool.copy()
    exp_k[slots] = k_new
    exp_v[slots] = v_new

    oracle.append_kv(k_new, v_new, slots, k_pool, v_pool)
    assert np.array_equal(k_pool, exp_k)
    assert np.array_equal(v_pool, exp_v)
    untouched = np.setdiff1d(np.arange(num_slots), slots)
    assert np.array_equal(k_pool[untouched], _distinct_pool(num_slots, H_kv, D, 0)[untouched])
    assert np.array_equal(v_pool[untouched], _distinct_pool(num_slots, H_kv, D, 0x8000)[untouched])


def test_append_head_rows_land_at_head_offsets():
    """Row of KV head g of token i sits at flat element (slot*H_kv + g)*D."""
    H_kv, D, num_slots = 3, 4, 6
    k_pool = np.zeros((num_slots, H_kv, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    # token i, head g, element e carries the code 0x1000*(i+1) + 0x100*g + e
    n = 2
    k_new = np.zeros((n, H_kv, D), np.uint16)
    for i in range(n):
        for g in range(H_kv):
            for e in range(D):
                k_new[i, g, e] = 0x1000 * (i + 1) + 0x100 * g + e
    v_new = (k_new | 0x8000).astype(np.uint16)
    slots = np.array([4, 1], np.int32)
    oracle.append_kv(k_new, v_new, slots, k_pool, v_pool)
    flat_k, flat_v = k_pool.reshape(-1), v_pool.reshape(-1)
    for i, s in enumerate(slots):
        for g in range(H_kv):
            for e in range(D):
                assert flat_k[(s * H_kv + g) * D + e] == 0x1000 * (i + 1) + 0x100 * g + e
                assert flat_v[(s * H_kv + g) * D + e] == (0x1000 * (i + 1) + 0x100 * g + e) | 0x8000
    written = {(s * H_kv + g) * D + e for s in slots for g in range(H_kv) for e in range(D)}
    for idx in range(flat_k.size):
        if idx not in written:
            assert flat_k[idx] == 0 and flat_v[idx] == 0


def test_append_later_token_wins_on_a_repeated_slot():
    """Tokens are written in order: a slot named twice holds the later row."""
    H_kv, D = 2, 8
    k_pool = np.zeros((5, H_kv, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    k_new = np.stack([np.full((H_kv, D), 0x3F80, np.uint16), np.full((H_kv, D), 0x4000, np.uint16)])
    v_new = np.stack([np.full((H_kv, D), 0xBF80, np.uint16), np.full((H_kv, D), 0xC000, np.uint16)])
    oracle.append_kv(k_new, v_new, np.array([3, 3], np.int32), k_pool, v_pool)
    assert np.all(k_pool[3] == 0x4000) and np.all(v_pool[3] == 0xC000)
    assert not k_pool[[0, 1, 2, 4]].any() and not v_pool[[0, 1, 2, 4]].any()


@pytest.mark.parametrize("bad", [-1, 6, 1 << 20])
def test_append_rejects_a_slot_outside_the_pool(bad):
    H_kv, D = 2, 4
    k_pool = _distinct_pool(6, H_kv, D, 0)
    v_pool = _distinct_pool(6, H_kv, D, 0x8000)
    before_k, before_v = k_pool.copy(), v_pool.copy()
    k_new = np.ones((1, H_kv, D), np.uint16)
    with pytest.raises(ValueError):
        oracle.append_kv(k_new, k_new, np.array([bad], np.int32), k_pool, v_pool)
    assert np.array_equal(k_pool, before_k) and np.array_equal(v_pool, before_v)


def test_appended_row_is_what_a_one_key_table_attends():
    """Consequence through the attention closed form (a single key: the
    output is its value row, lse = its scaled logit): after an append, a
    table listing only the new slot returns, for every query head h, the V
    row of KV head h // G that was appended."""
    H_q, H_kv, D = 4, 2, 8
    G = H_q // H_kv
    k_pool = np.zeros((9, H_kv, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    # values: small integers (exact in bf16); K rows: 1.0 in one dimension
    vals = np.arange(H_kv * D, dtype=np.float32).reshape(1, H_kv, D) + 1.0
    v_new = (vals.view(np.uint32) >> 16).astype(np.uint16)
    k_rows = np.zeros((1, H_kv, D), np.float32)
    k_rows[0, 0, 0] = 1.0
    k_rows[0, 1, 1] = 1.0
    k_new = (k_rows.view(np.uint32) >> 16).astype(np.uint16)
    oracle.append_kv(k_new, v_new, np.array([7], np.int32), k_pool, v_pool)
    q = np.zeros((1, 1, H_q, D), np.float32)
    q[..., 0] = 2.0
    q[..., 1] = 3.0
    qb = (q.view(np.uint32) >> 16).astype(np.uint16)
    table = np.array([[7]], np.int32)
    out, lse = oracle.draft_decode_attn(qb, k_pool, v_pool, table, np.array([1], np.int32), 0.5)
    for h in range(H_q):
        g = h // G
        assert np.array_equal(out[0, 0, h], vals[0, g].astype(np.float64))
        assert lse[0, 0, h] == 0.5 * (2.0 if g == 0 else 3.0)
