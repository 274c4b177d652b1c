"""Pins of the oracle's pruned draft prefill ("Windowed-MTP", §7 "Prefill
sparsification and TTFT"): the kept prompt positions are the keep rule at
kv length S, and filling the ring with the draft KV of only those positions
loses nothing -- every windowed draft step then attends exactly what it
attends over the full-length draft pool (bit for bit in fp64).  CPU only."""
import numpy as np
import pytest

import oracle

N_SINK, W, DEPTH = 4, 16, 3
H_q, H_kv, D = 4, 2, 8


def _bf16(x):
    x = np.asarray(x, np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("S", [0, 1, 3, 4, 10, 20, 21, 22, 57, 300])
def test_kept_positions_are_sinks_then_window(S):
    (pos,) = oracle.prefill_keep_positions([S], N_SINK, W)
    if S <= N_SINK + W:
        expect = list(range(S))
    else:
        expect = list(range(N_SINK)) + list(range(S - W, S))
    assert pos.tolist() == expect


@pytest.mark.parametrize("tree_k", [1, 4])
def test_pruned_ring_fill_is_lossless_for_every_draft_step(tree_k):
    rng = np.random.default_rng(7 + tree_k)
    S_list = [2, 19, 20, 21, 57, 300]
    B, gamma = len(S_list), DEPTH - 1
    scale = 0.35
    # the full draft KV of each prompt, and the draft steps' own rows
    K = [_bf16(rng.integers(-8, 9, size=(S, H_kv, D)) / 4) for S in S_list]
    V = [_bf16(rng.integers(-8, 9, size=(S, H_kv, D)) / 4) for S in S_list]
    kn = _bf16(rng.integers(-8, 9, size=(gamma, B, H_kv, D)) / 4)
    vn = _bf16(rng.integers(-8, 9, size=(gamma, B, H_kv, D)) / 4)
    q = _bf16(rng.standard_normal((gamma, B, 1, H_q, D)))

    # (a) unpruned: a full-length paged pool holding every prompt position
    cap = max(S_list) + gamma
    full_k = np.zeros((B * cap, H_kv, D), np.uint16)
    full_v = np.zeros_like(full_k)
    rtt = np.arange(B * cap, dtype=np.int32).reshape(B, cap)
    for b, S in enumerate(S_list):
        oracle.append_kv(K[b], V[b], rtt[b, :S], full_k, full_v)

    # (b) pruned: rings filled from the kept positions only
    R = N_SINK + W + DEPTH * tree_k
    ring_base = np.arange(B, dtype=np.int32) * R
    ring_k = np.full((B * R, H_kv, D), 0x7FC0, np.uint16)  # NaN: a read of an unfilled slot shows
    ring_v = ring_k.copy()
    stride = N_SINK + W
    rows_k = np.zeros((B, stride, H_kv, D), np.uint16)
    rows_v = np.zeros_like(rows_k)
    for b, pos in enumerate(oracle.prefill_keep_positions(S_list, N_SINK, W)):
        rows_k[b, :len(pos)] = K[b][pos]
        rows_v[b, :len(pos)] = V[b][pos]
    oracle.ring_fill(rows_k, rows_v, S_list, ring_base, N_SINK, W, DEPTH, ring_k, ring_v, tree_k=tree_k)

    seq = np.array(S_list, np.int32)
    kw = dict(gamma=gamma, n_sink=N_SINK, window=W, depth=DEPTH, tree_k=tree_k, windowed=True)
    t_full, l_full = oracle.build_draft_indices(seq, req_to_token=rtt, stride=N_SINK + W, **kw)
    t_ring, l_ring = oracle.build_draft_indices(seq, ring_base=ring_base, stride=N_SINK + W, **kw)
    assert np.array_equal(l_full, l_ring)
    for j in range(gamma):
        pos = seq + j
        oracle.append_kv(kn[j], vn[j], rtt[np.arange(B), pos], full_k, full_v)
        oracle.append_kv(kn[j], vn[j],
                         oracle.ring_map(ring_base, pos, np.arange(B, dtype=np.int32), N_SINK, W, DEPTH,
                                         tree_k), ring_k, ring_v)
        o_f, l_f = oracle.draft_decode_attn(q[j], full_k, full_v, t_full[j], l_full[j], scale)
        o_r, l_r = oracle.draft_decode_attn(q[j], ring_k, ring_v, t_ring[j], l_ring[j], scale)
        assert np.all(np.isfinite(o_r))
        assert np.array_equal(o_f, o_r) and np.array_equal(l_f, l_r), f"step {j}"


def test_ring_fill_writes_only_the_kept_slots():
    S_list = [3, 40]
    R = N_SINK + W + DEPTH
    ring_base = np.array([R, 0], np.int32)
    k_pool = np.zeros((2 * R, 1, D), np.uint16)
    v_pool = np.zeros_like(k_pool)
    rows = np.ones((2, N_SINK + W, 1, D), np.uint16)
    oracle.ring_fill(rows, rows, S_list, ring_base, N_SINK, W, DEPTH, k_pool, v_pool)
    written = set(np.nonzero(k_pool[:, 0, 0])[0].tolist())
    expect = set(range(R, R + 3))  # request 0: positions 0..2 at their own offsets
    for p in list(range(N_SINK)) + list(range(40 - W, 40)):
        expect.add(oracle.ring_slot(0, p, 0, N_SINK, W, DEPTH))
    assert written == expect
    assert len(expect) == 3 + N_SINK + W
