"""Pins of the oracle's draft-extend functions (CPU).

The union of the keep sets of draft steps 0..n-1 has a closed form (sinks
then one contiguous run, or a prefix) that the App. A keep rule implies; a
one-token extend is exactly one draft step; rows past a request's count are
empty."""
import numpy as np

import oracle


def _closed_form(S, n, n_sink, W, windowed):
    if n == 0:
        return []
    if windowed and S + 1 > n_sink + W:
        return list(range(n_sink)) + list(range(S + 1 - W, S + n))
    return list(range(S + n))


def test_union_matches_closed_form():
    n_sink, W = 4, 9
    for windowed in (True, False):
        for S in list(range(0, 30)) + [100, 257]:
            for n in range(0, 6):
                rtt = np.arange(400, dtype=np.int32).reshape(1, 400)
                t, l = oracle.build_extend_indices(np.array([S], np.int32), np.array([n], np.int32),
                                                   n_sink, W, 7, windowed=windowed, req_to_token=rtt)
                assert t[0, :l[0]].tolist() == _closed_form(S, n, n_sink, W, windowed), (S, n, windowed)


def test_union_on_the_ring_is_the_ring_map_of_the_union():
    n_sink, W, d = 4, 9, 7
    rb = np.array([1000], np.int32)
    for S in (0, 3, 12, 13, 14, 50):
        for n in (1, 3, 7):
            t, l = oracle.build_extend_indices(np.array([S], np.int32), np.array([n], np.int32),
                                               n_sink, W, d, ring_base=rb)
            pos = np.array(_closed_form(S, n, n_sink, W, True), np.int32)
            ref = oracle.ring_map(rb, pos, np.zeros(pos.size, np.int32), n_sink, W, d)
            assert t[0, :l[0]].tolist() == ref.tolist(), (S, n)


def test_one_token_extend_is_one_draft_step_and_empty_rows():
    rng = np.random.default_rng(5)
    H_q, H_kv, D, n_sink, W = 4, 2, 16, 4, 9
    num_slots = 200
    kp = rng.integers(0, 1 << 14, size=(num_slots, H_kv, D), dtype=np.uint16) & 0x3FFF
    vp = rng.integers(0, 1 << 14, size=(num_slots, H_kv, D), dtype=np.uint16) & 0x3FFF
    rtt = np.arange(2 * 100, dtype=np.int32).reshape(2, 100)
    S = np.array([40, 7], np.int32)
    q = rng.integers(0, 1 << 14, size=(2, 3, H_q, D), dtype=np.uint16) & 0x3FFF
    out, lse = oracle.draft_extend_attn(q, kp, vp, S, np.array([1, 0], np.int32), n_sink, W, 0.25,
                                        req_to_token=rtt)
    tab, ln = oracle.build_draft_indices(S, 1, n_sink, W, 2, req_to_token=rtt)
    ref, rl = oracle.draft_decode_attn(q[:, :1], kp, vp, tab[0], ln[0], 0.25)
    assert np.array_equal(out[0, 0], ref[0, 0]) and np.array_equal(lse[0, 0], rl[0, 0])
    assert np.all(out[0, 1:] == 0) and np.all(np.isneginf(lse[0, 1:]))
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))


def test_extend_rows_match_brute_force_softmax():
    # Row t against a direct softmax over keep(S+t+1) on tiny inputs.
    rng = np.random.default_rng(6)
    H_q, H_kv, D, n_sink, W = 2, 1, 8, 2, 5
    num_slots = 64
    vals = rng.standard_normal((num_slots, H_kv, D)).astype(np.float32)
    kp = (vals.view(np.uint32) >> 16).astype(np.uint16)
    vals2 = rng.standard_normal((num_slots, H_kv, D)).astype(np.float32)
    vp = (vals2.view(np.uint32) >> 16).astype(np.uint16)
    qv = rng.standard_normal((1, 4, H_q, D)).astype(np.float32)
    q = (qv.view(np.uint32) >> 16).astype(np.uint16)
    rtt = rng.permutation(num_slots).astype(np.int32).reshape(1, num_slots)
    S, n = 20, 4
    out, lse = oracle.draft_extend_attn(q, kp, vp, np.array([S], np.int32), np.array([n], np.int32),
                                        n_sink, W, 0.5, req_to_token=rtt)
    f = lambda u: (u.astype(np.uint32) << 16).view(np.float32).astype(np.float64)  # noqa: E731
    K, V, Q = f(kp), f(vp), f(q)
    for t in range(n):
        kv = S + t + 1
        pos = list(range(n_sink)) + list(range(kv - W, kv))
        slots = rtt[0, pos]
        for h in range(H_q):
            g = h // (H_q // H_kv)
            s = 0.5 * (K[slots, g] @ Q[0, t, h])
            w = np.exp(s - s.max())
            ref = (w[:, None] * V[slots, g]).sum(0) / w.sum()
            assert np.allclose(out[0, t, h], ref, rtol=1e-12, atol=1e-12)
            assert np.isclose(lse[0, t, h], s.max() + np.log(w.sum()), rtol=1e-12)


def test_chain_extend_equals_tree_attention_with_one_branch():
    # an extend of n = d tokens over the ring is the tree attention with
    # k = 1 and depth d (node i at position S + i sees keep(S + i + 1) with
    # the draft positions of its own, single branch): the equivalence the
    # library's tensor-core extend path is built on
    rng = np.random.default_rng(17)
    H_q, H_kv, D, n_sink, W, d = 4, 2, 16, 4, 9, 5
    R = n_sink + W + d
    S_list = np.array([0, 3, 12, 13, 14, 50, 200], np.int32)
    B = S_list.size
    rb = (np.arange(B, dtype=np.int32) * R + 3).astype(np.int32)
    num_slots = B * R + 3
    kp = rng.integers(0, 1 << 14, size=(num_slots, H_kv, D), dtype=np.uint16) & 0x3FFF
    vp = rng.integers(0, 1 << 14, size=(num_slots, H_kv, D), dtype=np.uint16) & 0x3FFF
    q = rng.integers(0, 1 << 14, size=(B, d, H_q, D), dtype=np.uint16) & 0x3FFF
    xo, xl = oracle.draft_extend_attn(q, kp, vp, S_list, np.full(B, d, np.int32), n_sink, W, 0.3,
                                      ring_base=rb, depth=d)
    to, tl = oracle.tree_draft_attn(q, kp, vp, S_list, rb, n_sink, W, d, 1, 0.3)
    assert np.all(np.isfinite(xo)) and np.all(np.isfinite(to))
    assert np.allclose(xo, to, rtol=1e-12, atol=1e-12) and np.allclose(xl, tl, rtol=1e-12, atol=1e-12)
    # the comparison discriminates: a tree with another window gives other rows
    so, _ = oracle.tree_draft_attn(q, kp, vp, S_list, rb, n_sink, W - 1, d, 1, 0.3)
    assert not np.allclose(so[S_list > n_sink + W], to[S_list > n_sink + W], rtol=1e-12, atol=1e-12)
