"""Pins of the oracle's attention: closed forms and special cases of softmax
attention, the GQA head mapping, the "reduced table is the key set" property of
"Windowed-MTP: Removing the Full-Context Draft-KV Tax at Million-Token Context"
(§4 Mechanism: slot order and layout do not change scores), the windowed ==
native degeneration (§7), and the tree mask (§7 tree speculation).

Inputs are built so that every logit is known exactly by construction; the
expected values come from closed forms, not from re-running the oracle's own
formula.
"""
import math

import numpy as np
import pytest

import oracle


def bf16_bits(x):
    """float array -> bf16 bit patterns (round to nearest even)."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bits_to_f64(b):
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _pool(rows_k, rows_v):
    k = bf16_bits(np.asarray(rows_k, np.float32))
    v = bf16_bits(np.asarray(rows_v, np.float32))
    return k, v


def test_bf16_helper_roundtrip():
    x = np.array([0.0, 1.0, -2.5, 3.140625, 1e-3], np.float32)
    assert np.all(bits_to_f64(bf16_bits(x))[:4] == x[:4].astype(np.float64))


def test_single_key_returns_its_value():
    rng = np.random.default_rng(0)
    D = 16
    q = bf16_bits(rng.standard_normal((1, 1, 1, D)))
    k, v = _pool(rng.standard_normal((3, 1, D)), rng.standard_normal((3, 1, D)))
    out, lse = oracle.draft_decode_attn(q, k, v, np.array([[2]], np.int32),
                                        np.array([1], np.int32), 0.25)
    np.testing.assert_array_equal(out[0, 0, 0], bits_to_f64(v[2, 0]))
    want_lse = 0.25 * float(np.dot(bits_to_f64(q[0, 0, 0]), bits_to_f64(k[2, 0])))
    assert lse[0, 0, 0] == pytest.approx(want_lse, rel=1e-15, abs=1e-15)


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(1)
    D, L = 8, 37
    q = np.zeros((1, 1, 2, D), np.uint16)  # +0.0 in bf16
    k, v = _pool(rng.standard_normal((L, 1, D)), rng.integers(-8, 8, (L, 1, D)))
    table = rng.permutation(L).astype(np.int32)[None, :]
    out, lse = oracle.draft_decode_attn(q, k, v, table, np.array([L], np.int32), 1.0)
    mean = bits_to_f64(v[:, 0]).sum(axis=0) / L
    np.testing.assert_allclose(out[0, 0, 0], mean, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(out[0, 0, 1], mean, rtol=1e-14, atol=1e-14)
    assert lse[0, 0, 0] == pytest.approx(math.log(L), rel=1e-15)


def test_two_keys_sigmoid_weights():
    # q = e0, k1 = a*e0, k2 = 0  ->  logits (scale*a, 0): weight of key 1 is
    # sigmoid(scale*a); lse = log(1 + exp(scale*a)).
    D = 4
    for a, scale in [(2.0, 0.5), (-3.0, 1.0), (8.0, 0.125), (1.5, 2.0)]:
        q = np.zeros((1, 1, 1, D), np.uint16)
        q[0, 0, 0, 0] = bf16_bits([1.0])[0]
        k, v = _pool([[[a, 0, 0, 0]], [[0, 0, 0, 0]]],
                     [[[1, 0, 5, 0]], [[0, 1, 5, 2]]])
        out, lse = oracle.draft_decode_attn(q, k, v, np.array([[0, 1]], np.int32),
                                            np.array([2], np.int32), scale)
        w = 1.0 / (1.0 + math.exp(-scale * a))
        np.testing.assert_allclose(out[0, 0, 0], [w, 1 - w, 5.0, 2 * (1 - w)],
                                   rtol=1e-14, atol=1e-15)
        assert lse[0, 0, 0] == pytest.approx(math.log1p(math.exp(scale * a)), rel=1e-14)


def test_dominant_key_wins():
    # One logit 60 above the rest: its value comes back to within e^-60.
    D, L = 4, 9
    q = np.zeros((1, 1, 1, D), np.uint16)
    q[0, 0, 0, 1] = bf16_bits([1.0])[0]
    kr = np.zeros((L, 1, D), np.float32)
    kr[5, 0, 1] = 60.0
    vr = np.arange(L * D, dtype=np.float32).reshape(L, 1, D)
    k, v = _pool(kr, vr)
    out, lse = oracle.draft_decode_attn(q, k, v, np.arange(L, dtype=np.int32)[None],
                                        np.array([L], np.int32), 1.0)
    np.testing.assert_allclose(out[0, 0, 0], vr[5, 0], rtol=1e-20, atol=1e-20 + 64 * math.exp(-60))
    assert lse[0, 0, 0] == pytest.approx(60.0 + math.log1p((L - 1) * math.exp(-60)), rel=1e-15)


def test_gqa_contiguous_head_groups():
    # Reading R6: query head h reads KV head h // (H_q / H_kv).  Each KV head's
    # values are a constant, so every query head returns its group's constant.
    rng = np.random.default_rng(2)
    H_q, H_kv, D, L = 8, 2, 16, 11
    q = bf16_bits(rng.standard_normal((1, 1, H_q, D)))
    kr = rng.standard_normal((L, H_kv, D))
    vr = np.empty((L, H_kv, D))
    vr[:, 0, :] = 3.0
    vr[:, 1, :] = -7.0
    k, v = _pool(kr, vr)
    out, _ = oracle.draft_decode_attn(q, k, v, np.arange(L, dtype=np.int32)[None],
                                      np.array([L], np.int32), 0.3)
    for h in range(H_q):
        np.testing.assert_allclose(out[0, 0, h], 3.0 if h < 4 else -7.0, rtol=1e-14)


def test_key_order_and_layout_do_not_change_scores():
    # §4 Mechanism: RoPE is baked into cached keys, so where a key sits (slot,
    # table order) does not change its score.  Same keys, permuted table and
    # relocated slots: fp64 results agree to round-off.
    rng = np.random.default_rng(4)
    H_q, H_kv, D, L = 4, 2, 32, 300
    q = bf16_bits(rng.standard_normal((1, 1, H_q, D)))
    kr, vr = rng.standard_normal((L, H_kv, D)), rng.standard_normal((L, H_kv, D))
    k, v = _pool(kr, vr)
    out_a, lse_a = oracle.draft_decode_attn(q, k, v, np.arange(L, dtype=np.int32)[None],
                                            np.array([L], np.int32), 0.2)
    perm = rng.permutation(L)                    # table order
    place = rng.permutation(2 * L)[:L]           # physical slots in a bigger pool
    k2 = np.zeros((2 * L, H_kv, D), np.uint16)
    v2 = np.zeros((2 * L, H_kv, D), np.uint16)
    k2[place], v2[place] = k, v
    table = place[perm].astype(np.int32)[None]
    out_b, lse_b = oracle.draft_decode_attn(q, k2, v2, table, np.array([L], np.int32), 0.2)
    np.testing.assert_allclose(out_b, out_a, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse_b, lse_a, rtol=1e-13)


def test_empty_key_set():
    q = np.zeros((1, 1, 1, 8), np.uint16)
    k = np.zeros((1, 1, 8), np.uint16)
    out, lse = oracle.draft_decode_attn(q, k, k, np.zeros((1, 1), np.int32),
                                        np.array([0], np.int32), 1.0)
    assert np.all(out == 0) and lse[0, 0, 0] == -np.inf


def test_out_of_range_slot_is_an_error():
    q = np.zeros((1, 1, 1, 8), np.uint16)
    k = np.zeros((4, 1, 8), np.uint16)
    with pytest.raises(ValueError):
        oracle.draft_decode_attn(q, k, k, np.array([[0, 4]], np.int32),
                                 np.array([2], np.int32), 1.0)


def test_windowed_equals_full_inside_window():
    # §7: with S <= n_sink + W the windowed draft is the native draft; the
    # tables are identical, so the fp64 outputs are identical bit for bit.
    rng = np.random.default_rng(5)
    S, n_sink, W, H_q, H_kv, D = 1000, 64, 1024, 8, 2, 128
    rtt = rng.permutation(S + 1).astype(np.int32)[None]
    k = bf16_bits(rng.standard_normal((S + 1, H_kv, D)))
    v = bf16_bits(rng.standard_normal((S + 1, H_kv, D)))
    q = bf16_bits(rng.standard_normal((1, 1, H_q, D)))
    outs = []
    for windowed in (True, False):
        tb, ln = oracle.build_draft_indices(np.array([S], np.int32), 1, n_sink, W,
                                            depth=2, windowed=windowed,
                                            req_to_token=rtt, stride=S + 1)
        outs.append(oracle.draft_decode_attn(q, k, v, tb[0], ln[0], 1 / math.sqrt(D)))
    np.testing.assert_array_equal(outs[0][0], outs[1][0])
    np.testing.assert_array_equal(outs[0][1], outs[1][1])


def test_ring_layout_equals_unringed_layout():
    # §6 Memory / App. A: storing the draft KV in the ring changes only where
    # rows live.  Logical K/V per position, written once into a full-length
    # (un-ringed) pool and once into the ring; same logical table order, so
    # the fp64 results are identical.
    rng = np.random.default_rng(6)
    n_sink, W, d, H_q, H_kv, D = 4, 24, 3, 4, 2, 16
    S = 150
    R = n_sink + W + d
    Kl = bf16_bits(rng.standard_normal((S + d, H_kv, D)))
    Vl = bf16_bits(rng.standard_normal((S + d, H_kv, D)))
    flat_k, flat_v = Kl.copy(), Vl.copy()
    ring_base = 2 * R
    ring_k = np.zeros((4 * R, H_kv, D), np.uint16)
    ring_v = np.zeros((4 * R, H_kv, D), np.uint16)
    lo = S + 1 - W
    live = list(range(n_sink)) + list(range(lo, S + d - 1))
    for p in live:
        s = oracle.ring_slot(ring_base, p, 0, n_sink, W, d)
        ring_k[s], ring_v[s] = Kl[p], Vl[p]
    q = bf16_bits(rng.standard_normal((d - 1, 1, 1, H_q, D)))
    seq = np.array([S], np.int32)
    tb_flat, ln = oracle.build_draft_indices(seq, d - 1, n_sink, W, depth=d,
                                             req_to_token=np.arange(S + d, dtype=np.int32)[None])
    tb_ring, ln2 = oracle.build_draft_indices(seq, d - 1, n_sink, W, depth=d,
                                              ring_base=np.array([ring_base], np.int32))
    np.testing.assert_array_equal(ln, ln2)
    for j in range(d - 1):
        a = oracle.draft_decode_attn(q[j], flat_k, flat_v, tb_flat[j], ln[j], 0.25)
        b = oracle.draft_decode_attn(q[j], ring_k, ring_v, tb_ring[j], ln2[j], 0.25)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


# --------------------------------------------------------------------- tree
def _ring_pool_for_tree(rng, S_list, n_sink, W, d, k, H_kv, D):
    R = n_sink + W + d * k
    B = len(S_list)
    ring_base = (np.arange(B) * R).astype(np.int32)
    kp = bf16_bits(rng.standard_normal((B * R, H_kv, D)))
    vp = bf16_bits(rng.standard_normal((B * R, H_kv, D)))
    return ring_base, kp, vp


def test_tree_width_one_is_the_chain():
    # A tree of width 1 is the chain: node i is draft step i.
    rng = np.random.default_rng(8)
    n_sink, W, d, H_q, H_kv, D = 3, 20, 4, 4, 2, 16
    S_list = [2, 17, 30, 90]
    ring_base, kp, vp = _ring_pool_for_tree(rng, S_list, n_sink, W, d, 1, H_kv, D)
    B = len(S_list)
    q = bf16_bits(rng.standard_normal((B, d, H_q, D)))
    out_t, lse_t = oracle.tree_draft_attn(q, kp, vp, S_list, ring_base, n_sink, W,
                                          d, 1, 0.25)
    tb, ln = oracle.build_draft_indices(np.array(S_list, np.int32), d, n_sink, W,
                                        depth=d, ring_base=ring_base)
    for i in range(d):
        out_c, lse_c = oracle.draft_decode_attn(q[:, i:i + 1], kp, vp, tb[i], ln[i], 0.25)
        np.testing.assert_array_equal(out_t[:, i:i + 1], out_c)
        np.testing.assert_array_equal(lse_t[:, i:i + 1], lse_c)


def test_tree_mask_sees_only_own_path():
    # q = 0 makes every visible key weigh the same, so out = mean of the visible
    # V rows.  V is a one-hot marker per draft node (dims 0..k*d-1) and marker
    # dim k*d for every committed key, so out reveals exactly which nodes a
    # node sees: its own branch's depths 0..i, each with weight 1/L.
    rng = np.random.default_rng(9)
    n_sink, W, d, k, H_q, H_kv = 2, 10, 3, 3, 2, 1
    D = 16
    S = 40
    R = n_sink + W + d * k
    kp = bf16_bits(rng.standard_normal((R, H_kv, D)))
    vr = np.zeros((R, H_kv, D), np.float32)
    vr[:, 0, k * d] = 1.0
    for b in range(k):
        for i in range(d):
            s = oracle.ring_slot(0, S + i, b, n_sink, W, d, k)
            vr[s, 0, :] = 0.0
            vr[s, 0, b * d + i] = 1.0
    vp = bf16_bits(vr)
    q = np.zeros((1, k * d, H_q, D), np.uint16)
    out, lse = oracle.tree_draft_attn(q, kp, vp, [S], np.array([0], np.int32),
                                      n_sink, W, d, k, 1.0)
    for b in range(k):
        for i in range(d):
            t = b * d + i
            L = n_sink + W  # S + i + 1 > n_sink + W here
            want = np.zeros(D)
            for i2 in range(i + 1):
                want[b * d + i2] = 1.0 / L
            want[k * d] = (L - (i + 1)) / L
            np.testing.assert_allclose(out[0, t, 0], want, rtol=1e-14, atol=1e-15)
            assert lse[0, t, 0] == pytest.approx(math.log(L), rel=1e-15)
