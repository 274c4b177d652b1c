"""Pins of the oracle's attention-mass diagnostics (App. C, Table 12) against
closed forms and a hand-computed case (CPU)."""
import math

import numpy as np

import oracle


def _bf16(x):
    x = np.asarray(x, np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)  # truncated; every check reads these bits


def _f(u):
    return (np.asarray(u).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _setup(L, n_kept, seed, D=8, const_v=None, zero_q=False):
    rng = np.random.default_rng(seed)
    kp = _bf16(rng.integers(-4, 5, size=(L, 1, D)).astype(np.float32) / 4)
    if const_v is None:
        vp = _bf16(rng.integers(-4, 5, size=(L, 1, D)).astype(np.float32) / 4 + 1)
    else:
        vp = _bf16(np.broadcast_to(np.asarray(const_v, np.float32), (L, 1, D)).copy())
    q = _bf16(np.zeros((1, 1, 2, D), np.float32) if zero_q
              else rng.integers(-4, 5, size=(1, 1, 2, D)).astype(np.float32) / 4)
    perm = rng.permutation(L).astype(np.int32)
    tf = perm.reshape(1, L)
    tw = np.full((1, L), -1, np.int32)
    tw[0, :n_kept] = perm[L - n_kept:]  # kept = the last n_kept keys of the row
    return q, kp, vp, tf, np.array([L], np.int32), tw, np.array([n_kept], np.int32)


def test_everything_kept():
    q, kp, vp, tf, lf, tw, lw = _setup(20, 20, 1)
    a, p, t = oracle.attn_mass(q, kp, vp, tf, lf, tw, lw, 0.5)
    assert np.allclose(a, 1.0) and np.allclose(p, 0.0, atol=1e-14) and np.allclose(t, 0.0, atol=1e-14)


def test_constant_values():
    v = np.linspace(-1, 1, 8)
    q, kp, vp, tf, lf, tw, lw = _setup(30, 7, 2, const_v=v)
    a, p, t = oracle.attn_mass(q, kp, vp, tf, lf, tw, lw, 0.5)
    assert np.allclose(p, 0.0, atol=1e-14)
    assert np.allclose(t, 1.0 - a, atol=1e-12)


def test_uniform_logits():
    q, kp, vp, tf, lf, tw, lw = _setup(40, 10, 3, zero_q=True)
    a, p, t = oracle.attn_mass(q, kp, vp, tf, lf, tw, lw, 0.5)
    assert np.allclose(a, 10 / 40)


def test_tail_identity_and_bounds():
    for seed in range(4):
        q, kp, vp, tf, lf, tw, lw = _setup(50, 13, 10 + seed)
        a, p, t = oracle.attn_mass(q, kp, vp, tf, lf, tw, lw, 0.75)
        assert np.all((a >= 0) & (a <= 1))
        # o_full = a o_win + o_far: the far share from the two read-outs alone
        K, V, Q = _f(kp[:, 0]), _f(vp[:, 0]), _f(q[0, 0])
        for h in range(2):
            z = 0.75 * K[tf[0]] @ Q[h]
            e = np.exp(z - z.max())
            kept = np.isin(tf[0], tw[0, :lw[0]])
            o_full = (e[:, None] * V[tf[0]]).sum(0) / e.sum()
            o_win = (e[kept][:, None] * V[tf[0]][kept]).sum(0) / e[kept].sum()
            ident = np.linalg.norm(o_full - a[0, 0, h] * o_win) / np.linalg.norm(o_full)
            assert math.isclose(t[0, 0, h], ident, rel_tol=1e-12, abs_tol=1e-14)


def test_two_keys_by_hand():
    # keys k0 = (1, 0..), k1 = (0, ..); q = (2, 0..); kept = {k1}; scale 1
    D = 8
    kp = _bf16(np.array([[[1] + [0] * 7], [[0] * 8]], np.float32))
    vp = _bf16(np.array([[[1] + [0] * 7], [[0, 1] + [0] * 6]], np.float32))
    q = _bf16(np.array([[[[2] + [0] * 7, [2] + [0] * 7]]], np.float32))
    tf = np.array([[0, 1]], np.int32)
    tw = np.array([[1, -1]], np.int32)
    a, p, t = oracle.attn_mass(q, kp, vp, tf, np.array([2], np.int32), tw, np.array([1], np.int32), 1.0)
    p0 = math.exp(2) / (math.exp(2) + 1)  # softmax weight of the far key
    assert math.isclose(a[0, 0, 0], 1 - p0, rel_tol=1e-12)
    o_full = np.array([p0, 1 - p0])
    assert math.isclose(p[0, 0, 0], np.linalg.norm(o_full - np.array([0, 1])) / np.linalg.norm(o_full),
                        rel_tol=1e-12)
    assert math.isclose(t[0, 0, 0], p0 / np.linalg.norm(o_full), rel_tol=1e-12)


# --- the far keys: the complement of the keep rule ("Windowed-MTP", §5 "A
# partition-function view": Z = Z_w + Z_far over the kept and the dropped keys)

def test_far_positions_closed_form_and_partition():
    for n_sink, W in [(0, 1), (1, 1), (2, 3), (4, 16), (64, 100), (5, 7)]:
        for s_kv in range(0, 200):
            far = oracle.far_positions(s_kv, n_sink, W)
            expect = list(range(n_sink, s_kv - W)) if s_kv > n_sink + W else []
            assert far.tolist() == expect, (s_kv, n_sink, W)
            kept = oracle.keep(s_kv, n_sink, W).tolist()
            assert sorted(kept + far.tolist()) == list(range(s_kv))  # disjoint cover of [0, s_kv)


def test_far_table_through_the_page_table():
    rng = np.random.default_rng(5)
    n_sink, W, gamma = 3, 10, 3
    S_list = [0, 5, 13, 14, 40]
    cap = max(S_list) + gamma
    rtt = np.stack([rng.permutation(1000)[:cap] for _ in S_list]).astype(np.int32)
    table, lens = oracle.build_far_indices(np.array(S_list, np.int32), gamma, n_sink, W, rtt)
    for j in range(gamma):
        for b, S in enumerate(S_list):
            kv = S + j + 1
            pos = np.arange(n_sink, kv - W) if kv > n_sink + W else np.arange(0)
            assert lens[j, b] == len(pos)
            assert np.array_equal(table[j, b, :len(pos)], rtt[b, pos])
            assert np.all(table[j, b, len(pos):] == -1)


def test_window_and_far_attention_merge_to_the_full_attention():
    """The decomposition the GPU diagnostics use: with a = Z_w / Z and
    b = Z_far / Z from the two log partition functions, a o_win + b o_far is
    the full-context output and log(e^lse_win + e^lse_far) its lse."""
    rng = np.random.default_rng(11)
    n_sink, W, gamma, H_q, H_kv, D = 2, 9, 2, 4, 2, 8
    S = 60
    pool = S + gamma
    kp = _bf16(rng.standard_normal((pool, H_kv, D)))
    vp = _bf16(rng.standard_normal((pool, H_kv, D)))
    q = _bf16(rng.standard_normal((1, 1, H_q, D)))
    rtt = rng.permutation(pool).astype(np.int32).reshape(1, -1)
    seq = np.array([S], np.int32)
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=gamma + 1, req_to_token=rtt)
    tf, lf = oracle.build_draft_indices(seq, windowed=False, stride=pool, **kw)
    tw, lw = oracle.build_draft_indices(seq, windowed=True, stride=n_sink + W, **kw)
    tr, lr = oracle.build_far_indices(seq, gamma, n_sink, W, rtt)
    for j in range(gamma):
        of, lsf = oracle.draft_decode_attn(q, kp, vp, tf[j], lf[j], 0.4)
        ow, lsw = oracle.draft_decode_attn(q, kp, vp, tw[j], lw[j], 0.4)
        o_r, lsr = oracle.draft_decode_attn(q, kp, vp, tr[j], lr[j], 0.4)
        a = 1.0 / (1.0 + np.exp(lsr - lsw))
        b = 1.0 / (1.0 + np.exp(lsw - lsr))
        merged = a[..., None] * ow + b[..., None] * o_r
        assert np.allclose(merged, of, rtol=1e-12, atol=1e-14)
        assert np.allclose(np.logaddexp(lsw, lsr), lsf, rtol=1e-13, atol=1e-13)
        # and the diagnostics' tail fraction is b ||o_far|| / ||o_full||
        ra, rp, rt = oracle.attn_mass(q, kp, vp, tf[j], lf[j], tw[j], lw[j], 0.4)
        nf = np.linalg.norm(of, axis=-1)
        assert np.allclose(rt, b * np.linalg.norm(o_r, axis=-1) / nf, rtol=1e-11)
        assert np.allclose(rp, b * np.linalg.norm(o_r - ow, axis=-1) / nf, rtol=1e-11)
        assert np.allclose(ra, a, rtol=1e-12)
