"""Pins of the oracle's integer parts: key selection, index tables, ring slots,
and the acceptance-length formula.

Each test checks the oracle against something other than itself: the block
table printed in "arXiv'26 | Wind-MTP" (marsggbo.github.io) §3.1, a set
predicate that describes the same key set in one line, closed forms, and
brute-force invariants of the ring of "Windowed-MTP: Removing the Full-Context
Draft-KV Tax at Million-Token Context" (App. A; §6 Memory; §7 tree).
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = rest
    return vals


def _ranges(tokens):
    parts = []
    for tok in tokens:
        lo, hi = (int(x) for x in tok.split("-"))
        parts.append(np.arange(lo, hi + 1, dtype=np.int64))
    return np.concatenate(parts)


def test_worked_example_block_table():
    g = _read_golden("worked_example_block_table.txt")
    S, n_sink, W = int(g["S"][0]), int(g["n_sink"][0]), int(g["W"][0])
    win = oracle.keep(S, n_sink, W, windowed=True) + 1  # page prints 1-based ids
    nat = oracle.keep(S, n_sink, W, windowed=False) + 1
    np.testing.assert_array_equal(win, _ranges(g["windowed"]))
    np.testing.assert_array_equal(nat, _ranges(g["native"]))
    assert win.size == n_sink + W == 4096


@pytest.mark.parametrize("n_sink", [0, 1, 3, 8])
@pytest.mark.parametrize("W", [1, 2, 5, 16, 64])
def test_keep_matches_set_predicate(n_sink, W):
    # One predicate covers both branches of the pseudocode: a position is kept
    # iff it is a sink or one of the last W.  Order is ascending, no repeats.
    for s_kv in range(0, 200):
        got = oracle.keep(s_kv, n_sink, W, windowed=True)
        want = np.array([p for p in range(s_kv) if p < n_sink or p >= s_kv - W],
                        dtype=np.int64)
        np.testing.assert_array_equal(got, want)
        assert got.size == min(s_kv, n_sink + W)
        if s_kv:
            assert got[-1] == s_kv - 1  # the step's own token is always seen


def test_windowed_degenerates_to_full():
    # §7 "when to window": for contexts inside the window the windowed draft is
    # the native draft.
    for s_kv in range(0, 1089):
        np.testing.assert_array_equal(oracle.keep(s_kv, 64, 1024, True),
                                      oracle.keep(s_kv, 64, 1024, False))


def test_build_draft_indices_paged():
    rng = np.random.default_rng(7)
    n_sink, W, gamma = 4, 16, 3
    seq_lens = np.array([5, 17, 20, 21, 60], dtype=np.int32)
    B = seq_lens.size
    max_ctx = 80
    rtt = np.stack([rng.permutation(1000)[:max_ctx] for _ in range(B)]).astype(np.int32)
    pool_idx = np.array([4, 2, 0, 1, 3], dtype=np.int32)
    for windowed in (True, False):
        table, lens = oracle.build_draft_indices(
            seq_lens, gamma, n_sink, W, depth=gamma + 1, windowed=windowed,
            req_to_token=rtt, req_pool_idx=pool_idx, stride=max_ctx)
        for j in range(gamma):
            for b in range(B):
                kv = int(seq_lens[b]) + j + 1
                n = int(lens[j, b])
                assert n == (min(kv, n_sink + W) if windowed else kv)
                row = rtt[pool_idx[b]]
                got = table[j, b, :n]
                # the step's own token (position S + j) closes the list
                assert got[-1] == row[kv - 1]
                # every entry is the slot of a kept position, in ascending order
                pos = np.array([int(np.where(row == s)[0][0]) for s in got])
                assert np.all(np.diff(pos) > 0)
                assert set(pos.tolist()) == {p for p in range(kv)
                                             if not windowed or p < n_sink or p >= kv - W}
                assert np.all(table[j, b, n:] == -1)


def test_build_draft_indices_capacity_error():
    with pytest.raises(ValueError):
        oracle.build_draft_indices(np.array([100], np.int32), 1, 4, 16, depth=2,
                                   windowed=False,
                                   req_to_token=np.zeros((1, 200), np.int32),
                                   stride=50)


def test_worked_example_through_builder():
    # A draft step whose kv length is 1,000,000 (committed S = 999,999, step 0)
    # with block ids = position + 1 reproduces the page's windowed table.
    g = _read_golden("worked_example_block_table.txt")
    S = int(g["S"][0])
    rtt = (np.arange(S + 8, dtype=np.int32) + 1)[None, :]
    table, lens = oracle.build_draft_indices(
        np.array([S - 1], np.int32), 1, int(g["n_sink"][0]), int(g["W"][0]),
        depth=7, windowed=True, req_to_token=rtt, stride=4096)
    np.testing.assert_array_equal(table[0, 0, :lens[0, 0]],
                                  _ranges(g["windowed"]).astype(np.int32))


# ---------------------------------------------------------------- ring slots
def test_ring_agrees_with_literal_formula_below_modulus():
    # App. A / blog §3.1: slot = ring_base + pos mod (n_sink + W + d).  Below the
    # modulus this is ring_base + pos, which the pinned-sink reading reproduces
    # for the chain (k = 1) and for branch 0 of a tree.
    for (n_sink, W, d, k) in [(64, 4032, 7, 1), (64, 1024, 7, 4), (3, 8, 3, 2)]:
        R = n_sink + W + d * k
        for p in range(R):
            assert oracle.ring_slot(1000, p, 0, n_sink, W, d, k) == 1000 + p


def _live_positions(S, n_sink, W, d, k):
    """Every (position, branch) a decode step can touch: sinks, the committed
    positions any draft step's window reads, and each branch's d draft nodes."""
    live = [(p, 0) for p in range(min(n_sink, S))]
    lo = max(n_sink, S + 1 - W) if S + 1 > n_sink + W else n_sink
    live += [(p, 0) for p in range(lo, S)]
    live += [(S + i, b) for b in range(k) for i in range(d)]
    return live


@pytest.mark.parametrize("n_sink,W,d,k", [(3, 8, 3, 1), (3, 8, 3, 2), (0, 5, 2, 4),
                                          (2, 4, 4, 3), (64, 1024, 7, 4)])
def test_ring_live_tokens_never_collide(n_sink, W, d, k):
    R = n_sink + W + d * k
    S_values = range(1, 3 * R) if R < 200 else range(R - 40, R + 400)
    for S in S_values:
        live = _live_positions(S, n_sink, W, d, k)
        slots = [oracle.ring_slot(0, p, b, n_sink, W, d, k) for p, b in live]
        assert len(set(slots)) == len(slots), (S, live)
        assert min(slots) >= 0 and max(slots) < R


def test_literal_modulus_overwrites_sinks():
    # Why the sinks are pinned (reading R4): taken literally, pos mod
    # (n_sink + W + d) sends live window positions onto the sink slots once
    # the context passes the ring size.
    n_sink, W, d = 64, 4032, 7
    R = n_sink + W + d
    S = 4200
    live = _live_positions(S, n_sink, W, d, 1)
    literal = [p % R for p, _ in live]
    assert len(set(literal)) < len(literal)
    pinned = [oracle.ring_slot(0, p, b, n_sink, W, d, 1) for p, b in live]
    assert len(set(pinned)) == len(pinned)


def test_ring_map_vector_form():
    rb = np.array([0, 5000, 12000], np.int32)
    pos = np.array([0, 63, 64, 4102, 4103, 999999, 5, 70], np.int32)
    req = np.array([0, 0, 1, 1, 2, 2, 1, 2], np.int32)
    br = np.array([0, 0, 0, 1, 2, 3, 0, 1], np.int32)
    got = oracle.ring_map(rb, pos, req, 64, 4032, 7, 4, branch=br)
    want = [oracle.ring_slot(int(rb[r]), int(p), int(b), 64, 4032, 7, 4)
            for p, r, b in zip(pos, req, br)]
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------ acceptance length
def test_acceptance_length_telescopes():
    # Eq. (4) against the telescoping identity AL = 1 + E[N] (N = accepted
    # drafts per step), on random histograms.
    rng = np.random.default_rng(3)
    for gamma in (1, 2, 4, 6, 8):
        for _ in range(50):
            H = rng.integers(0, 1000, size=gamma + 1).astype(np.float64)
            if H.sum() == 0:
                continue
            alpha, al = oracle.acceptance_length(H)
            mean_n = float((np.arange(gamma + 1) * H).sum() / H.sum())
            assert al == pytest.approx(1.0 + mean_n, rel=1e-12, abs=1e-12)
            assert 1.0 <= al <= gamma + 1
            assert np.all((alpha >= 0) & (alpha <= 1))


def test_acceptance_alpha_is_conditional_frequency():
    # alpha_j = Pr[accept j | reached j], measured by brute force on samples.
    rng = np.random.default_rng(11)
    gamma = 6
    N = rng.binomial(gamma, 0.6, size=20000)
    H = np.bincount(N, minlength=gamma + 1).astype(np.float64)
    alpha, _ = oracle.acceptance_length(H)
    for j in range(1, gamma + 1):
        reached = (N >= j - 1).sum()
        assert alpha[j - 1] == pytest.approx((N >= j).sum() / reached, rel=1e-12)


def test_acceptance_extremes():
    _, al = oracle.acceptance_length([0, 0, 0, 0, 0, 0, 5.0])
    assert al == 7.0
    _, al = oracle.acceptance_length([9.0, 0, 0, 0, 0, 0, 0])
    assert al == 1.0
