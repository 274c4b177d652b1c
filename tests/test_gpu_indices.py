"""GPU parity of the draft KV-index builder and the ring mapper / KV append
against the oracle: bit-exact (integer and byte work)."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import synth
from wmtp_testutil import bits, host_i32

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    wm.build()
    wm.load()
    wm.device_error(clear=True)
    yield
    assert wm.device_error(clear=True) == 0


def _compare_tables(tg, lg, tr, lr):
    tg, lg = host_i32(tg), host_i32(lg)
    np.testing.assert_array_equal(lg, lr)
    for j in range(lr.shape[0]):
        for b in range(lr.shape[1]):
            n = int(lr[j, b])
            np.testing.assert_array_equal(tg[j, b, :n], tr[j, b, :n], err_msg=f"step {j} req {b}")


@pytest.mark.parametrize("windowed", [True, False])
@pytest.mark.parametrize("layout", ["paged", "ring"])
@pytest.mark.parametrize("n_sink,W,gamma", [(0, 1, 1), (3, 8, 3), (4, 16, 6), (64, 1024, 2)])
def test_indices_small(windowed, layout, n_sink, W, gamma):
    rng = np.random.default_rng(n_sink * 100 + W + gamma)
    seq = np.array([0, 1, n_sink, n_sink + W - 1, n_sink + W, n_sink + W + 5, 3 * (n_sink + W) + 7,
                    int(rng.integers(1, 5000))], np.int32)
    B = seq.size
    d = gamma + 1
    max_ctx = int(seq.max()) + gamma + 1
    stride = (n_sink + W) if windowed else max_ctx
    kw = dict(gamma=gamma, n_sink=n_sink, window=W, depth=d, windowed=windowed, stride=stride)
    if layout == "paged":
        rtt = np.stack([rng.permutation(10 * max_ctx)[:max_ctx] for _ in range(B)]).astype(np.int32)
        pidx = rng.permutation(B).astype(np.int32)
        rtt_g = torch.from_numpy(rtt).to(DEV)
        tg, lg = wm.build_draft_indices(torch.from_numpy(seq).to(DEV), req_to_token=rtt_g,
                                        req_pool_idx=torch.from_numpy(pidx).to(DEV), **kw)
        tr, lr = oracle.build_draft_indices(seq, req_to_token=rtt, req_pool_idx=pidx, **kw)
    else:
        rb = (np.arange(B) * (n_sink + W + d) * 3 + 11).astype(np.int32)
        tg, lg = wm.build_draft_indices(torch.from_numpy(seq).to(DEV),
                                        ring_base=torch.from_numpy(rb).to(DEV), **kw)
        tr, lr = oracle.build_draft_indices(seq, ring_base=rb, **kw)
    _compare_tables(tg, lg, tr, lr)


def test_indices_tiny_windowed_workload():
    # S = 8192 and S = 1000, n_sink 64, W 1024, one draft step, permuted pool.
    for S in (8192, 1000):
        rtt = synth.permutation(S + 1, 1000, "cpu").numpy()[None, :]
        for windowed in (True, False):
            kw = dict(gamma=1, n_sink=64, window=1024, depth=2, windowed=windowed, stride=S + 1)
            tg, lg = wm.build_draft_indices(torch.tensor([S], dtype=torch.int32, device=DEV),
                                            req_to_token=torch.from_numpy(rtt).to(DEV), **kw)
            tr, lr = oracle.build_draft_indices(np.array([S], np.int32), req_to_token=rtt, **kw)
            _compare_tables(tg, lg, tr, lr)


@pytest.mark.parametrize("S", [131072, 1048576])
def test_indices_long_context(S):
    # gamma = 6 tables at 131K and 1M, full and windowed, permuted pool.
    rtt = synth.permutation(S + 8, 1002, DEV).view(1, -1)
    rtt_h = host_i32(rtt)
    seq = np.array([S], np.int32)
    for windowed in (True, False):
        kw = dict(gamma=6, n_sink=64, window=4032, depth=7, windowed=windowed,
                  stride=4096 if windowed else S + 8)
        tg, lg = wm.build_draft_indices(torch.from_numpy(seq).to(DEV), req_to_token=rtt, **kw)
        tr, lr = oracle.build_draft_indices(seq, req_to_token=rtt_h, **kw)
        _compare_tables(tg, lg, tr, lr)


def test_indices_batched_ring():
    lens = synth.uniform_lengths(6, 900_000, 1_048_576, 1003)
    R = 64 + 4032 + 7
    rb = np.array(synth.ring_bases(6, R, 12, 1003), np.int32)
    seq = np.array(lens, np.int32)
    kw = dict(gamma=6, n_sink=64, window=4032, depth=7, windowed=True, stride=4096)
    tg, lg = wm.build_draft_indices(torch.from_numpy(seq).to(DEV),
                                    ring_base=torch.from_numpy(rb).to(DEV), **kw)
    tr, lr = oracle.build_draft_indices(seq, ring_base=rb, **kw)
    _compare_tables(tg, lg, tr, lr)


def test_indices_overflow_is_latched():
    seq = torch.tensor([100], dtype=torch.int32, device=DEV)
    rtt = torch.arange(200, dtype=torch.int32, device=DEV).view(1, -1)
    tg, lg = wm.build_draft_indices(seq, gamma=1, n_sink=4, window=16, depth=2, windowed=False,
                                    req_to_token=rtt, stride=50)
    assert int(lg[0, 0]) == 101
    assert wm.device_error(clear=True) == 2
    np.testing.assert_array_equal(host_i32(tg)[0, 0], np.arange(50))


# ------------------------------------------------------------------ ring map
@pytest.mark.parametrize("n_sink,W,d,k", [(64, 4032, 7, 1), (64, 1024, 7, 4), (3, 8, 3, 2), (0, 5, 2, 4)])
def test_ring_map_matches_oracle(n_sink, W, d, k):
    rng = np.random.default_rng(n_sink + W + d + k)
    n = 5000
    nreq = 5
    rb = (rng.permutation(nreq) * (n_sink + W + d * k)).astype(np.int32)
    pos = rng.integers(0, 3_000_000, n).astype(np.int32)
    pos[:200] = rng.integers(0, max(n_sink, 1) + 2 * d, 200)  # the sink edge
    req = rng.integers(0, nreq, n).astype(np.int32)
    br = rng.integers(0, k, n).astype(np.int32)
    got = wm.ring_map(torch.from_numpy(rb).to(DEV), torch.from_numpy(pos).to(DEV),
                      torch.from_numpy(req).to(DEV), n_sink, W, d, k,
                      branch=torch.from_numpy(br).to(DEV))
    want = oracle.ring_map(rb, pos, req, n_sink, W, d, k, branch=br)
    np.testing.assert_array_equal(host_i32(got), want)


def test_append_kv_matches_oracle():
    H_kv, D, n, num_slots = 2, 256, 37, 500
    kp = synth.normal_bf16((num_slots, H_kv, D), 1, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 2, DEV)
    kn = synth.normal_bf16((n, H_kv, D), 3, DEV)
    vn = synth.normal_bf16((n, H_kv, D), 4, DEV)
    slots = synth.permutation(num_slots, 5, DEV)[:n].contiguous()
    kp_h, vp_h = bits(kp), bits(vp)
    oracle.append_kv(bits(kn), bits(vn), host_i32(slots), kp_h, vp_h)
    wm.append_kv(kn, vn, slots, kp, vp)
    np.testing.assert_array_equal(bits(kp), kp_h)
    np.testing.assert_array_equal(bits(vp), vp_h)


def test_append_kv_bad_slot_is_skipped_and_latched():
    H_kv, D = 2, 128
    kp = torch.zeros((8, H_kv, D), dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    kn = torch.ones((2, H_kv, D), dtype=torch.bfloat16, device=DEV)
    slots = torch.tensor([3, 8], dtype=torch.int32, device=DEV)
    wm.append_kv(kn, kn, slots, kp, vp)
    assert wm.device_error(clear=True) == 1
    assert float(kp[3].float().sum()) == H_kv * D
    assert float(kp.float().sum()) == H_kv * D
