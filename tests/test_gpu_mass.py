"""GPU attention-mass diagnostics ("Windowed-MTP", §5 "A partition-function
view"; App. C, Table 12) against the oracle's direct fp64 definitions.

The GPU computes them from the windowed attention and the attention over the
far keys (the far table of wmtp_build_far_indices), so a small far share
keeps its relative accuracy.  Two regimes: N(0,1) keys (almost all mass far
on long rows) and the regime the pages measure, queries whose mass sits
almost entirely inside the window (in-window mass >= 0.99, tail 1e-3 to
1e-2), where the comparison is on a relative basis.  The merged output is
also the full-context attention (checked against the oracle)."""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_draft_build_gb300 as wm
from speculative_decoding_draft_build_gb300 import synth
from wmtp_testutil import assert_attn_close, bits, host_i32

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    wm.build()
    wm.load()
    wm.device_error(clear=True)
    yield
    assert wm.device_error(clear=True) == 0


def _tables(seq, rtt, gamma, n_sink, W):
    tf, lf = wm.build_draft_indices(seq, gamma, n_sink, W, gamma + 1, windowed=False, req_to_token=rtt)
    tw, lw = wm.build_draft_indices(seq, gamma, n_sink, W, gamma + 1, windowed=True, req_to_token=rtt)
    tr, lr = wm.build_far_indices(seq, gamma, n_sink, W, rtt)
    return tf, lf, tw, lw, tr, lr


@pytest.mark.parametrize("S", [0, 500, 1087, 1088, 3000, 131_072])
def test_far_table_matches_oracle(S):
    n_sink, W, gamma = 64, 1024, 3
    pool = S + gamma
    rtt = synth.permutation(pool, 600 + S, DEV).view(1, -1)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    tr, lr = wm.build_far_indices(seq, gamma, n_sink, W, rtt)
    ref_t, ref_l = oracle.build_far_indices(np.array([S], np.int32), gamma, n_sink, W, host_i32(rtt))
    got_t, got_l = host_i32(tr), host_i32(lr)
    assert np.array_equal(got_l, ref_l)
    for j in range(gamma):
        n = ref_l[j, 0]
        assert np.array_equal(got_t[j, 0, :n], ref_t[j, 0, :n]), f"step {j}"


def _check(got, ref, atol, rtol, what):
    g = got.double().cpu().numpy().reshape(ref.shape)
    err = np.abs(g - ref)
    assert np.all(err <= atol + rtol * np.abs(ref)), (
        f"{what}: max err {err.max():.3e}, worst rel {np.max(err / np.maximum(np.abs(ref), 1e-300)):.3e}")


def _run(q, kp, vp, tabs, scale, gamma):
    tf, lf, tw, lw, tr, lr = tabs
    res = []
    for j in range(gamma):
        ow, lsw = wm.draft_decode_attn(q[j], kp, vp, tw[j], lw[j], scale)
        o_r, lsr = wm.draft_decode_attn(q[j], kp, vp, tr[j], lr[j], scale)
        o_full = torch.empty_like(ow)
        lse_full = torch.empty_like(lsw)
        a, p, t = wm.attn_mass_diagnostics(ow, lsw, o_r, lsr, o_full=o_full, lse_full=lse_full)
        res.append((ow, lsw, a, p, t, o_full, lse_full))
    return res


@pytest.mark.parametrize("S", [200, 1087, 3000, 20_000])
def test_mass_diagnostics_normal_keys(S):
    D, H_q, H_kv, n_sink, W, gamma = 128, 8, 2, 64, 1024, 2
    scale = 1 / math.sqrt(D)
    pool = S + gamma
    kp = synth.normal_bf16((pool, H_kv, D), 700 + S, DEV)
    # values with a common offset keep ||o|| away from zero
    vp = (synth.normal_bf16((pool, H_kv, D), 701 + S, DEV).float() + 0.5).to(torch.bfloat16)
    synth.scale_random_rows_(kp, 0.01, 4.0, 702 + S)
    q = synth.normal_bf16((gamma, 1, 1, H_q, D), 703 + S, DEV)
    rtt = synth.permutation(pool, 704 + S, DEV).view(1, -1)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    tabs = _tables(seq, rtt, gamma, n_sink, W)
    tf, lf, tw, lw = tabs[:4]
    for j, (ow, lsw, a, p, t, o_full, lse_full) in enumerate(_run(q, kp, vp, tabs, scale, gamma)):
        ra, rp, rt = oracle.attn_mass(bits(q[j]), bits(kp), bits(vp), host_i32(tf[j]), host_i32(lf[j]),
                                      host_i32(tw[j]), host_i32(lw[j]), scale)
        _check(a, ra, 1e-5, 1e-4, f"S={S} step {j} in_win")
        _check(p, rp, 1e-6, 1e-3, f"S={S} step {j} win_perturb")
        _check(t, rt, 1e-6, 1e-3, f"S={S} step {j} tail_out_frac")
        ro, rl = oracle.draft_decode_attn(bits(q[j]), bits(kp), bits(vp), host_i32(tf[j]), host_i32(lf[j]), scale)
        assert_attn_close(o_full, lse_full, ro, rl, what=f"S={S} step {j} merged full attention")
        if S + j + 1 <= n_sink + W:  # nothing beyond the window: exact
            assert torch.all(a == 1) and torch.all(p == 0) and torch.all(t == 0)
            assert torch.equal(o_full, ow) and torch.equal(lse_full, lsw)


@pytest.mark.parametrize("S,tail", [(20_000, 1e-2), (20_000, 1e-3), (131_072, 1e-2), (131_072, 2e-3)])
def test_mass_diagnostics_concentrated_in_window(S, tail):
    """Queries aligned with the sink and window keys (a common direction u):
    the kept keys' logits sit `shift` above the far keys', chosen so the far
    share is about `tail`; the diagnostics must match the fp64 definitions
    within 1e-3 relative."""
    D, H_q, H_kv, n_sink, W, gamma = 128, 8, 2, 64, 1024, 2
    scale = 1 / math.sqrt(D)
    pool = S + gamma
    n_far = S + 1 - n_sink - W
    shift = math.log(n_far / (n_sink + W)) + math.log(1 / tail)
    c = math.sqrt(shift / scale)  # query weight on u times key weight on u
    gen = synth.generator(800 + S, DEV)
    u = torch.randn(D, generator=gen, device=DEV)
    u = u / u.norm()
    rtt = synth.permutation(pool, 801 + S, DEV).view(1, -1)
    kf = torch.randn((pool, H_kv, D), generator=gen, device=DEV) * 0.5
    aligned = torch.cat([torch.arange(n_sink, device=DEV), torch.arange(S + 1 - W, pool, device=DEV)])
    kf[rtt[0, aligned].long()] += c * u
    kp = kf.to(torch.bfloat16)
    vp = (torch.randn((pool, H_kv, D), generator=gen, device=DEV) + 0.5).to(torch.bfloat16)
    q = (c * u + 0.3 * torch.randn((gamma, 1, 1, H_q, D), generator=gen, device=DEV)).to(torch.bfloat16)
    seq = torch.tensor([S], dtype=torch.int32, device=DEV)
    tabs = _tables(seq, rtt, gamma, n_sink, W)
    tf, lf, tw, lw = tabs[:4]
    kp_h, vp_h = bits(kp), bits(vp)
    for j, (ow, lsw, a, p, t, o_full, lse_full) in enumerate(_run(q, kp, vp, tabs, scale, gamma)):
        ra, rp, rt = oracle.attn_mass(bits(q[j]), kp_h, vp_h, host_i32(tf[j]), host_i32(lf[j]),
                                      host_i32(tw[j]), host_i32(lw[j]), scale)
        assert ra.min() >= 0.97 and rt.max() <= 5 * tail and rt.min() >= tail / 5, (ra.min(), rt.min(), rt.max())
        _check(a, ra, 1e-6, 1e-5, f"S={S} step {j} in_win")
        _check(p, rp, 1e-9, 1e-3, f"S={S} step {j} win_perturb")
        _check(t, rt, 1e-9, 1e-3, f"S={S} step {j} tail_out_frac")
        _check(1 - a.double(), 1 - ra, 1e-9, 2e-3, f"S={S} step {j} far share 1 - in_win")
        ro, rl = oracle.draft_decode_attn(bits(q[j]), kp_h, vp_h, host_i32(tf[j]), host_i32(lf[j]), scale)
        assert_attn_close(o_full, lse_full, ro, rl, what=f"S={S} step {j} merged full attention")
