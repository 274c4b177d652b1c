"""GPU attention-mass diagnostics (App. C, Table 12) against the oracle's
direct fp64 definitions, from GPU full-context and windowed attention of the
same queries."""
import math

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


@pytest.mark.parametrize("S", [200, 1087, 3000, 20_000])
def test_mass_diagnostics_match_definition(S):
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
    tf, lf = wm.build_draft_indices(seq, gamma, n_sink, W, gamma + 1, windowed=False, req_to_token=rtt)
    tw, lw = wm.build_draft_indices(seq, gamma, n_sink, W, gamma + 1, windowed=True, req_to_token=rtt)
    for j in range(gamma):
        # the same split count: inside the window both runs then agree bit for bit
        of, lsf = wm.draft_decode_attn(q[j], kp, vp, tf[j], lf[j], scale, n_split=4)
        ow, lsw = wm.draft_decode_attn(q[j], kp, vp, tw[j], lw[j], scale, n_split=4)
        a, p, t = wm.attn_mass_diagnostics(of, lsf, ow, lsw)
        ra, rp, rt = oracle.attn_mass(bits(q[j]), bits(kp), bits(vp), host_i32(tf[j]), host_i32(lf[j]),
                                      host_i32(tw[j]), host_i32(lw[j]), scale)
        for got, ref, what in ((a, ra, "in_win"), (p, rp, "win_perturb"), (t, rt, "tail_out_frac")):
            g = got.double().cpu().numpy().reshape(ref.shape)
            assert np.all(np.abs(g - ref) <= 1e-3 + 1e-2 * np.abs(ref)), (
                f"S={S} step {j} {what}: max err {np.abs(g - ref).max():.3e}")
        if S + j + 1 <= n_sink + W:  # nothing beyond the window
            assert torch.all(a == 1) and torch.all(p == 0) and torch.all(t == 0)
