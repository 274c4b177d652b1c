"""GPU tests of the overlapped draft step (wmtp_draft_decode_attn_append_overlap
and wmtp_draft_decode_attn_ring_overlap): the gamma draft forwards of a
decode step run back to back ("Windowed-MTP", §3 Eq. (1)), and from step 1
on each launch copies every kept key but the last `hold` entries while the
previous step is still running.  Only the moment of the copies changes, so a
chain of overlapped steps must give the bits of the same chain without
overlap: outputs, lse and the pools after the appends.  The chains also run
as CUDA graphs (where consecutive launches really do overlap), and one chain
is checked against the fp64 oracle."""
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
GAMMA = 6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    wm.build()
    wm.load()
    wm.device_error(clear=True)
    yield
    assert wm.device_error(clear=True) == 0


def _graph(fn):
    cur = torch.cuda.current_stream(DEV)
    cap = torch.cuda.Stream(DEV)
    cap.wait_stream(cur)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(gr, stream=cap):
            fn()
    cur.wait_stream(cap)
    torch.cuda.synchronize(DEV)
    return gr


class _Chain:
    """gamma fused draft steps over a paged pool (permuted page table)."""

    def __init__(self, seed, S_list, H_q, H_kv, D, n_sink, W, windowed, n_split):
        B = len(S_list)
        self.B, self.D, self.H_kv = B, D, H_kv
        ctx = [s + GAMMA for s in S_list]
        total = sum(ctx)
        self.kp0 = synth.normal_bf16((total, H_kv, D), seed, DEV)
        self.vp0 = synth.normal_bf16((total, H_kv, D), seed + 1, DEV)
        perm = synth.permutation(total, seed + 2, DEV)
        self.rtt = torch.zeros((B, max(ctx)), dtype=torch.int32, device=DEV)
        off = 0
        for b in range(B):
            self.rtt[b, :ctx[b]] = perm[off:off + ctx[b]]
            off += ctx[b]
        self.seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
        self.tab, self.lens = wm.build_draft_indices(self.seq, GAMMA, n_sink, W, GAMMA + 1, windowed=windowed,
                                                     req_to_token=self.rtt)
        req = torch.arange(B, device=DEV)
        self.slots = torch.stack([self.rtt[req, (self.seq + j).long()] for j in range(GAMMA)]).contiguous()
        self.kn = synth.normal_bf16((GAMMA, B, H_kv, D), seed + 3, DEV)
        self.vn = synth.normal_bf16((GAMMA, B, H_kv, D), seed + 4, DEV)
        self.q = synth.normal_bf16((GAMMA, B, 1, H_q, D), seed + 5, DEV)
        self.scale = 1 / math.sqrt(D)
        self.ns = n_split if n_split is not None else wm.attn_num_splits(B, 1, H_kv, self.tab.shape[-1], DEV)
        self.ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, self.ns), DEV)
        self.kp, self.vp = self.kp0.clone(), self.vp0.clone()
        self.out = torch.empty((GAMMA, B, 1, H_q, D), dtype=torch.float32, device=DEV)
        self.lse = torch.empty((GAMMA, B, 1, H_q), dtype=torch.float32, device=DEV)

    def reset(self):
        self.kp.copy_(self.kp0)
        self.vp.copy_(self.vp0)
        self.out.fill_(float("nan"))
        self.lse.fill_(float("nan"))

    def run(self, hold):
        for j in range(GAMMA):
            wm.draft_decode_attn_append(self.kn[j], self.vn[j], self.slots[j], self.q[j], self.kp, self.vp,
                                        self.tab[j], self.lens[j], self.scale, out=self.out[j], lse=self.lse[j],
                                        n_split=self.ns, workspace=self.ws,
                                        overlap_hold=None if hold is None else (hold if j > 0 else -1))

    def result(self):
        torch.cuda.synchronize(DEV)
        return self.out.clone(), self.lse.clone(), self.kp.clone(), self.vp.clone()


def _same(a, b, what):
    names = ("out", "lse", "k_pool", "v_pool")
    for x, y, n in zip(a, b, names):
        assert torch.equal(x, y), f"{what}: {n} differs"


def _check_chain(ch, holds, what):
    ch.reset()
    ch.run(None)
    ref = ch.result()
    for hold in holds:
        ch.reset()
        ch.run(hold)
        _same(ref, ch.result(), f"{what} eager hold={hold}")
        gr = _graph(lambda: ch.run(hold))
        for rep in range(3):
            ch.reset()
            gr.replay()
            _same(ref, ch.result(), f"{what} graph hold={hold} replay {rep}")
    return ref


@pytest.mark.parametrize("n_split", [1, 5, 16, 32, 37, None])
def test_overlapped_windowed_chain_short_and_ragged_rows(n_split):
    # rows from one key (everything held) to past the window; D = 128
    # (hold -1: chained launches that read nothing early)
    ch = _Chain(11, [0, 3, 1000, 1088, 70_000], 8, 2, 128, 64, 1024, True, n_split)
    _check_chain(ch, (-1, 2, 5), f"windowed D=128 n_split={n_split}")


@pytest.mark.parametrize("n_split", [1, 32, None])
def test_overlapped_windowed_chain_headline_geometry(n_split):
    # H_q = 16, H_kv = 2, D = 256, n_sink = 64, W = 4032, one 300K request
    ch = _Chain(21, [300_000], 16, 2, 256, 64, 4032, True, n_split)
    _check_chain(ch, (2,), f"windowed D=256 n_split={n_split}")


@pytest.mark.parametrize("n_split", [2, 76])
def test_overlapped_full_context_chain(n_split):
    # full rows: with 2 splits the held entries sit in tiles issued inside
    # the loop (after the wait), with 76 in the first tiles of the last split
    ch = _Chain(31, [20_000, 12_345], 16, 2, 256, 64, 4032, False, n_split)
    _check_chain(ch, (2,), f"full-context n_split={n_split}")


def test_overlapped_chain_against_oracle():
    ch = _Chain(41, [5, 1000, 4000], 8, 2, 128, 64, 1024, True, None)
    ref = _check_chain(ch, (2,), "oracle case")
    out, lse = ref[0], ref[1]
    kp_h, vp_h = bits(ch.kp0), bits(ch.vp0)
    tabs, lens = host_i32(ch.tab), host_i32(ch.lens)
    for j in range(GAMMA):
        oracle.append_kv(bits(ch.kn[j]), bits(ch.vn[j]), host_i32(ch.slots[j]), kp_h, vp_h)
        ro, rl = oracle.draft_decode_attn(bits(ch.q[j]), kp_h, vp_h, tabs[j], lens[j], ch.scale)
        assert_attn_close(out[j], lse[j], ro, rl, what=f"overlapped chain step {j}")
    assert np.array_equal(bits(ref[2]), kp_h) and np.array_equal(bits(ref[3]), vp_h)


@pytest.mark.parametrize("D,H_q,H_kv", [(256, 16, 2), (128, 8, 2)])
@pytest.mark.parametrize("n_split", [1, 5, 16, None])
def test_overlapped_ring_chain(D, H_q, H_kv, n_split):
    # table-free ring steps; D = 256 windows arrive partly as TMA boxes
    n_sink, W, d = 64, 1024, 7
    S_list = [10, 1000, 1088, 1089, 70_000]
    B = len(S_list)
    R = n_sink + W + d
    rb = synth.ring_bases(B, R, B + 3, 51 + D)
    ring_base = torch.tensor(rb, dtype=torch.int32, device=DEV)
    kp0 = synth.normal_bf16(((B + 3) * R, H_kv, D), 52 + D, DEV)
    vp0 = synth.normal_bf16(((B + 3) * R, H_kv, D), 53 + D, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    kn = synth.normal_bf16((GAMMA, B, H_kv, D), 54, DEV)
    vn = synth.normal_bf16((GAMMA, B, H_kv, D), 55, DEV)
    qs = synth.normal_bf16((GAMMA, B, 1, H_q, D), 56, DEV)
    scale = 1 / math.sqrt(D)
    ns = n_split if n_split is not None else wm.attn_num_splits(B, 1, H_kv, n_sink + W, DEV)
    ws = wm.AttnWorkspace(wm.attn_workspace_bytes(B, 1, H_q, H_kv, D, ns), DEV)
    kp, vp = kp0.clone(), vp0.clone()
    out = torch.empty((GAMMA, B, 1, H_q, D), dtype=torch.float32, device=DEV)
    lse = torch.empty((GAMMA, B, 1, H_q), dtype=torch.float32, device=DEV)

    def run(hold):
        for j in range(GAMMA):
            wm.draft_decode_attn_ring(qs[j], kp, vp, seq, ring_base, j, n_sink, W, d, scale, k_new=kn[j],
                                      v_new=vn[j], out=out[j], lse=lse[j], n_split=ns, workspace=ws,
                                      overlap_hold=None if hold is None else (hold if j > 0 else -1))

    def reset():
        kp.copy_(kp0)
        vp.copy_(vp0)
        out.fill_(float("nan"))
        lse.fill_(float("nan"))

    def result():
        torch.cuda.synchronize(DEV)
        return out.clone(), lse.clone(), kp.clone(), vp.clone()

    reset()
    run(None)
    ref = result()
    reset()
    run(2)
    _same(ref, result(), f"ring D={D} n_split={n_split} eager")
    gr = _graph(lambda: run(2))
    for rep in range(3):
        reset()
        gr.replay()
        _same(ref, result(), f"ring D={D} n_split={n_split} graph replay {rep}")


def test_overlap_hold_range():
    ch = _Chain(61, [100], 8, 2, 128, 4, 60, True, 1)
    with pytest.raises(ValueError):
        wm.draft_decode_attn_append(ch.kn[1], ch.vn[1], ch.slots[1], ch.q[1], ch.kp, ch.vp, ch.tab[1],
                                    ch.lens[1], ch.scale, n_split=1, overlap_hold=-2)


@pytest.mark.parametrize("hold", [0, 1, 3, 9])
def test_overlap_two_new_rows_and_hold_values(hold):
    # one launch, two new rows per request (their slots are the last two
    # entries of each row), every hold value giving the same bits as the
    # plain call: keys read from the new rows are always held, the rest
    # follow `hold`
    B, H_q, H_kv, D, n_new = 3, 8, 2, 128, 2
    lens_list = [3000, 130, 2]
    num_slots = 8000
    kp = synth.normal_bf16((num_slots, H_kv, D), 71, DEV)
    vp = synth.normal_bf16((num_slots, H_kv, D), 72, DEV)
    q = synth.normal_bf16((B, 1, H_q, D), 73, DEV)
    perm = synth.permutation(num_slots, 74, DEV)
    stride = max(lens_list)
    table = torch.full((B, stride), -1, dtype=torch.int32, device=DEV)
    off = 0
    for b, L in enumerate(lens_list):
        table[b, :L] = perm[off:off + L]
        off += L
    lens = torch.tensor(lens_list, dtype=torch.int32, device=DEV)
    new_slots = torch.stack([table[b, L - n_new:L] for b, L in enumerate(lens_list)]).contiguous()
    kn = synth.normal_bf16((B, n_new, H_kv, D), 75, DEV)
    vn = synth.normal_bf16((B, n_new, H_kv, D), 76, DEV)
    for n_split in (1, 7, 37):
        a_k, a_v = kp.clone(), vp.clone()
        b_k, b_v = kp.clone(), vp.clone()
        oa, la = wm.draft_decode_attn_append(kn, vn, new_slots, q, a_k, a_v, table, lens, 0.09, n_split=n_split)
        ob, lb = wm.draft_decode_attn_append(kn, vn, new_slots, q, b_k, b_v, table, lens, 0.09, n_split=n_split,
                                             overlap_hold=hold)
        assert torch.equal(oa, ob) and torch.equal(la, lb), f"hold={hold} n_split={n_split}"
        assert torch.equal(a_k, b_k) and torch.equal(a_v, b_v)


def test_overlapped_tree_ring_layout_chain():
    # ring of a k = 4 tree layout (modulus W + d*k); chained fused steps on
    # branch 0 equal the plain ones
    n_sink, W, d, k = 64, 1024, 7, 4
    D, H_q, H_kv = 256, 16, 2
    S_list = [5, 1100, 70_000]
    B = len(S_list)
    R = n_sink + W + d * k
    rb = synth.ring_bases(B, R, B + 1, 81)
    ring_base = torch.tensor(rb, dtype=torch.int32, device=DEV)
    kp0 = synth.normal_bf16(((B + 1) * R, H_kv, D), 82, DEV)
    vp0 = synth.normal_bf16(((B + 1) * R, H_kv, D), 83, DEV)
    seq = torch.tensor(S_list, dtype=torch.int32, device=DEV)
    kn = synth.normal_bf16((GAMMA, B, H_kv, D), 84, DEV)
    vn = synth.normal_bf16((GAMMA, B, H_kv, D), 85, DEV)
    qs = synth.normal_bf16((GAMMA, B, 1, H_q, D), 86, DEV)
    res = []
    for hold in (None, 2):
        kp, vp = kp0.clone(), vp0.clone()
        outs = []
        for j in range(GAMMA):
            o, l = wm.draft_decode_attn_ring(qs[j], kp, vp, seq, ring_base, j, n_sink, W, d, 1 / 16, k_new=kn[j],
                                             v_new=vn[j], tree_k=k,
                                             overlap_hold=None if hold is None else (hold if j > 0 else -1))
            outs.append((o, l))
        torch.cuda.synchronize()
        res.append((outs, kp, vp))
    for j in range(GAMMA):
        assert torch.equal(res[0][0][j][0], res[1][0][j][0]) and torch.equal(res[0][0][j][1], res[1][0][j][1])
    assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])
