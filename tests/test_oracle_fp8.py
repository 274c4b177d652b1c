"""Pins of the oracle's fp8 (E4M3) KV path: the codec against the OCP FP8
E4M3 format's fixed points and against PyTorch's own float8_e4m3fn
conversion, the quantising append against the same library conversion, and
the fp8 attention against the (separately pinned) bf16 attention over the
decoded values and against the closed form that per-head scales give
(scores linear in k, outputs linear in v).  CPU only."""
import math

import numpy as np
import pytest
import torch

import oracle


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
        .view(np.uint16)


def _bits_to_f32(u):
    return (np.asarray(u).astype(np.uint32) << 16).view(np.float32)


# ---- codec ------------------------------------------------------------------

def test_format_fixed_points():
    t = oracle.e4m3_table()
    assert t[0x00] == 0.0 and math.copysign(1.0, t[0x80]) == -1.0
    assert t[0x01] == 2.0 ** -9            # smallest subnormal
    assert t[0x07] == 7 * 2.0 ** -9        # largest subnormal
    assert t[0x08] == 2.0 ** -6            # smallest normal
    assert t[0x38] == 1.0                  # exponent field 7 = bias
    assert t[0x39] == 1.125
    assert t[0x7E] == 448.0                # largest finite: 1.75 * 2^8
    assert t[0x77] == 240.0 and t[0x78] == 256.0
    assert math.isnan(t[0x7F]) and math.isnan(t[0xFF])
    assert np.isfinite(t).sum() == 254     # no infinities, two NaN codes
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0)        # codes ordered like their values
    assert np.array_equal(t[0x80:0xFF], -pos)


def test_decode_matches_library():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    t = oracle.e4m3_table()
    fin = np.isfinite(lib)
    assert np.array_equal(np.isfinite(t), fin)
    assert np.array_equal(t[fin], lib[fin])


def test_every_code_round_trips():
    t = oracle.e4m3_table()
    for c in range(256):
        if not math.isfinite(t[c]):
            continue
        assert oracle.f32_to_e4m3(t[c]) == c, hex(c)


@pytest.mark.parametrize("x,code", [
    (1.0625, 0x38),          # tie between 1.0 (0x38) and 1.125 (0x39): even
    (1.1875, 0x3A),          # tie between 1.125 (0x39) and 1.25 (0x3A): even
    (2.0 ** -10, 0x00),      # tie between 0 and the smallest subnormal
    (3 * 2.0 ** -10, 0x02),  # tie between 2^-9 and 2^-8 (subnormals): even
    (-1.0625, 0xB8),
    (1.07, 0x39),
    (447.0, 0x7E),
    (460.0, 0x7E),
    (1e9, 0x7E),             # saturation
    (-1e9, 0xFE),
    (float("inf"), 0x7E),
    (1e-30, 0x00),
    (-1e-30, 0x80),
])
def test_rounding_ties_and_saturation(x, code):
    assert oracle.f32_to_e4m3(x) == code


def test_encode_matches_library_in_range():
    # PyTorch's float8_e4m3fn conversion rounds to nearest even and does not
    # saturate; on |x| < 464 (the tie between 448 and the NaN code) the two
    # definitions agree.
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.standard_normal(4000) * 3,
        rng.uniform(-463.9, 463.9, 2000),
        rng.standard_normal(2000) * 2.0 ** -7,
        (oracle.e4m3_table()[:0x7E] + oracle.e4m3_table()[1:0x7F]) / 2,  # every positive tie
    ]).astype(np.float32)
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle.f32_to_e4m3(v) for v in x], np.uint8)
    assert np.array_equal(mine, lib)


# ---- quantising append ----------------------------------------------------------

def test_append_fp8_matches_library_quantisation():
    rng = np.random.default_rng(5)
    n, H_kv, D, num_slots = 5, 3, 16, 40
    kn = _bf16_bits(rng.standard_normal((n, H_kv, D)) * 2)
    vn = _bf16_bits(rng.standard_normal((n, H_kv, D)))
    ks = np.array([0.02, 0.25, 3.0], np.float32)
    vs = np.array([0.5, 0.012, 1.0], np.float32)
    slots = np.array([7, 0, 39, 12, 20], np.int32)
    kp = np.full((num_slots, H_kv, D), 0x55, np.uint8)
    vp = np.full((num_slots, H_kv, D), 0x55, np.uint8)
    oracle.append_kv_fp8(kn, vn, slots, ks, vs, kp, vp)

    def lib_codes(bits, s):
        x = torch.from_numpy(_bits_to_f32(bits))
        inv = torch.from_numpy((np.float32(1.0) / s).astype(np.float32))
        y = x * inv.view(1, -1, 1)
        assert y.abs().max() < 464
        return y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()

    assert np.array_equal(kp[slots], lib_codes(kn, ks))
    assert np.array_equal(vp[slots], lib_codes(vn, vs))
    untouched = np.setdiff1d(np.arange(num_slots), slots)
    assert np.all(kp[untouched] == 0x55) and np.all(vp[untouched] == 0x55)


def test_append_fp8_saturates_and_rejects_bad_slots():
    kn = _bf16_bits(np.full((1, 1, 4), 1000.0))
    vn = _bf16_bits(np.full((1, 1, 4), -1000.0))
    kp = np.zeros((2, 1, 4), np.uint8)
    vp = np.zeros((2, 1, 4), np.uint8)
    one = np.ones(1, np.float32)
    oracle.append_kv_fp8(kn, vn, np.array([1], np.int32), one, one, kp, vp)
    assert np.all(kp[1] == 0x7E) and np.all(vp[1] == 0xFE)
    with pytest.raises(ValueError):
        oracle.append_kv_fp8(kn, vn, np.array([2], np.int32), one, one, kp, vp)


# ---- attention over fp8 pools ---------------------------------------------------

def _fp8_case(seed, B=2, H_q=4, H_kv=2, D=16, num_slots=300, lens=(250, 37)):
    rng = np.random.default_rng(seed)
    kp = rng.integers(0, 256, size=(num_slots, H_kv, D)).astype(np.uint8)
    vp = rng.integers(0, 256, size=(num_slots, H_kv, D)).astype(np.uint8)
    # avoid the NaN codes and keep magnitudes modest (|code value| <= 16)
    for p in (kp, vp):
        p[(p & 0x7F) > 0x50] &= 0xC7
        p[(p & 0x7F) == 0x7F] = 0x38
    q = _bf16_bits(rng.standard_normal((B, 1, H_q, D)))
    stride = max(lens)
    table = np.full((B, stride), -1, np.int32)
    perm = rng.permutation(num_slots).astype(np.int32)
    off = 0
    for b, L in enumerate(lens):
        table[b, :L] = perm[off:off + L]
        off += L
    return q, kp, vp, table, np.array(lens, np.int32)


def _decoded_bf16_pool(codes, mult):
    t = oracle.e4m3_table()
    vals = t[codes] * np.asarray(mult, np.float64).reshape(1, -1, 1)
    bits = _bf16_bits(vals.astype(np.float32))
    assert np.array_equal(_bits_to_f32(bits).astype(np.float64), vals)  # exact in bf16
    return bits


def test_fp8_attention_equals_bf16_attention_of_decoded_values():
    # power-of-two scales keep the decoded values exact in bf16, so the fp8
    # attention must reproduce the bf16 attention over those values exactly
    q, kp, vp, table, lens = _fp8_case(3)
    ks = np.array([0.5, 4.0], np.float32)
    vs = np.array([2.0, 0.125], np.float32)
    o8, l8 = oracle.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.25)
    ob, lb = oracle.draft_decode_attn(q, _decoded_bf16_pool(kp, ks), _decoded_bf16_pool(vp, vs),
                                      table, lens, 0.25)
    assert np.array_equal(o8, ob) and np.array_equal(l8, lb)


def test_fp8_attention_per_head_scales_closed_form():
    # scores are linear in k and outputs in v: scale k_scale[g] into the
    # softmax scale of the heads reading KV head g and v_scale[g] into their
    # outputs
    q, kp, vp, table, lens = _fp8_case(4)
    H_q, H_kv = q.shape[2], kp.shape[1]
    ks = np.array([0.37, 1.9], np.float32)
    vs = np.array([0.011, 3.3], np.float32)
    one = np.ones(H_kv, np.float32)
    o8, l8 = oracle.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.3)
    G = H_q // H_kv
    for g in range(H_kv):
        o1, l1 = oracle.draft_decode_attn_fp8(q, kp, vp, one, one, table, lens,
                                              0.3 * float(ks[g]))
        hs = slice(g * G, (g + 1) * G)
        assert np.allclose(o8[:, :, hs], float(vs[g]) * o1[:, :, hs], rtol=1e-12, atol=1e-14)
        assert np.allclose(l8[:, :, hs], l1[:, :, hs], rtol=1e-12, atol=1e-12)


def test_fp8_attention_single_key_and_empty_row():
    q, kp, vp, table, _ = _fp8_case(6)
    ks = np.array([0.5, 1.0], np.float32)
    vs = np.array([0.25, 2.0], np.float32)
    lens = np.array([1, 0], np.int32)
    o, l = oracle.draft_decode_attn_fp8(q, kp, vp, ks, vs, table, lens, 0.1)
    t = oracle.e4m3_table()
    G = q.shape[2] // kp.shape[1]
    qf = _bits_to_f32(q).astype(np.float64)
    for h in range(q.shape[2]):
        g = h // G
        slot = table[0, 0]
        assert np.array_equal(o[0, 0, h], t[vp[slot, g]] * float(vs[g]))
        assert l[0, 0, h] == pytest.approx(0.1 * float(np.dot(qf[0, 0, h], t[kp[slot, g]] * float(ks[g]))),
                                          rel=1e-12, abs=1e-12)
    assert np.all(o[1] == 0.0) and np.all(np.isneginf(l[1]))
