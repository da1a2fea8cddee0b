"""Pins for the CPU oracle against facts other than its own formula.

Every check here comes from outside the oracle's code: exact rational brute
force, hand-derived closed forms, invariants the definition implies, a library
routine (torch scaled_dot_product_attention in float64) on the special cases
that reduce to it, and bit positions derived by hand from the PTX ISA's
m16n8k16 fragment tables.  A dropped term, a wrong rounding rule, the fp32
scale in place of the stored fp16 one, a missing clamp or a transposed operand
each fail at least one test below.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import synthetic as S

F16 = np.float16


def _fr(x) -> Fraction:
    return Fraction(float(x))


# ---------------------------------------------------------------- closed forms
def test_closed_form_exact_grid_2bit():
    # min 0, max 1.5, 2-bit: scale = 1.5 / 3 = 0.5 exactly, zero = 0, code = x / 0.5
    x = np.array([0.0, 0.5, 1.0, 1.5] * 8, dtype=F16)
    c, s, z = O.quantize_groups(x, 2)
    assert float(s) == 0.5 and float(z) == 0.0
    assert c.tolist() == [0, 1, 2, 3] * 8


def test_closed_form_integers_4bit_and_8bit():
    x = np.array(list(range(16)) + list(range(15, -1, -1)), dtype=F16) - F16(3)
    c, s, z = O.quantize_groups(x, 4)
    assert float(s) == 1.0 and float(z) == -3.0
    assert c.tolist() == list(range(16)) + list(range(15, -1, -1))
    x8 = np.array([0, 255] + list(range(7, 37)), dtype=F16)
    c, s, z = O.quantize_groups(x8, 8)
    assert float(s) == 1.0 and float(z) == 0.0
    assert c.tolist() == [0, 255] + list(range(7, 37))


def test_ties_round_half_to_even():
    # min -1, max 2, 2-bit: scale 1, zero -1; (x - zero) = 1.5, 0.5, 2.5 are exact
    # ties -> 2, 0, 2 under half-to-even (half-up would give 2, 1, 3).
    x = np.array([-1.0, 2.0, 0.5, -0.5, 1.5, 0.0, 1.0] + [0.0] * 25, dtype=F16)
    c, s, z = O.quantize_groups(x, 2)
    assert float(s) == 1.0 and float(z) == -1.0
    assert c[:7].tolist() == [0, 3, 2, 0, 2, 1, 2]


def test_scale_is_rounded_to_fp16_and_codes_use_it():
    # min 0, max 1, 4-bit: exact scale 1/15 = 0.0666..., whose nearest fp16 value
    # is 1092 * 2^-14 = 0.06665039.  Codes divide by that stored value:
    # 1 / 0.06665039 = 15.0037 -> 15; 0.5 / 0.06665039 = 7.5018 -> 8;
    # 0.25 / 0.06665039 = 3.7509 -> 4.
    x = np.array([0.0, 1.0, 0.5] + [0.25] * 29, dtype=F16)
    c, s, z = O.quantize_groups(x, 4)
    assert s == F16(1092 * 2.0 ** -14)
    assert c[:3].tolist() == [0, 15, 8]
    assert c[3] == 4  # 0.25 / 0.0666504 = 3.7509 -> 4


def test_constant_group_reconstructs_exactly():
    for val in (3.25, -7.0, 0.0, -0.0, 60000.0):
        x = np.full(32, val, dtype=F16)
        for b in (2, 4, 8):
            c, s, z = O.quantize_groups(x, b)
            assert (c == 0).all()
            assert float(s) == 0.0 and not np.signbit(s)
            assert float(z) == abs(val) if val == 0 else float(z) == val
            assert not np.signbit(z) or val < 0
            xh = O.dequantize(c, s, z)
            assert (xh == x.astype(np.float64)).all()


def test_negative_zero_canonicalised():
    x = np.array([-0.0] + [1.0] * 31, dtype=F16)
    c, s, z = O.quantize_groups(x, 2)
    assert float(z) == 0.0 and not np.signbit(z)


# ------------------------------------------------------------- brute force
def _brute_force_check(x, bits):
    """Exact rational check of one group's scale, zero and codes."""
    c, s, z = O.quantize_groups(x, bits)
    xs = [_fr(v) for v in x]
    mn, mx = min(xs), max(xs)
    assert _fr(z) == mn  # zero point = group minimum, exactly
    exact_scale = (mx - mn) / (2 ** bits - 1)
    sf = _fr(s)
    # stored scale is one of the two fp16 neighbours of the exact scale, the
    # nearer one unless fp32 rounding first made the choice a near-tie
    if exact_scale == 0:
        assert sf == 0
    else:
        lo = _fr(np.float16(float(exact_scale)))
        err = abs(sf - exact_scale)
        best = abs(lo - exact_scale)
        assert err <= best * (1 + Fraction(1, 2 ** 10)) + Fraction(1, 2 ** 40)
    levels = range(2 ** bits)
    for xi, ci in zip(xs, c.tolist()):
        assert 0 <= ci < 2 ** bits
        if sf == 0:
            assert ci == 0
            continue
        d = {k: abs(xi - (mn + sf * k)) for k in levels}
        best = min(d.values())
        if d[ci] == best:
            continue
        # only a near-tie may go either way: exact quotient within 2^-20 of k + 1/2
        q = (xi - mn) / sf
        frac = q - int(q)
        assert abs(frac - Fraction(1, 2)) < Fraction(1, 2 ** 20) * (1 + abs(q)), (xi, ci, q)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("dist,scale", [("normal", 1.0), ("normal", 30.0),
                                        ("uniform", 1e-3), ("lognormal", 1.0),
                                        ("normal", 1e-6)])
def test_brute_force_random_groups(bits, dist, scale):
    x = S.random_groups(seed=bits * 100 + int(scale * 7) % 97, n=24, dist=dist, scale=scale)
    for row in x:
        _brute_force_check(row, bits)


def test_brute_force_subnormal_scale():
    # fp16 subnormal scale: range 3 * 2^-24 at 2-bit -> scale 2^-24
    x = np.array([0, 2.0 ** -24, 2 * 2.0 ** -24, 3 * 2.0 ** -24] * 8, dtype=F16)
    c, s, z = O.quantize_groups(x, 2)
    assert float(s) == 2.0 ** -24
    assert c.tolist() == [0, 1, 2, 3] * 8
    _brute_force_check(x, 2)


# ------------------------------------------------------------- invariants
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_invariants_range_min_max_error(bits):
    x = S.random_groups(seed=7 + bits, n=256, dist="normal", scale=3.0)
    c, s, z = O.quantize_groups(x, bits)
    assert c.max() <= 2 ** bits - 1
    for row, cr, sr in zip(x, c, s):
        assert cr[np.argmin(row)] == 0
        assert cr[np.argmax(row)] == 2 ** bits - 1
    xh = O.dequantize(c, s, z)
    err = np.abs(xh - x.astype(np.float64))
    # |x - x_hat| <= scale_h / 2 (normal fp16 scales; fp32 rounding slack 2^-9)
    assert (err <= s.astype(np.float64)[:, None] * 0.5 * (1 + 2.0 ** -9)).all()


@pytest.mark.parametrize("bits", [2, 4])
def test_power_of_two_scaling_invariance(bits):
    x = S.random_groups(seed=11, n=64, dist="normal", scale=1.0)
    c0, s0, z0 = O.quantize_groups(x, bits)
    for k in (-3, 2, 5):
        xk = (x.astype(np.float32) * 2.0 ** k).astype(F16)
        assert (xk.astype(np.float32) == x.astype(np.float32) * 2.0 ** k).all()
        ck, sk, zk = O.quantize_groups(xk, bits)
        assert (ck == c0).all()
        assert (sk.astype(np.float64) == s0.astype(np.float64) * 2.0 ** k).all()
        assert (zk.astype(np.float64) == z0.astype(np.float64) * 2.0 ** k).all()


def test_permutation_within_group():
    x = S.random_groups(seed=3, n=16, dist="normal")
    rng = np.random.default_rng(0)
    perm = rng.permutation(32)
    c, s, z = O.quantize_groups(x, 4)
    cp, sp, zp = O.quantize_groups(x[:, perm], 4)
    assert (cp == c[:, perm]).all() and (sp == s).all() and (zp == z).all()


def test_key_groups_are_per_channel_over_tokens():
    # An outlier at (token 7, channel 5) widens exactly one key group: channel 5 of
    # tokens 0..31.  Per-token grouping, or a transposed reshape, would widen others.
    rng = np.random.default_rng(1)
    k = rng.standard_normal((64, 64)).astype(F16)
    _, s0, z0 = O.quantize_keys(k, 2)
    k2 = k.copy()
    k2[7, 5] = F16(500)
    c2, s2, z2 = O.quantize_keys(k2, 2)
    changed = np.argwhere(s2 != s0)
    assert changed.tolist() == [[0, 5]]
    assert s2.shape == (2, 64)


def test_value_groups_are_per_token_over_channels():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((64, 128)).astype(F16)
    _, s0, _ = O.quantize_values(v, 2)
    v2 = v.copy()
    v2[7, 70] = F16(500)  # channel group 70 // 32 = 2 of token 7
    _, s2, _ = O.quantize_values(v2, 2)
    assert np.argwhere(s2 != s0).tolist() == [[7, 2]]
    assert s2.shape == (64, 4)


def test_key_grouping_axis_matters_on_outlier_channels():
    # The article (paragraph 4): per-channel key groups isolate outlier channels.
    # On the outlier recipe, per-channel reconstruction error is far below
    # per-token grouping of the same keys.
    w = S.LLAMA2_13B.scaled(batch=1, n_q_heads=2, n_kv_heads=2, context=256)
    inp = S.generate(w)
    k = np.swapaxes(inp["K"][0], 0, 1)  # [H, T, D]
    c, s, z = O.quantize_keys(k, 2)
    err_ch = np.abs(O.dequantize_keys(c, s, z) - k.astype(np.float64)).mean()
    c2, s2, z2 = O.quantize_values(k, 2)  # per-token groups of the keys
    err_tok = np.abs(O.dequantize_values(c2, s2, z2) - k.astype(np.float64)).mean()
    assert err_ch < 0.5 * err_tok


# ------------------------------------------------------------- attention
def _sdpa64(q, k, v, scale):
    qt = torch.from_numpy(q.astype(np.float64))[:, None, :]  # [H, 1, D]
    kt = torch.from_numpy(k.astype(np.float64))
    vt = torch.from_numpy(v.astype(np.float64))
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return o[:, 0, :].numpy()


def test_all_tail_equals_sdpa_float64():
    # n_quant = 0: every token is fp16 in the tail; the oracle must equal exact
    # attention (north_star: "with no quantization the result matches exact attention").
    w = S.LLAMA31_8B_128K.scaled(context=96, n_tail=96, tail_cap=96)
    inp = S.generate(w)
    st = O.quantize_sequence(inp["K"][0], inp["V"][0], 96, 96, 2)
    out = O.sequence_attention(inp["q"][0], st, w.sm_scale)
    k = np.swapaxes(inp["K"][0], 0, 1)
    v = np.swapaxes(inp["V"][0], 0, 1)
    kk = np.repeat(k, w.gqa, axis=0)
    vv = np.repeat(v, w.gqa, axis=0)
    ref = _sdpa64(inp["q"][0], kk, vv, w.sm_scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_dequantized_cache_equals_sdpa_on_dequantized_inputs():
    w = S.TINY
    inp = S.generate(w)
    st = O.quantize_sequence(inp["K"][0], inp["V"][0], 256, 0, 2)
    keys, values = O.sequence_kv(st)
    out = O.sequence_attention(inp["q"][0], st, w.sm_scale)
    ref = _sdpa64(inp["q"][0], keys, values, w.sm_scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(5)
    d, n = 64, 40
    keys = rng.standard_normal((1, n, d))
    row = rng.standard_normal(d)
    q = rng.standard_normal((1, d)).astype(F16)
    # all V rows equal -> output is that row
    out = O.decode_attention(q, keys, np.tile(row, (1, n, 1)), 0.125)
    np.testing.assert_allclose(out[0], row, atol=1e-13)
    # q = 0 -> uniform weights -> mean of V
    values = rng.standard_normal((1, n, d))
    out = O.decode_attention(np.zeros((1, d), F16), keys, values, 0.125)
    np.testing.assert_allclose(out[0], values[0].mean(0), atol=1e-13)
    # a single token -> its V row
    out = O.decode_attention(q, keys[:, :1], values[:, :1], 0.125)
    np.testing.assert_allclose(out[0], values[0, 0], atol=1e-13)
    # two tokens, hand softmax: weights e^{l0}/(e^{l0}+e^{l1})
    l0 = 0.125 * keys[0, 0] @ q[0].astype(np.float64)
    l1 = 0.125 * keys[0, 1] @ q[0].astype(np.float64)
    p0 = 1.0 / (1.0 + np.exp(l1 - l0))
    out = O.decode_attention(q, keys[:, :2], values[:, :2], 0.125)
    np.testing.assert_allclose(out[0], p0 * values[0, 0] + (1 - p0) * values[0, 1], atol=1e-12)
    # empty context -> zeros
    assert (O.decode_attention(q, keys[:, :0], values[:, :0], 0.125) == 0).all()


def test_gqa_equals_mha_with_repeated_kv_heads():
    rng = np.random.default_rng(6)
    keys = rng.standard_normal((2, 33, 32))
    values = rng.standard_normal((2, 33, 32))
    q = rng.standard_normal((8, 32)).astype(F16)
    gqa = O.decode_attention(q, keys, values, 0.2)
    mha = O.decode_attention(q, np.repeat(keys, 4, 0), np.repeat(values, 4, 0), 0.2)
    np.testing.assert_allclose(gqa, mha, atol=1e-14)
    # query head 5 reads KV head 1 (contiguous groups of 4)
    one = O.decode_attention(q[5:6], keys[1:2], values[1:2], 0.2)
    np.testing.assert_allclose(gqa[5], one[0], atol=1e-14)


def test_attention_token_permutation_invariance():
    rng = np.random.default_rng(7)
    keys = rng.standard_normal((1, 50, 16))
    values = rng.standard_normal((1, 50, 16))
    q = rng.standard_normal((1, 16)).astype(F16)
    perm = rng.permutation(50)
    a = O.decode_attention(q, keys, values, 0.25)
    b = O.decode_attention(q, keys[:, perm], values[:, perm], 0.25)
    np.testing.assert_allclose(a, b, atol=1e-14)


# ------------------------------------------------------------- tail / append
def test_append_flushes_only_when_tail_full():
    assert O.append_lengths(64, 31, 32) == (64, 32, False)
    assert O.append_lengths(64, 32, 32) == (96, 1, True)
    assert O.append_lengths(0, 64, 64) == (32, 33, True)
    assert O.append_lengths(0, 0, 32) == (0, 1, False)


def test_flushed_group_equals_prefill_quantization():
    # Appending tokens one by one (flush of the oldest 32 when the tail is full)
    # leaves the same quantized region as quantizing the whole prefix at once,
    # because key groups are aligned 32-token spans from token 0.
    w = S.TINY.scaled(context=160)
    inp = S.generate(w)
    k, v = inp["K"][0], inp["V"][0]
    nq, nt = 0, 0
    for _ in range(160):
        nq, nt, _ = O.append_lengths(nq, nt, 32)
    assert nq + nt == 160 and nq == 128 and nt == 32
    st = O.quantize_sequence(k, v, 160, nt, 2)
    ref = O.quantize_sequence(k[:128], v[:128], 128, 0, 2)
    assert (st["k_codes"] == ref["k_codes"]).all() and (st["k_scale"] == ref["k_scale"]).all()


# ------------------------------------------------------------- layout pins
# Positions derived by hand from the PTX ISA's mma.m16n8k16 .f16 A-fragment
# table (a0: row gid, cols 2*tig..+1; a1: row gid+8; a2: cols +8; a3: both) and
# the tile rules: lane = 4*gid + tig; pair P -> word P // (16/b), slot P % (16/b);
# first code at bits [p, +b), second at [16 + p, +b) with p the slot's bit position (b*slot at 4
# and 8 bits; 2-bit slots 0..7 at 0, 2, 8, 10, 4, 6, 12, 14); lane word w at
# byte ((w // 4) * 32 + lane) * 16 + (w % 4) * 4.
KPOS_2BIT_D128 = [
    # (token, channel) -> (byte offset of the 32-bit word, bit offset); 2-bit slot
    # bit positions (0, 2, 8, 10, 4, 6, 12, 14)
    ((0, 0), (0, 0)), ((0, 1), (0, 16)), ((8, 0), (0, 2)), ((0, 8), (0, 8)),
    ((8, 9), (0, 26)), ((16, 0), (0, 4)), ((24, 8), (0, 14)), ((1, 0), (64, 0)),
    ((0, 2), (16, 0)), ((0, 16), (4, 0)), ((0, 64), (512, 0)), ((31, 127), (1020, 30)),
]
KPOS_4BIT_D128 = [((0, 0), (0, 0)), ((16, 0), (4, 0)), ((8, 1), (0, 20)), ((0, 16), (8, 0)),
                  ((0, 32), (512, 0))]
VPOS_2BIT_D128 = [
    ((0, 0), (0, 0)), ((1, 0), (0, 16)), ((0, 8), (0, 2)), ((8, 0), (0, 8)),
    ((16, 0), (0, 4)), ((2, 0), (16, 0)), ((0, 1), (64, 0)), ((0, 16), (4, 0)),
]


@pytest.mark.parametrize("kind,bits,table", [("K", 2, KPOS_2BIT_D128), ("K", 4, KPOS_4BIT_D128),
                                             ("V", 2, VPOS_2BIT_D128)])
def test_tile_layout_hand_positions(kind, bits, table):
    codes = np.zeros((32, 128), np.uint8)
    for (t, d), (byte, bit) in table:
        codes[:] = 0
        codes[t, d] = 2 ** bits - 1
        packed = O.pack_tiles(codes, kind, bits)
        words = packed.view("<u4")
        nz = np.nonzero(words)[0]
        assert nz.tolist() == [byte // 4], (t, d)
        assert int(words[byte // 4]) == (2 ** bits - 1) << bit, (t, d)


def test_metadata_order_hand_positions():
    # key block slot -> (field, channel); word 16kt + 4tig + 2r + f holds field f
    # (0 zero, 1 scale) of channels 16kt + 2tig + 8r and +1
    ko = O.key_meta_order(128)
    assert ko[:8].tolist() == [[0, 0], [0, 1], [1, 0], [1, 1], [0, 8], [0, 9], [1, 8], [1, 9]]
    assert ko[8:10].tolist() == [[0, 2], [0, 3]]  # word 4 = (kt 0, tig 1, r 0, zero)
    assert ko[32:34].tolist() == [[0, 16], [0, 17]]  # word 16 = (kt 1, tig 0, r 0, zero)
    assert ko[254:256].tolist() == [[1, 126], [1, 127]]  # word 127 = (kt 7, tig 3, r 1, scale)
    # value plane slot -> j*32 + token; pair (tig, j, kt, r) at 16j + 4tig + 2kt + r
    vo = O.value_meta_order(128)
    assert vo[:8].tolist() == [0, 1, 8, 9, 16, 17, 24, 25]
    assert vo[8:10].tolist() == [2, 3]  # pair 4 = (tig 1, j 0, kt 0, r 0)
    assert vo[32:34].tolist() == [32, 33]  # pair 16 = (tig 0, j 1, kt 0, r 0)
    # packing places a planted value where the order says
    sc = np.zeros(128, np.float16)
    sc[19] = 5  # channel 19 = 16 + 2*1 + 1: (kt 1, tig 1, r 0), scale -> word 16+4+1 = 21, second half -> slot 43
    assert np.nonzero(O.pack_key_meta(sc, np.zeros_like(sc)).reshape(-1))[0].tolist() == [43]
    zp = np.zeros(128, np.float16)
    zp[19] = 5  # the zero point of the same channel: word 20 -> slot 41
    assert np.nonzero(O.pack_key_meta(np.zeros_like(zp), zp).reshape(-1))[0].tolist() == [41]
    vs = np.zeros((32, 4), np.float16)
    vs[16, 1] = 7  # token 16 of channel group 1 -> pair (tig 0, j 1, kt 1, r 0) = 18 -> slot 36
    assert np.nonzero(O.pack_value_meta(vs, np.zeros_like(vs))[0])[0].tolist() == [36]


@pytest.mark.parametrize("kind", ["K", "V"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
def test_tile_layout_is_a_bijection(kind, bits, d):
    word, bit = O.tile_code_positions(kind, d, bits)
    fields = set(zip((word * 32 + bit).ravel().tolist()))
    assert len(fields) == 32 * d
    assert word.max() + 1 == 32 * d * bits // 32
    rng = np.random.default_rng(bits + d)
    codes = rng.integers(0, 2 ** bits, (2, 32, d), dtype=np.uint8)
    assert (O.unpack_tiles(O.pack_tiles(codes, kind, bits), kind, d, bits) == codes).all()


# ------------------------------------------------------------- mixed width
def _small_trizone(seed=4, t_old=200, fresh=8, d=64, probs=None):
    w = S.TRIZONE.scaled(batch=1, n_q_heads=4, n_kv_heads=1, head_dim=d,
                         context=t_old + fresh, trizone_fresh=fresh, seed=seed,
                         **({"v_width_probs": probs} if probs else {}))
    inp = S.generate(w)
    return w, inp


def test_trizone_all_fp16_equals_exact_attention():
    # every old token at width 16 (no V quantization) and K at 8 bits: the V side
    # is exact; with the K codes dequantized first, the result equals SDPA.
    w, inp = _small_trizone(probs=(0, 0, 0, 0, 1.0))
    k, v = inp["K"][0, :, 0], inp["V"][0, :, 0]
    tz = O.trizone_quantize(k, v, inp["v_width"][0, 0], np.full(64, 8, np.uint8))
    keys, values = O.trizone_kv(tz)
    assert (values == v.astype(np.float64)).all()
    out = O.trizone_attention(inp["q"][0], [tz], w.sm_scale)
    ref = _sdpa64(inp["q"][0], np.repeat(keys[None], 4, 0), np.repeat(values[None], 4, 0), w.sm_scale)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_trizone_all_evicted_leaves_fresh_tokens():
    w, inp = _small_trizone(probs=(1.0, 0, 0, 0, 0))
    k, v = inp["K"][0, :, 0], inp["V"][0, :, 0]
    tz = O.trizone_quantize(k, v, inp["v_width"][0, 0], inp["k_width"][0, 0])
    assert tz["blocks"] == []
    out = O.trizone_attention(inp["q"][0], [tz], w.sm_scale)
    ref = _sdpa64(inp["q"][0], np.repeat(k[200:][None], 4, 0), np.repeat(v[200:][None], 4, 0),
                  w.sm_scale)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_trizone_blocks_are_width_uniform_and_cover_kept_tokens():
    w, inp = _small_trizone()
    vw = inp["v_width"][0, 0]
    blocks = O.trizone_blocks(vw)
    seen = np.concatenate([t for _, t in blocks])
    assert sorted(seen.tolist()) == np.nonzero(vw)[0].tolist()
    for width, toks in blocks:
        assert (vw[toks] == width).all() and 1 <= len(toks) <= 32
    widths = [wd for wd, _ in blocks]
    assert widths == sorted(widths)


def test_trizone_matches_uniform_when_widths_are_uniform():
    # all V widths 4, all K widths 4, 192 old tokens: blocks are the uniform
    # cache's 32-token groups, so codes and attention coincide.
    w, inp = _small_trizone(t_old=192, probs=(0, 0, 1.0, 0, 0))
    k, v = inp["K"][0, :, 0], inp["V"][0, :, 0]
    tz = O.trizone_quantize(k, v, inp["v_width"][0, 0], np.full(64, 4, np.uint8))
    st = O.quantize_sequence(k[:, None], v[:, None], 200, 8, 4)
    kc = np.concatenate([b["k_codes"] for b in tz["blocks"]])
    assert (kc == st["k_codes"][0]).all()
    a = O.trizone_attention(inp["q"][0], [tz], w.sm_scale)
    b = O.sequence_attention(inp["q"][0], st, w.sm_scale)
    np.testing.assert_allclose(a, b, atol=1e-13)


# ------------------------------------------------------- mixed-width layout
def test_trizone_channel_order_by_hand():
    # channels 1 and 3 at 2 bits, channel 0 at 8 bits, the other 125 at 4 bits:
    # class 2 -> [1, 3] + 14 pads; class 4 -> 2, 4, 5, ..., 127 + 3 pads; class 8 -> [0] + 15 pads
    kw = np.full(128, 4, np.uint8)
    kw[[1, 3]] = 2
    kw[0] = 8
    slots, kts = O.trizone_channel_order(kw)
    assert kts == (1, 8, 1)
    assert slots[:2].tolist() == [1, 3] and (slots[2:16] == -1).all()
    assert slots[16:19].tolist() == [2, 4, 5] and slots[140] == 127 and (slots[141:144] == -1).all()
    assert slots[144] == 0 and (slots[145:160] == -1).all()
    assert len(slots) == 160


# (kt, bits) -> {(token, class channel): (lane word index w*32 + lane, bit)}, derived by
# hand from the fragment layout: lane 4 gid + tig; pair P = 8 kt + 4 mt + i covers
# token 16 mt + gid + 8 (i % 2), channels 16 kt + 2 tig + 8 (i // 2) and +1.
KSUB_POS = {
    (1, 2): {(0, 0): (0, 0), (0, 1): (0, 16), (8, 0): (0, 2), (0, 8): (0, 8), (8, 8): (0, 10),
             (16, 0): (0, 4), (31, 15): (31, 30), (31, 14): (31, 14)},
    (3, 4): {(25, 2): (37, 4), (25, 3): (37, 20), (0, 16): (64, 0), (31, 47): (191, 28)},
    (2, 8): {(9, 1): (4, 24), (0, 0): (0, 0), (16, 16): (192, 0)},
}


@pytest.mark.parametrize("kt,bits", list(KSUB_POS))
def test_trizone_key_subtile_positions_by_hand(kt, bits):
    word, bit = O.trizone_ksub_positions(kt, bits)
    for (t, c), pos in KSUB_POS[(kt, bits)].items():
        assert (int(word[t, c]), int(bit[t, c])) == pos, (t, c)
    assert len(set(zip((word * 32 + bit).ravel().tolist()))) == 32 * 16 * kt
    assert word.max() + 1 == 16 * kt * bits


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_trizone_key_subtile_is_the_uniform_tile_word_interleaved(bits):
    # with all 128 channels in one class the sub-tile holds the uniform key tile's
    # lane words, word w of lane L at 4 (32 w + L) instead of 16 (32 (w // 4) + L) + 4 (w % 4)
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, (32, 128), dtype=np.uint8)
    uni = O.pack_tiles(codes[None], "K", bits).reshape(-1).view("<u4")
    word, bit = O.trizone_ksub_positions(8, bits)
    sub = O._pack_words(codes, word, bit, 16 * 8 * bits).view("<u4")
    nw = 128 * bits // 32
    for lane in range(32):
        for w in range(nw):
            assert sub[w * 32 + lane] == uni[(w // 4) * 32 * 4 + lane * 4 + w % 4]


def test_trizone_block_bytes_closed_form():
    # K: 64 kt c bytes per class + 64 per k-tile of metadata; V: codes + 512 B meta, or fp16 rows
    assert O.trizone_block_bytes((5, 3, 1), 2) == 1920 + 576 + 1024 + 512
    assert O.trizone_block_bytes((5, 3, 1), 4) == 1920 + 576 + 2048 + 512
    assert O.trizone_block_bytes((5, 3, 1), 8) == 1920 + 576 + 4096 + 512
    assert O.trizone_block_bytes((5, 3, 1), 16) == 1920 + 576 + 8192
    assert O.trizone_block_bytes((0, 8, 0), 4) == O.tile_bytes(128, 4) * 2 + 1024


def test_trizone_pack_block_fields():
    # a partial block of 20 tokens: decode every field of the record independently
    w, inp = _small_trizone(t_old=400, fresh=0, d=128, probs=(0, 1.0, 0, 0, 0))
    k, v = inp["K"][0, :, 0], inp["V"][0, :, 0]
    kw = np.array([2, 4, 8, 4] * 32, np.uint8)
    tz = O.trizone_quantize(k[:20], v[:20], np.full(20, 2, np.uint8), kw)
    blk = tz["blocks"][0]
    slots, kts = O.trizone_channel_order(kw)
    assert kts == (2, 4, 2)
    rec = O.trizone_pack_block(blk, slots, kts)
    off = 0
    for kt, c in zip(kts, (2, 4, 8)):
        word, bit = O.trizone_ksub_positions(kt, c)
        sub = rec[off:off + 64 * kt * c].view("<u4")
        got = (sub[word] >> bit.astype(np.uint32)) & (2 ** c - 1)
        cls = slots[sum(16 * x for x in kts[:(2, 4, 8).index(c)]):][:16 * kt]
        for j, ch in enumerate(cls):
            assert (got[:20, j] == blk["k_codes"][:, ch]).all() and (got[20:, j] == 0).all()
        off += 64 * kt * c
    meta = rec[off:off + 64 * 8].view(np.float16)
    # (kt=1, tig=2, r=1) covers slots 16 + 4 + 8 = 28 and 29: its zero-point pair is
    # pair 16 + 8 + 2 = 26 (halves 52, 53), its scale pair 27 (halves 54, 55)
    assert meta[54].view(np.uint16) == blk["k_scale"][slots[28]].view(np.uint16)
    assert meta[53].view(np.uint16) == blk["k_zero"][slots[29]].view(np.uint16)
    assert meta[52].view(np.uint16) == blk["k_zero"][slots[28]].view(np.uint16)
    # the first pairs: zero points of slots 0, 1, scales of 0, 1, zero points of 8, 9
    assert (meta[:6].view(np.uint16) == np.array([blk["k_zero"][slots[0]], blk["k_zero"][slots[1]],
                                                   blk["k_scale"][slots[0]], blk["k_scale"][slots[1]],
                                                   blk["k_zero"][slots[8]], blk["k_zero"][slots[9]]],
                                                  np.float16).view(np.uint16)).all()
    off += 512
    vcodes = O.unpack_tiles(rec[off:off + 1024][None], "V", 128, 2)[0]
    assert (vcodes[:20] == blk["v_codes"]).all() and (vcodes[20:] == 0).all()
    off += 1024
    vm = rec[off:].view(np.float16)
    assert vm.size == 256 and (vm.view(np.uint16) != 0).sum() > 0
    assert off + 512 == rec.size


# 16-bit tiles: {(token, channel): (byte offset of the 32-bit word, bit)}, by hand from
# the fragment layouts (word w of lane L at 16 (32 (w // 4) + L) + 4 (w % 4))
FP16_POS = {
    "V": {(0, 0): (0, 0), (1, 0): (0, 16), (2, 0): (16, 0), (8, 0): (8, 0), (0, 8): (4, 0),
          (16, 0): (512, 0), (0, 16): (1024, 0), (0, 1): (64, 0)},
    "K": {(0, 0): (0, 0), (0, 1): (0, 16), (8, 0): (4, 0), (0, 8): (8, 0), (16, 0): (512, 0),
          (0, 16): (1024, 0), (1, 0): (64, 0)},
}


@pytest.mark.parametrize("kind", ["K", "V"])
def test_fp16_tile_positions_by_hand(kind):
    rows = np.zeros((32, 128), np.float16)
    for n, (t, c) in enumerate(FP16_POS[kind]):
        rows[t, c] = np.float16(n + 1)
    tile = O._fp16_tile(rows, kind, 128)
    words = tile.view("<u4")
    for n, ((t, c), (byte, bit)) in enumerate(FP16_POS[kind].items()):
        assert (words[byte // 4] >> bit) & 0xFFFF == np.float16(n + 1).view(np.uint16), (t, c)
    assert (O.unpack_tiles(tile, kind, 128, 16) == rows.view(np.uint16)).all()


def test_trizone_pack_index_and_stream():
    w, inp = _small_trizone(t_old=700, fresh=40, d=128)
    k, v = inp["K"][0, :, 0], inp["V"][0, :, 0]
    vw, kw = inp["v_width"][0, 0], inp["k_width"][0, 0]
    tz = O.trizone_quantize(k, v, vw, kw)
    pk = O.trizone_pack(tz)
    hdr = pk["index"][:128].view(np.int32)
    n_tok = [int((vw == c).sum()) for c in (2, 4, 8, 16)]
    assert hdr[0:4].tolist() == n_tok and hdr[4] == 40
    assert hdr[5:9].tolist() == [(n + 31) // 32 for n in n_tok] and hdr[9] == 2
    assert hdr[10:13].tolist() == [int((kw == c).sum()) for c in (2, 4, 8)]
    assert hdr[13:16].tolist() == [(int((kw == c).sum()) + 15) // 16 for c in (2, 4, 8)]
    assert hdr[20] == 16384 and hdr[21] == 0 and (hdr[27:] == 0).all()
    assert all(hdr[21 + i + 1] == hdr[21 + i] + hdr[5 + i] * hdr[16 + i] for i in range(4))
    assert hdr[26] == hdr[25] + 2 * 16384 == pk["data"].size
    # stream order: kept tokens by width class, ascending positions inside a class
    exp = np.concatenate([np.nonzero(vw == c)[0] for c in (2, 4, 8, 16)])
    assert (pk["tokens"] == exp).all()
    sl = pk["index"][128:448].view(np.int16)
    assert sorted(sl[sl >= 0].tolist()) == list(range(128))
    # the fresh blocks hold the fresh rows (the second one 8 rows, the rest zero)
    fb = pk["data"][hdr[25] + 16384:]
    kt = O.unpack_tiles(fb[:8192], "K", 128, 16)
    assert (kt[:8] == k[732:740].view(np.uint16)).all() and (kt[8:] == 0).all()
    vt = O.unpack_tiles(fb[8192:], "V", 128, 16)
    assert (vt[:8] == v[732:740].view(np.uint16)).all() and (vt[8:] == 0).all()


# ------------------------------------------------------------- attention sinks
def _sink_inp(T=200, H=2, seed=11):
    w = S.LLAMA31_8B_128K.scaled(n_q_heads=4 * H, n_kv_heads=H, context=T, seed=seed)
    return w, S.generate(w)


def test_sink_zero_is_the_plain_cache():
    w, inp = _sink_inp(T=160)
    a = O.quantize_sequence(inp["K"][0], inp["V"][0], 160, 32, 2)
    b = O.quantize_sequence(inp["K"][0], inp["V"][0], 160, 32, 2, n_sink_cap=0)
    assert b["n_sink"] == 0 and (a["k_codes"] == b["k_codes"]).all()
    np.testing.assert_array_equal(O.sequence_attention(inp["q"][0], a, w.sm_scale),
                                  O.sequence_attention(inp["q"][0], b, w.sm_scale))


def test_sink_rows_are_exact_and_groups_start_after_them():
    # 4 sinks, 128 quantized tokens, 20 tail tokens: the groups are those of a
    # plain cache over tokens [4, 152), the sinks the fp16 rows themselves
    w, inp = _sink_inp(T=152)
    st = O.quantize_sequence(inp["K"][0], inp["V"][0], 152, 20, 4, n_sink_cap=4)
    assert (st["n_sink"], st["n_quant"], st["n_tail"]) == (4, 128, 20)
    plain = O.quantize_sequence(inp["K"][0][4:], inp["V"][0][4:], 148, 20, 4)
    for f in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero"):
        assert (st[f].view(np.uint8) == plain[f].view(np.uint8)).all(), f
    keys, values = O.sequence_kv(st)
    k0 = np.swapaxes(inp["K"][0][:4], 0, 1).astype(np.float64)
    assert (keys[:, :4] == k0).all()


def test_all_sink_sequence_is_exact_attention():
    # fewer tokens than the sink window: everything stays fp16, attention = SDPA
    w, inp = _sink_inp(T=40)
    st = O.quantize_sequence(inp["K"][0], inp["V"][0], 24, 0, 2, n_sink_cap=32)
    assert (st["n_sink"], st["n_quant"], st["n_tail"]) == (24, 0, 0)
    k = np.swapaxes(inp["K"][0][:24], 0, 1).astype(np.float64)
    v = np.swapaxes(inp["V"][0][:24], 0, 1).astype(np.float64)
    ref = _sdpa64(inp["q"][0], np.repeat(k, 4, 0), np.repeat(v, 4, 0), w.sm_scale)
    np.testing.assert_allclose(O.sequence_attention(inp["q"][0], st, w.sm_scale), ref, atol=1e-12)


def test_append_with_sinks_fills_the_window_then_the_tail():
    # after n tokens: min(n, S) sinks, and the plain append state of the rest
    S_, R = 5, 32
    state = (0, 0, 0)
    plain = (0, 0)
    for n in range(1, 200):
        state = O.append_lengths_sink(*state, S_, R)
        if n > S_:
            plain = O.append_lengths(*plain, R)[:2]
        assert state == (min(n, S_),) + plain, n


# ------------------------------------------------------------- pre-RoPE keys
def test_rope_rotation_by_hand():
    # one pair (D = 2): theta_0 = 1, so the key at position t turns by t radians
    k = np.array([[1.0, 0.0], [0.0, 2.0], [3.0, 4.0]])
    got = O.rope_rotate(k, np.array([0, 1, 2]), 10000.0)
    assert np.allclose(got[0], [1.0, 0.0])
    assert np.allclose(got[1], [-2.0 * math.sin(1.0), 2.0 * math.cos(1.0)])
    assert np.allclose(got[2], [3 * math.cos(2.0) - 4 * math.sin(2.0), 3 * math.sin(2.0) + 4 * math.cos(2.0)])
    # theta_i = base^(-2i/D): D = 4, base 100 -> theta_1 = 0.1
    assert np.allclose(O.rope_angles(np.array([5]), 4, 100.0), [[5.0, 0.5]])


def test_rope_preserves_norms_and_relative_scores():
    rng = np.random.default_rng(7)
    k = rng.standard_normal((6, 16))
    q = rng.standard_normal(16)
    pos = np.arange(6) + 3
    rk = O.rope_rotate(k, pos, 500000.0)
    assert np.allclose(np.linalg.norm(rk, axis=1), np.linalg.norm(k, axis=1))
    # q at position p against keys at t depends on p - t only: shift both by 11
    rq = O.rope_rotate(q[None], np.array([9]), 500000.0)[0]
    rq2 = O.rope_rotate(q[None], np.array([20]), 500000.0)[0]
    rk2 = O.rope_rotate(k, pos + 11, 500000.0)
    assert np.allclose(rk @ rq, rk2 @ rq2)


def test_rope_attention_position_zero_is_plain():
    # a single cached token sits at position 0: no rotation, plain attention
    rng = np.random.default_rng(8)
    k16 = rng.standard_normal((1, 1, 64)).astype(np.float16)
    v16 = rng.standard_normal((1, 1, 64)).astype(np.float16)
    st = O.quantize_sequence(k16, v16, 1, 1, 2)
    q = rng.standard_normal((2, 64)).astype(np.float16)
    assert np.allclose(O.sequence_attention_rope(q, st, 0.125, 10000.0), O.sequence_attention(q, st, 0.125))
