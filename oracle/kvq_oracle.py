"""CPU oracle for asymmetric low-bit KV-cache quantization and decode attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline and reference legs of ``bench.py`` may import this module.  It
shares no code with the CUDA path and imports nothing from it.

Everything here is the plain definition, written for a reader to check against
the pages by eye:

* Uniform asymmetric integer quantization per group (ihal.it article,
  paragraph 3): a group's range [min, max] is divided into the 2^b levels of a
  b-bit code, with a scale factor and a zero point per group.
* Grouping axes (same article, paragraphs 1, 4-6): keys are grouped per
  channel (one channel over 32 consecutive tokens), values per token (32
  consecutive channels of one token), group size 32.
* Recent tokens kept in full precision (same article, paragraph 8): tokens that
  do not yet fill a 32-token key group stay in an fp16 tail and are quantized
  in groups once enough have arrived.
* Decode attention (same article, paragraphs 2 and 5): the output is a
  softmax-weighted sum of value vectors over every cached token, computed here
  in float64 over the dequantized cache.
* Attention-sink windows (same article, paragraph 9): the first tokens of a
  sequence may stay fp16 beside the recent tail.
* Pre-RoPE keys (same article, paragraph 7 and the closing paragraph): keys are
  quantized before the rotary position embedding and rotated to their
  positions after dequantization.
* The mixed-width packed layout (RDKV summary, gist.science 2605.08317,
  sections 2.1-2.2 and "2.2 TriZone"): widths {0,2,4,8,16} per V token, width
  0 = evicted, 16 = kept in fp16; K channels at {2,4,8} bits for kept tokens
  only; rows grouped by width; fresh tokens fp16.

Readings taken where the pages are silent (all of them are listed in the
design notes of the repository):

* scale = fp16( fp32(max - min) / (2^b - 1) ), zero = fp16(min); both -0 -> +0.
* code = clamp( rint_half_even( (fp32(x) - fp32(zero_h)) / fp32(scale_h) ),
  0, 2^b - 1 ) with every fp32 operation rounded to nearest even, computed
  against the STORED fp16 scale and zero; a zero stored scale gives code 0.
* dequantized value = fp64(zero_h) + fp64(scale_h) * code (exact in fp64).
* An empty context (no cached token) gives an all-zero output.
"""
from __future__ import annotations

import functools

import numpy as np

GROUP = 32
F16 = np.float16
F32 = np.float32
F64 = np.float64


# ---------------------------------------------------------------------------
# Quantizer (ihal.it article, paragraph 3: range split into 2^b levels with a
# scale factor and zero point per group).
# ---------------------------------------------------------------------------
def quantize_groups(x16: np.ndarray, bits: int):
    """Quantize groups along the last axis.

    x16: float16 [..., n] (n = 32 for full groups; fewer for a partial group).
    Returns (codes uint8 [..., n], scale float16 [...], zero float16 [...]).
    """
    if bits not in (2, 4, 8):
        raise ValueError(f"bits must be 2, 4 or 8, got {bits}")
    x16 = np.asarray(x16, dtype=F16)
    x = x16.astype(F32)
    if not np.all(np.isfinite(x)):
        raise ValueError("inputs must be finite")
    # 1. group min / max, as fp32 values (exact for fp16 inputs)
    mn = x.min(axis=-1)
    mx = x.max(axis=-1)
    # 2. range and scale in IEEE fp32, round to nearest even
    rng = (mx - mn).astype(F32)
    scale32 = (rng / F32(2 ** bits - 1)).astype(F32)
    # 3. stored fp16 scale and zero point, -0 canonicalised to +0
    scale_h = scale32.astype(F16)
    zero_h = mn.astype(F16)
    scale_h = np.where(scale_h == 0, F16(0.0), scale_h).astype(F16)
    zero_h = np.where(zero_h == 0, F16(0.0), zero_h).astype(F16)
    # 4. codes against the stored scale and zero, fp32 subtract and divide,
    #    round half to even, clamp to [0, 2^b - 1]; zero scale -> code 0
    s = scale_h.astype(F32)[..., None]
    z = zero_h.astype(F32)[..., None]
    diff = (x - z).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = (diff / s).astype(F32)
    code = np.rint(quot)
    code = np.clip(code, 0, 2 ** bits - 1)
    code = np.where(s == 0, 0.0, code)
    return code.astype(np.uint8), scale_h, zero_h


def dequantize(codes: np.ndarray, scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """x_hat = zero + scale * code, in float64 (exact).  scale/zero broadcast
    against codes' last axis the way quantize_groups produced them."""
    return zero.astype(F64)[..., None] + scale.astype(F64)[..., None] * codes.astype(F64)


def quantize_keys(k16: np.ndarray, bits: int):
    """Keys, per channel over 32-token spans (article, paragraph 4).

    k16: float16 [..., n, D] with n a multiple of 32.
    Returns codes uint8 [..., n, D], scale/zero float16 [..., n/32, D].
    """
    *lead, n, d = k16.shape
    if n % GROUP:
        raise ValueError("key groups need whole 32-token spans")
    x = k16.reshape(*lead, n // GROUP, GROUP, d)
    x = np.swapaxes(x, -1, -2)  # [..., G, D, 32]: one channel over 32 tokens
    c, s, z = quantize_groups(x, bits)
    c = np.swapaxes(c, -1, -2).reshape(*lead, n, d)
    return c, s, z


def dequantize_keys(codes, scale, zero) -> np.ndarray:
    """Inverse view of quantize_keys, float64 [..., n, D]."""
    *lead, n, d = codes.shape
    c = np.swapaxes(codes.reshape(*lead, n // GROUP, GROUP, d), -1, -2)
    x = dequantize(c, scale, zero)  # [..., G, D, 32]
    return np.swapaxes(x, -1, -2).reshape(*lead, n, d)


def quantize_values(v16: np.ndarray, bits: int):
    """Values, per token over 32-channel spans (article, paragraphs 5-6).

    v16: float16 [..., n, D] with D a multiple of 32.
    Returns codes uint8 [..., n, D], scale/zero float16 [..., n, D/32].
    """
    *lead, n, d = v16.shape
    x = v16.reshape(*lead, n, d // GROUP, GROUP)
    c, s, z = quantize_groups(x, bits)
    return c.reshape(*lead, n, d), s, z


def dequantize_values(codes, scale, zero) -> np.ndarray:
    *lead, n, d = codes.shape
    x = dequantize(codes.reshape(*lead, n, d // GROUP, GROUP), scale, zero)
    return x.reshape(*lead, n, d)


# ---------------------------------------------------------------------------
# Decode attention (article, paragraphs 2 and 5): one query per head attends to
# every cached token; output = softmax-weighted sum of value vectors.
# ---------------------------------------------------------------------------
def decode_attention(q16: np.ndarray, keys: np.ndarray, values: np.ndarray,
                     sm_scale: float) -> np.ndarray:
    """q16: float16 [Hq, D]; keys/values: float64 [Hkv, N, D].  Query head h reads
    KV head h // (Hq / Hkv).  Returns float64 [Hq, D]."""
    hq, d = q16.shape
    hkv = keys.shape[0]
    group = hq // hkv
    out = np.zeros((hq, d), dtype=F64)
    if keys.shape[1] == 0:
        return out
    for h in range(hq):
        kh = h // group
        logits = sm_scale * (keys[kh] @ q16[h].astype(F64))
        p = np.exp(logits - logits.max())
        p /= p.sum()
        out[h] = p @ values[kh]
    return out


# ---------------------------------------------------------------------------
# Uniform cache state: tokens [0, n_quant) quantized in 32-token groups, tokens
# [n_quant, n_quant + n_tail) kept fp16 (article, paragraph 8).
# ---------------------------------------------------------------------------
def split_sequence(seq_len: int, n_tail: int, n_sink_cap: int = 0):
    """(n_sink, n_quant) of a sequence: the first min(n_sink_cap, seq_len) tokens
    are sinks, the last n_tail tokens the tail, the rest whole 32-token groups."""
    n_sink = min(n_sink_cap, seq_len)
    n_quant = seq_len - n_sink - n_tail
    if n_quant < 0 or n_quant % GROUP:
        raise ValueError("quantized region must be a whole number of 32-token groups")
    return n_sink, n_quant


def quantize_sequence(k16: np.ndarray, v16: np.ndarray, seq_len: int, n_tail: int,
                      bits: int, n_sink_cap: int = 0) -> dict:
    """One sequence.  k16/v16: float16 [T, Hkv, D] (T >= seq_len).
    Returns per-head arrays (leading axis Hkv).

    Attention sinks ("KV-cache quantization axes", ihal.it, paragraph 9: high-
    precision windows for the recent tokens and for the attention sinks): with
    n_sink_cap > 0 the first min(n_sink_cap, seq_len) tokens stay fp16 and the
    quantized groups start after them."""
    n_sink, n_quant = split_sequence(seq_len, n_tail, n_sink_cap)
    k = np.ascontiguousarray(np.swapaxes(k16[:seq_len], 0, 1))  # [Hkv, T, D]
    v = np.ascontiguousarray(np.swapaxes(v16[:seq_len], 0, 1))
    q0, q1 = n_sink, n_sink + n_quant
    kc, ks, kz = quantize_keys(k[:, q0:q1], bits)
    vc, vs, vz = quantize_values(v[:, q0:q1], bits)
    return {
        "bits": bits, "n_quant": n_quant, "n_tail": n_tail, "n_sink": n_sink,
        "k_codes": kc, "k_scale": ks, "k_zero": kz,
        "v_codes": vc, "v_scale": vs, "v_zero": vz,
        "k_tail": k[:, q1:seq_len], "v_tail": v[:, q1:seq_len],
        "k_sink": k[:, :n_sink], "v_sink": v[:, :n_sink],
    }


def sequence_kv(state: dict):
    """Dequantized keys and values of a sequence, float64 [Hkv, n, D]: the fp16
    sinks, the quantized region, then the fp16 tail (exact in float64)."""
    kq = dequantize_keys(state["k_codes"], state["k_scale"], state["k_zero"])
    vq = dequantize_values(state["v_codes"], state["v_scale"], state["v_zero"])
    ks = state.get("k_sink", kq[:, :0]).astype(F64)
    vs = state.get("v_sink", vq[:, :0]).astype(F64)
    keys = np.concatenate([ks, kq, state["k_tail"].astype(F64)], axis=1)
    values = np.concatenate([vs, vq, state["v_tail"].astype(F64)], axis=1)
    return keys, values


def sequence_attention(q16: np.ndarray, state: dict, sm_scale: float) -> np.ndarray:
    keys, values = sequence_kv(state)
    return decode_attention(q16, keys, values, sm_scale)


# ---------------------------------------------------------------------------
# Pre-RoPE keys ("KV-cache quantization axes", ihal.it, paragraph 7 and the
# closing paragraph: keys are quantized before the rotary position embedding and
# the rotation is applied after dequantization).  Readings: RoPE rotates the
# adjacent channel pairs (2i, 2i+1) of a key at position t by the angle
# t * theta_i, theta_i = base^(-2i/D); a token's position is its index in the
# sequence (sinks, then the quantized groups, then the tail); the query is given
# already rotated to its own position.
# ---------------------------------------------------------------------------
def rope_angles(positions: np.ndarray, d: int, base: float) -> np.ndarray:
    """Angles t * theta_i, float64 [len(positions), d/2]."""
    i = np.arange(d // 2, dtype=F64)
    theta = np.power(F64(base), -2.0 * i / d)
    return np.asarray(positions, dtype=F64)[:, None] * theta[None, :]


def rope_rotate(keys: np.ndarray, positions: np.ndarray, base: float) -> np.ndarray:
    """keys float64 [..., N, D] rotated pair by pair: (k0, k1) ->
    (k0 cos - k1 sin, k0 sin + k1 cos) with the angle of each token's position."""
    keys = np.asarray(keys, dtype=F64)
    ang = rope_angles(positions, keys.shape[-1], base)
    c, s = np.cos(ang), np.sin(ang)
    k0, k1 = keys[..., 0::2], keys[..., 1::2]
    out = np.empty_like(keys)
    out[..., 0::2] = k0 * c - k1 * s
    out[..., 1::2] = k0 * s + k1 * c
    return out


def sequence_attention_rope(q16: np.ndarray, state: dict, sm_scale: float, base: float) -> np.ndarray:
    """Decode attention over a cache of pre-RoPE keys: every key (sinks,
    dequantized groups, tail) is rotated to its position after dequantization."""
    keys, values = sequence_kv(state)
    keys = rope_rotate(keys, np.arange(keys.shape[1]), base)
    return decode_attention(q16, keys, values, sm_scale)


def append_lengths(n_quant: int, n_tail: int, tail_cap: int):
    """Lengths after appending one token (article, paragraph 8): when the tail
    is full, its oldest 32 tokens become the next quantized group first."""
    flushed = n_tail == tail_cap
    if flushed:
        n_quant += GROUP
        n_tail -= GROUP
    return n_quant, n_tail + 1, flushed


def append_lengths_sink(n_sink: int, n_quant: int, n_tail: int, sink_cap: int, tail_cap: int):
    """Lengths after appending one token with a sink window: the token is a sink
    while fewer than sink_cap tokens have arrived, else as append_lengths."""
    if n_sink < sink_cap:
        return n_sink + 1, n_quant, n_tail
    n_quant, n_tail, _ = append_lengths(n_quant, n_tail, tail_cap)
    return n_sink, n_quant, n_tail


# ---------------------------------------------------------------------------
# Packed byte layout of the uniform cache.  The pages fix no bit layout; this is
# the library's own, written out from its specification:
#
# A tile holds the codes of 32 consecutive tokens x D channels at b bits.  It is
# cut into 32 lanes (gid = lane // 4, tig = lane % 4).  Each lane owns D/2 code
# PAIRS, enumerated in this order:
#   K tile: for kt in [0, D/16), mt in [0, 2), i in [0, 4):
#             token t = 16*mt + gid + 8*(i % 2), channel d = 16*kt + 2*tig + 8*(i // 2)
#             pair = (code[t][d], code[t][d + 1])
#   V tile: for mt in [0, D/16), kt in [0, 2), i in [0, 4):
#             channel d = 16*mt + gid + 8*(i % 2), token t = 16*kt + 2*tig + 8*(i // 2)
#             pair = (code[t][d], code[t + 1][d])
# Pair P of a lane goes to the lane's word P // (16/b), slot k = P % (16/b): the
# first code at bits [p, p + b), the second at bits [16 + p, 16 + p + b), with
# p = SLOT_BITPOS[b][k].  A lane's word w sits at byte ((w // 4) * 32 + lane) * 16
# + (w % 4) * 4 of the tile, little-endian.  Tile bytes: 32 * D * b / 8.
#
# Metadata, stored as pairs of fp16 values (32-bit words), each block holding a
# scale plane then a zero-point plane of D/2 pairs:
#   K, per group (the two planes interleaved): word 16*kt + 4*tig + 2*r + f
#                        (kt < D/16, tig < 4, r < 2, f < 2) = (x[c], x[c + 1]) of
#                        the zero points (f = 0) or the scales (f = 1) for channel
#                        c = 16*kt + 2*tig + 8*r (one 16-byte load gives a lane
#                        the zero points and scales of a k-tile)
#   V, per 32-token tile: pair index 16*j + 4*tig + 2*kt + r
#                        (tig < 4, j < D/32, kt < 2, r < 2)
#                        = (x[j][t], x[j][t + 1]) for channel group j and token
#                        t = 16*kt + 2*tig + 8*r of the tile
# ---------------------------------------------------------------------------
SLOT_BITPOS = {2: (0, 2, 8, 10, 4, 6, 12, 14), 4: (0, 4, 8, 12), 8: (0, 8), 16: (0,)}


@functools.lru_cache(maxsize=None)
def tile_code_positions(kind: str, d: int, bits: int):
    """Word index and bit offset of every code of a 32 x D tile.
    Returns (word int64 [32, D], bit int64 [32, D])."""
    if kind not in ("K", "V"):
        raise ValueError(kind)
    per_word = 16 // bits
    word = np.full((GROUP, d), -1, dtype=np.int64)
    bit = np.full((GROUP, d), -1, dtype=np.int64)
    for lane in range(32):
        gid, tig = lane // 4, lane % 4
        pairs = []
        if kind == "K":
            for kt in range(d // 16):
                for mt in range(2):
                    for i in range(4):
                        t = 16 * mt + gid + 8 * (i % 2)
                        c = 16 * kt + 2 * tig + 8 * (i // 2)
                        pairs.append(((t, c), (t, c + 1)))
        else:
            for mt in range(d // 16):
                for kt in range(2):
                    for i in range(4):
                        c = 16 * mt + gid + 8 * (i % 2)
                        t = 16 * kt + 2 * tig + 8 * (i // 2)
                        pairs.append(((t, c), (t + 1, c)))
        for p, (first, second) in enumerate(pairs):
            w, k = p // per_word, p % per_word
            gword = ((w // 4) * 32 + lane) * 4 + (w % 4)
            pos = SLOT_BITPOS[bits][k]
            for (t, c), off in ((first, pos), (second, 16 + pos)):
                assert word[t, c] == -1, "layout must place each code once"
                word[t, c] = gword
                bit[t, c] = off
    assert (word >= 0).all()
    word.setflags(write=False)
    bit.setflags(write=False)
    return word, bit


def tile_bytes(d: int, bits: int) -> int:
    return GROUP * d * bits // 8


def pack_tiles(codes: np.ndarray, kind: str, bits: int) -> np.ndarray:
    """codes uint8 [..., 32, D] (token, channel) -> packed uint8 [..., 32*D*b/8]."""
    *lead, n, d = codes.shape
    assert n == GROUP
    word, bit = tile_code_positions(kind, d, bits)
    n_words = GROUP * d * bits // 32
    flat = codes.reshape(*lead, GROUP * d).astype(np.uint32)
    w_flat, b_flat = word.ravel(), bit.ravel()
    # every code ORs into its own bit field of its word (fields never overlap)
    order = np.argsort(w_flat, kind="stable")
    per = 32 // bits
    gathered = flat[..., order].reshape(*lead, n_words, per)
    shifts = b_flat[order].reshape(n_words, per).astype(np.uint32)
    out = np.ascontiguousarray(np.bitwise_or.reduce(gathered << shifts, axis=-1), dtype="<u4")
    return out.view(np.uint8).reshape(*lead, n_words * 4)


def unpack_tiles(packed: np.ndarray, kind: str, d: int, bits: int) -> np.ndarray:
    """Inverse of pack_tiles: packed uint8 [..., 32*D*b/8] -> codes uint8 [..., 32, D]
    (uint16 for 16-bit fields)."""
    *lead, nb = packed.shape
    words = np.ascontiguousarray(packed).view("<u4").astype(np.uint32)
    word, bit = tile_code_positions(kind, d, bits)
    vals = (words[..., word] >> bit.astype(np.uint32)) & np.uint32(2 ** bits - 1)
    return vals.astype(np.uint16 if bits == 16 else np.uint8)


@functools.lru_cache(maxsize=None)
def key_meta_order(d: int) -> np.ndarray:
    """(field, channel) of every fp16 slot of a key metadata block (2D slots):
    field 0 = zero point, 1 = scale; int64 [2D, 2]."""
    order = np.full((2 * d, 2), -1, dtype=np.int64)
    for kt in range(d // 16):
        for tig in range(4):
            for r in range(2):
                for f in range(2):
                    w = 16 * kt + 4 * tig + 2 * r + f
                    c = 16 * kt + 2 * tig + 8 * r
                    order[2 * w] = (f, c)
                    order[2 * w + 1] = (f, c + 1)
    assert sorted(map(tuple, order.tolist())) == [(f, c) for f in range(2) for c in range(d)]
    order.setflags(write=False)
    return order


@functools.lru_cache(maxsize=None)
def value_meta_order(d: int) -> np.ndarray:
    """(channel group j) * 32 + token t of every fp16 slot of a value metadata
    plane (length D)."""
    order = np.full(d, -1, dtype=np.int64)
    for tig in range(4):
        for j in range(d // GROUP):
            for kt in range(2):
                for r in range(2):
                    pair = 16 * j + 4 * tig + 2 * kt + r
                    t = 16 * kt + 2 * tig + 8 * r
                    order[2 * pair], order[2 * pair + 1] = j * GROUP + t, j * GROUP + t + 1
    assert sorted(order.tolist()) == list(range(d))
    order.setflags(write=False)
    return order


def pack_key_meta(scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """scale/zero float16 [..., D] of key groups -> float16 [..., 2, D] block (the
    2D slots in key_meta_order, viewed as two rows of D)."""
    d = scale.shape[-1]
    order = key_meta_order(d)
    both = np.stack([zero, scale], axis=-2)  # field 0 = zero, 1 = scale
    flat = both[..., order[:, 0], order[:, 1]]
    return flat.reshape(flat.shape[:-1] + (2, d))


def pack_value_meta(scale: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """scale/zero float16 [..., 32, D/32] (token, channel group) of one value tile
    -> float16 [..., 2, D] block."""
    d = scale.shape[-1] * GROUP
    order = value_meta_order(d)
    flat_s = np.swapaxes(scale, -1, -2).reshape(*scale.shape[:-2], d)  # j * 32 + t
    flat_z = np.swapaxes(zero, -1, -2).reshape(*zero.shape[:-2], d)
    return np.stack([flat_s[..., order], flat_z[..., order]], axis=-2)


# ---------------------------------------------------------------------------
# Mixed-width cache (RDKV summary, sections 2.1-2.2 and "2.2 TriZone").
#
# Per (sequence, KV head): every old token t has a V width in {0,2,4,8,16}
# (0 = evicted, 16 = fp16) and every channel d a K width in {2,4,8}; K is kept
# only for kept tokens.  Kept tokens are grouped by V width (stable, widths in
# ascending order), and each width class is cut into consecutive 32-token
# blocks (the last block of a class may be partial), so every block has one V
# width.  A block's V rows are quantized per token over 32-channel spans at the
# block's width (width 16: fp16 rows).  A block's K is quantized per channel
# over the block's tokens at that channel's width.  Fresh tokens stay fp16.
# ---------------------------------------------------------------------------
TRIZONE_V_WIDTHS = (2, 4, 8, 16)
TRIZONE_K_WIDTHS = (2, 4, 8)


def trizone_blocks(v_width: np.ndarray):
    """Stream order of the kept old tokens: list of (width, token indices)."""
    blocks = []
    for w in TRIZONE_V_WIDTHS:
        toks = np.nonzero(v_width == w)[0]
        for i in range(0, len(toks), GROUP):
            blocks.append((w, toks[i:i + GROUP]))
    return blocks


def trizone_quantize(k16: np.ndarray, v16: np.ndarray, v_width: np.ndarray,
                     k_width: np.ndarray) -> dict:
    """One (sequence, KV head).  k16/v16: float16 [T, D]; the first len(v_width)
    tokens are old, the rest fresh."""
    t_old = len(v_width)
    d = k16.shape[1]
    out_blocks = []
    for w, toks in trizone_blocks(v_width):
        kb = k16[toks]  # [n, D]
        blk = {"width": int(w), "tokens": toks,
               "k_codes": np.zeros((len(toks), d), np.uint8),
               "k_scale": np.zeros((d,), F16), "k_zero": np.zeros((d,), F16)}
        for kw in TRIZONE_K_WIDTHS:
            ch = np.nonzero(k_width == kw)[0]
            if len(ch) == 0:
                continue
            c, s, z = quantize_groups(kb[:, ch].T, kw)  # one group per channel
            blk["k_codes"][:, ch] = c.T
            blk["k_scale"][ch] = s
            blk["k_zero"][ch] = z
        if w == 16:
            blk["v_fp16"] = v16[toks]
        else:
            c, s, z = quantize_values(v16[toks], w)
            blk.update(v_codes=c, v_scale=s, v_zero=z)
        out_blocks.append(blk)
    return {"blocks": out_blocks, "fresh_k": k16[t_old:], "fresh_v": v16[t_old:],
            "k_width": k_width, "t_old": t_old}


def trizone_kv(tz: dict):
    """Dequantized keys/values float64 [n, D] of the kept old tokens in ORIGINAL
    token order, followed by the fresh tokens."""
    d = tz["fresh_k"].shape[1]
    kept, keys, values = [], [], []
    for blk in tz["blocks"]:
        khat = (blk["k_zero"].astype(F64)[None, :]
                + blk["k_scale"].astype(F64)[None, :] * blk["k_codes"].astype(F64))
        if blk["width"] == 16:
            vhat = blk["v_fp16"].astype(F64)
        else:
            vhat = dequantize_values(blk["v_codes"], blk["v_scale"], blk["v_zero"])
        kept.append(blk["tokens"])
        keys.append(khat)
        values.append(vhat)
    if kept:
        order = np.argsort(np.concatenate(kept), kind="stable")
        keys = np.concatenate(keys)[order]
        values = np.concatenate(values)[order]
    else:
        keys = np.zeros((0, d))
        values = np.zeros((0, d))
    keys = np.concatenate([keys, tz["fresh_k"].astype(F64)])
    values = np.concatenate([values, tz["fresh_v"].astype(F64)])
    return keys, values


def trizone_attention(q16: np.ndarray, tz_heads: list, sm_scale: float) -> np.ndarray:
    """q16 float16 [Hq, D]; tz_heads: trizone_quantize output per KV head."""
    kv = [trizone_kv(tz) for tz in tz_heads]
    out = np.zeros(q16.shape, dtype=F64)
    group = q16.shape[0] // len(tz_heads)
    for kh, (keys, values) in enumerate(kv):
        sl = slice(kh * group, (kh + 1) * group)
        out[sl] = decode_attention(q16[sl], keys[None], values[None], sm_scale)
    return out


# ---------------------------------------------------------------------------
# Packed byte layout of the mixed-width cache (the library's own; the pages
# describe the zones, not their bytes):
#
# Channels of a (sequence, KV head) are permuted by K width class: the 2-bit
# channels in ascending order, then 4-bit, then 8-bit; each class is padded to
# whole 16-channel k-tiles with "pad" slots (code 0, scale 0, zero 0).
#
# One 32-token block (tokens of one V-width class, in stream order) is one
# contiguous record:
#   K codes: for each K class c (2, 4, 8) with kt_c k-tiles: 32 tokens x 16*kt_c
#     channels at c bits; lane L (gid = L//4, tig = L%4) owns the pairs
#     (kt < kt_c, mt < 2, i < 4): token 16mt + gid + 8(i%2), class channels
#     16kt + 2tig + 8(i//2) and +1; pair P -> word P // (16/c), slot P % (16/c)
#     at bit SLOT_BITPOS[c][slot] (+16 for the second code); lane word w at byte
#     (w*32 + L)*4 of the sub-tile (64 * kt_c * c bytes).
#   K metadata: 16 * KT half pairs (KT = sum kt_c, k-tiles of all classes in
#     order); pair 16kt + 4tig + 2r + f holds the zero points (f = 0) or the
#     scales (f = 1) of permuted slots 16kt + 2tig + 8r and +1 (the key order of
#     the uniform cache, over k-tiles of mixed widths).
#   V: width 2/4/8: the uniform value tile at that width (pack_tiles "V") and its
#     metadata block (pack_value_meta); width 16: the fp16 values as a 16-bit value
#     tile (pack_tiles "V" with 16-bit fields: word = half2 of tokens t, t + 1 of
#     one channel), the A fragments of P.V as they are.
#   Tokens past the block's count are zero everywhere.
# Fresh tokens form "fresh blocks" of up to 32 tokens: the fp16 keys as a 16-bit
# key tile (natural channel order; word = half2 of channels c, c + 1 of one token,
# the A fragments of Q.K^T) followed by the fp16 values as a 16-bit value tile.
# A (sequence, KV head) stores its blocks class by class (V width 2, 4, 8, 16),
# then its fresh blocks; all blocks of one kind have the same size.
#
# Index record of a (sequence, KV head), 512 bytes: int32 fields
#   [0:4] kept tokens per V width (2, 4, 8, 16), [4] fresh tokens,
#   [5:9] blocks per V width, [9] fresh blocks, [10:13] channels per K width
#   (2, 4, 8), [13:16] k-tiles per K width, [16:21] bytes of one block of each
#   kind (widths 2, 4, 8, 16, fresh), [21:26] byte offset of each kind's first
#   block, [26] total bytes, [27:32] zero;
# then int16 [160] permuted channel slots (-1 = pad, and past the last k-tile),
# then 64 zero bytes.
# ---------------------------------------------------------------------------
TRIZONE_KT_MAX = 10  # sum of ceil(n_c / 16) over three classes of 128 channels


def trizone_channel_order(k_width: np.ndarray):
    """Permuted channel slots (original channel, or -1 for a pad slot) and the
    k-tiles per K class."""
    slots, kts = [], []
    for c in TRIZONE_K_WIDTHS:
        ch = [int(d) for d in np.nonzero(k_width == c)[0]]
        kt = (len(ch) + 15) // 16
        slots += ch + [-1] * (16 * kt - len(ch))
        kts.append(kt)
    return np.asarray(slots, dtype=np.int64), tuple(kts)


@functools.lru_cache(maxsize=None)
def trizone_ksub_positions(kt: int, c: int):
    """(word, bit) of every code of a K sub-tile [32 tokens, 16*kt channels]."""
    per_word = 16 // c
    n = 16 * kt
    word = np.full((GROUP, n), -1, dtype=np.int64)
    bit = np.full((GROUP, n), -1, dtype=np.int64)
    for lane in range(32):
        gid, tig = lane // 4, lane % 4
        p = 0
        for k in range(kt):
            for mt in range(2):
                for i in range(4):
                    t = 16 * mt + gid + 8 * (i % 2)
                    ch = 16 * k + 2 * tig + 8 * (i // 2)
                    w, s = p // per_word, p % per_word
                    pos = SLOT_BITPOS[c][s]
                    for cc, off in ((ch, pos), (ch + 1, 16 + pos)):
                        assert word[t, cc] == -1
                        word[t, cc] = w * 32 + lane
                        bit[t, cc] = off
                    p += 1
    assert (word >= 0).all()
    word.setflags(write=False)
    bit.setflags(write=False)
    return word, bit


def _pack_words(codes: np.ndarray, word: np.ndarray, bit: np.ndarray, n_words: int) -> np.ndarray:
    out = np.zeros(n_words, dtype=np.uint64)
    np.add.at(out, word.ravel(), codes.ravel().astype(np.uint64) << bit.ravel().astype(np.uint64))
    return out.astype("<u4").view(np.uint8)


TRIZONE_FRESH_BLOCK = 2 * GROUP * 128 * 2  # fp16 key tile + fp16 value tile, D = 128
TRIZONE_INDEX_BYTES = 512


def trizone_block_bytes(kts, width: int, d: int = 128) -> int:
    kb = sum(64 * kt * c for kt, c in zip(kts, TRIZONE_K_WIDTHS)) + 64 * sum(kts)
    vb = GROUP * d * 2 if width == 16 else GROUP * d * width // 8 + 4 * d
    return kb + vb


def _fp16_tile(rows16: np.ndarray, kind: str, d: int) -> np.ndarray:
    """fp16 rows [n <= 32, D] -> 16-bit tile bytes (rows past n are zero)."""
    bits = np.zeros((GROUP, d), np.uint16)
    bits[:len(rows16)] = np.asarray(rows16, F16).view(np.uint16)
    return pack_tiles(bits, kind, 16)


def trizone_pack_block(blk: dict, slots: np.ndarray, kts, d: int = 128) -> np.ndarray:
    """Bytes of one block record (trizone_quantize block -> uint8 array)."""
    n = len(blk["tokens"])
    parts = []
    # K codes per class, channels permuted, tokens padded to 32
    codes = np.zeros((GROUP, len(slots)), dtype=np.uint8)
    valid = slots >= 0
    codes[:n, valid] = blk["k_codes"][:, slots[valid]]
    base = 0
    for kt, c in zip(kts, TRIZONE_K_WIDTHS):
        if kt:
            word, bit = trizone_ksub_positions(kt, c)
            parts.append(_pack_words(codes[:, base:base + 16 * kt], word, bit, 16 * kt * c))
        base += 16 * kt
    # K metadata, lane order over all k-tiles, zero points and scales interleaved
    kt_all = sum(kts)
    fields = np.zeros((2, 16 * kt_all), np.float16)  # [zero, scale] per permuted slot
    fields[0, valid] = blk["k_zero"][slots[valid]]
    fields[1, valid] = blk["k_scale"][slots[valid]]
    meta = np.empty(32 * kt_all, np.float16)
    for kt in range(kt_all):
        for tig in range(4):
            for r in range(2):
                s = 16 * kt + 2 * tig + 8 * r
                for f in range(2):
                    pr = 16 * kt + 4 * tig + 2 * r + f
                    meta[2 * pr], meta[2 * pr + 1] = fields[f, s], fields[f, s + 1]
    parts.append(meta.view(np.uint8))
    # V
    w = blk["width"]
    if w == 16:
        parts.append(_fp16_tile(blk["v_fp16"], "V", d))
    else:
        vc = np.zeros((GROUP, d), np.uint8)
        vc[:n] = blk["v_codes"]
        vs = np.zeros((GROUP, d // GROUP), np.float16)
        vz = np.zeros((GROUP, d // GROUP), np.float16)
        vs[:n], vz[:n] = blk["v_scale"], blk["v_zero"]
        parts.append(pack_tiles(vc, "V", w))
        parts.append(pack_value_meta(vs, vz).view(np.uint8).ravel())
    out = np.concatenate(parts)
    assert out.size == trizone_block_bytes(kts, w, d)
    return out


def trizone_pack_fresh(k16: np.ndarray, v16: np.ndarray, d: int = 128) -> list:
    """Fresh tokens -> fresh block records (32 tokens each, the last partial)."""
    out = []
    for i in range(0, len(k16), GROUP):
        out.append(np.concatenate([_fp16_tile(k16[i:i + GROUP], "K", d),
                                   _fp16_tile(v16[i:i + GROUP], "V", d)]))
    return out


def trizone_pack(tz: dict, d: int = 128) -> dict:
    """The packed form of one (sequence, KV head): index record, stream order of
    the kept tokens, and the block bytes back to back."""
    slots, kts = trizone_channel_order(tz["k_width"])
    n_tok = [0, 0, 0, 0]
    n_blk = [0, 0, 0, 0]
    recs, order = [], []
    for blk in tz["blocks"]:
        ci = TRIZONE_V_WIDTHS.index(blk["width"])
        n_tok[ci] += len(blk["tokens"])
        n_blk[ci] += 1
        recs.append(trizone_pack_block(blk, slots, kts, d))
        order.append(blk["tokens"])
    fresh = trizone_pack_fresh(tz["fresh_k"], tz["fresh_v"], d)
    recs += fresh
    rec_bytes = [trizone_block_bytes(kts, w, d) for w in TRIZONE_V_WIDTHS] + [TRIZONE_FRESH_BLOCK]
    counts = n_blk + [len(fresh)]
    offs = np.concatenate([[0], np.cumsum(np.multiply(counts, rec_bytes))]).tolist()
    hdr = np.zeros(32, np.int32)
    hdr[0:4] = n_tok
    hdr[4] = len(tz["fresh_k"])
    hdr[5:10] = counts
    hdr[10:13] = [int((tz["k_width"] == c).sum()) for c in TRIZONE_K_WIDTHS]
    hdr[13:16] = kts
    hdr[16:21] = rec_bytes
    hdr[21:26] = offs[:5]
    hdr[26] = offs[5]
    sl = np.full(160, -1, np.int16)
    sl[:len(slots)] = slots
    index = np.concatenate([hdr.view(np.uint8), sl.view(np.uint8), np.zeros(64, np.uint8)])
    assert index.size == TRIZONE_INDEX_BYTES
    data = np.concatenate(recs) if recs else np.zeros(0, np.uint8)
    assert data.size == offs[5]
    tokens = np.concatenate(order) if order else np.zeros(0, np.int64)
    return {"index": index, "tokens": tokens.astype(np.int32), "data": data,
            "slots": slots, "kts": kts, "header": hdr}
