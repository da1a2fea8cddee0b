"""The grouping-axis effects ("KV-cache quantization axes", ihal.it, paragraphs
3-6) measured on the library's own output: the per-channel keys and per-token
values are the codes and scales `kvq_quantize_prefill` wrote (read back from the
cache and unpacked through the oracle's layout description), and the end-to-end
leg is `kvq_decode_attn` itself.  The other axis of each comparison is the
oracle's quantizer run on the transposed grouping, the same data and width.
The input recipes are those of the CPU ablation (stable outlier key channels;
value rows of log-normal magnitude under sparse attention)."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from tests.test_axis_ablation import _keys, _values

pytestmark = pytest.mark.gpu

T, D, BITS = 1024, 128, 2


def _library_cache(k16: np.ndarray, v16: np.ndarray) -> kvq.QuantizedKVCache:
    """One sequence, one KV head, every token in whole 32-token groups."""
    cache = kvq.QuantizedKVCache(1, 1, D, BITS, T, 32)
    k = torch.from_numpy(k16.reshape(1, T, 1, D)).cuda()
    v = torch.from_numpy(v16.reshape(1, T, 1, D)).cuda()
    cache.prefill(k, v, [T], [0])
    torch.cuda.synchronize()
    return cache


def _library_keys(cache) -> np.ndarray:
    """Dequantized keys from the cache's key tiles and key metadata, float64 [T, D]."""
    views = cache.views()
    ng = T // 32
    codes = O.unpack_tiles(views["k_codes"][0, 0, :ng].cpu().numpy(), "K", D, BITS)  # [ng, 32, D]
    meta = views["k_meta"][0, 0, :ng].cpu().numpy().reshape(ng, 2 * D)
    order = O.key_meta_order(D)
    fields = np.zeros((ng, 2, D), np.float16)  # field 0 zero point, 1 scale
    fields[:, order[:, 0], order[:, 1]] = meta
    return O.dequantize_keys(codes.reshape(T, D), fields[:, 1], fields[:, 0])


def _library_values(cache) -> np.ndarray:
    """Dequantized values from the cache's value tiles and value metadata, float64 [T, D]."""
    views = cache.views()
    ng = T // 32
    codes = O.unpack_tiles(views["v_codes"][0, 0, :ng].cpu().numpy(), "V", D, BITS)  # [ng, 32, D]
    meta = views["v_meta"][0, 0, :ng].cpu().numpy().reshape(ng, 2, D)
    order = O.value_meta_order(D)  # slot -> channel group j * 32 + token t
    scale = np.zeros((ng, D), np.float16)
    zero = np.zeros((ng, D), np.float16)
    scale[:, order], zero[:, order] = meta[:, 0], meta[:, 1]
    # [ng, j, t] -> [ng, t, j] -> per token [T, D/32]
    scale = np.swapaxes(scale.reshape(ng, D // 32, 32), 1, 2).reshape(T, D // 32)
    zero = np.swapaxes(zero.reshape(ng, D // 32, 32), 1, 2).reshape(T, D // 32)
    return O.dequantize_values(codes.reshape(T, D), scale, zero)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


@pytest.mark.parametrize("seed", range(3))
def test_library_keys_per_channel_beat_per_token(seed):
    k16, q = _keys(seed, T, D)
    # values every 2-bit per-token group holds exactly (integers 0..3, each group
    # spanning 0 and 3), so the end-to-end leg below measures the keys alone
    rng = np.random.default_rng(500 + seed)
    vi = rng.integers(0, 4, (T, D))
    vi[:, 0::32], vi[:, 1::32] = 0, 3
    v16 = vi.astype(np.float16)
    cache = _library_cache(k16, v16)
    kf = k16.astype(np.float64)
    k_lib = _library_keys(cache)
    # the cache holds the oracle's per-channel codes exactly, and the values exactly
    c, s, z = O.quantize_keys(k16, BITS)
    assert np.array_equal(k_lib, O.dequantize_keys(c, s, z))
    assert np.array_equal(_library_values(cache), v16.astype(np.float64))
    c, s, z = O.quantize_values(k16, BITS)  # the other axis: per token over 32 channels
    k_tok = O.dequantize_values(c, s, z)
    assert _rel(k_lib, kf) * 2 < _rel(k_tok, kf)
    assert _rel(k_lib @ q, kf @ q) * 2 < _rel(k_tok @ q, kf @ q)
    # end to end: the library's decode against exact attention over the fp16 keys,
    # next to attention over per-token keys (same values)
    sm_scale = 1.0 / np.sqrt(D)
    q16 = q.astype(np.float16).reshape(1, 1, D)
    out = cache.decode(torch.from_numpy(q16).cuda(), sm_scale).cpu().numpy()[0, 0].astype(np.float64)
    vf = v16.astype(np.float64)[None]
    exact = O.decode_attention(q16[0], kf[None], vf, sm_scale)[0]
    tok = O.decode_attention(q16[0], k_tok[None], vf, sm_scale)[0]
    assert _rel(out, exact) * 2 < _rel(tok, exact), (_rel(out, exact), _rel(tok, exact))


def test_library_values_per_token_win_at_the_attention_output():
    ratios = []
    for seed in range(100, 108):
        v16, p = _values(seed, T, D)
        rng = np.random.default_rng(seed)
        k16 = (rng.standard_normal((T, D)) * 0.3).astype(np.float16)
        cache = _library_cache(k16, v16)
        vf = v16.astype(np.float64)
        v_lib = _library_values(cache)
        c, s, z = O.quantize_values(v16, BITS)
        assert np.array_equal(v_lib, O.dequantize_values(c, s, z))
        c, s, z = O.quantize_keys(v16, BITS)  # the other axis: per channel over 32 tokens
        v_ch = O.dequantize_keys(c, s, z)
        ref = p @ vf
        ratios.append(_rel(p @ v_ch, ref) / _rel(p @ v_lib, ref))
    assert np.mean(ratios) > 2.5, ratios
