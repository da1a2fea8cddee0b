"""GPU parity of the decode over pre-RoPE keys ("KV-cache quantization axes",
ihal.it, paragraph 7 and the closing paragraph: keys quantized before the rotary
position embedding, rotated after dequantization) against the oracle, through
the C ABI, within 2e-3 max-abs / 1e-3 mean-abs: every code width, GQA group
sizes 1-8, fp16 tails in the ring, sink windows whose length is not a multiple
of 32 (positions off the 32-token block grid), ragged batches, and appends."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu

BASE = 500000.0  # Llama-3.1's rotary base
# (workload, bits, sink window)
CASES = {
    "gqa4_2bit": (S.LLAMA31_8B_128K.scaled(context=2112, n_tail=64), 2, 0),
    "gqa4_4bit_sink5": (S.LLAMA31_8B_128K.scaled(context=1061, n_tail=0, bits=4), 4, 5),
    "gqa8_8bit": (S.LLAMA31_8B_128K.scaled(n_q_heads=64, context=544, n_tail=32, bits=8), 8, 0),
    "mha_2bit_sink3": (S.LLAMA2_13B.scaled(batch=2, n_q_heads=4, n_kv_heads=4, context=1027, n_tail=0), 2, 3),
    "gqa2_4bit": (S.LLAMA31_8B_128K.scaled(n_q_heads=16, context=800, n_tail=0, bits=4), 4, 0),
    "ragged_2bit_sink4": (S.SERVING.scaled(batch=3, context=1400, ragged=(40, 1400), bits=2), 2, 4),
}


def _inp(name):
    w, bits, sink = CASES[name]
    inp = S.generate(w)
    if w.ragged is not None or sink:  # tail = what is left after the window and whole groups
        inp["n_tail"] = ((inp["seq_len"] - np.minimum(sink, inp["seq_len"])) % 32).astype(np.int32)
    return w, bits, sink, inp


def _check(cache, inp, w, bits, sink, states=None):
    q = torch.from_numpy(inp["q"]).cuda()
    table = cache.rope_table(BASE)
    out = cache.decode_rope(q, table, w.sm_scale).cpu().numpy()
    assert cache.device_errors() == 0
    states = H.oracle_states(inp, bits, sink_cap=sink) if states is None else states
    for b, st in enumerate(states):
        ref = O.sequence_attention_rope(inp["q"][b], st, w.sm_scale, BASE)
        H.assert_close(out[b], ref)
    return out


@pytest.mark.parametrize("name", list(CASES))
def test_rope_decode_matches_oracle(name):
    w, bits, sink, inp = _inp(name)
    cache = H.device_cache(w, inp, bits, sink_cap=sink)
    _check(cache, inp, w, bits, sink)


def test_rope_differs_from_plain_decode():
    # the rotation matters: with real positions the two decodes disagree
    w, bits, sink, inp = _inp("gqa4_2bit")
    cache = H.device_cache(w, inp, bits)
    q = torch.from_numpy(inp["q"]).cuda()
    plain = cache.decode(q, w.sm_scale).cpu().numpy()
    rope = cache.decode_rope(q, cache.rope_table(BASE), w.sm_scale).cpu().numpy()
    assert np.abs(plain - rope).max() > 1e-2


def test_rope_after_appends():
    # tokens appended one by one (flushes included) keep their positions
    w = S.LLAMA31_8B_128K.scaled(context=200, n_tail=8)
    inp = S.generate(w)
    cache = H.device_cache(w, inp, 2, max_tokens=512)
    extra = S.generate(w.scaled(seed=77))
    for i in range(70):  # the 57th append flushes the full 64-token tail
        cache.append(torch.from_numpy(extra["K"][:, i]).cuda().contiguous(),
                     torch.from_numpy(extra["V"][:, i]).cuda().contiguous())
    kk = np.concatenate([inp["K"][0], extra["K"][0, :70]])
    vv = np.concatenate([inp["V"][0], extra["V"][0, :70]])
    nq, nt = 192, 8
    for _ in range(70):
        nq, nt, _ = O.append_lengths(nq, nt, w.tail_cap)
    assert nq == 224 and nt == 46
    st = O.quantize_sequence(kk, vv, 270, nt, 2)
    _check(cache, inp, w, 2, 0, states=[st])


def test_table_of_another_width_is_reported():
    # the fp16 pieces are cut for the cache's code width: a table built for a
    # 4-bit cache of the same geometry, used on a 2-bit cache, sets the device
    # error bit (both tables have the same size, so every read stays in bounds)
    w, bits, sink, inp = _inp("gqa4_2bit")
    c2 = H.device_cache(w, inp, 2)
    c4 = H.device_cache(w, inp, 4)
    q = torch.from_numpy(inp["q"]).cuda()
    c2.decode_rope(q, c2.rope_table(BASE), w.sm_scale)
    assert c2.device_errors() == 0
    t4 = c4.rope_table(BASE)
    assert t4.numel() == c2.rope_table(BASE).numel()
    c2.decode_rope(q, t4, w.sm_scale)
    assert c2.device_errors() & kvq.KVQ_DEVERR_BAD_TABLE
