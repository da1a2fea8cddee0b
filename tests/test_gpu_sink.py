"""GPU parity of the attention-sink window ("KV-cache quantization axes",
ihal.it, paragraph 9: high-precision windows for the recent tokens and the
attention sinks) against the oracle, through the C ABI: the first S tokens stay
fp16, the quantized groups start after them (bit-exact), appends fill the window
first, and decode attends over sinks + groups + tail within 2e-3 / 1e-3."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu

# (workload, bits, sink window); lengths leave whole groups after the window
CASES = {
    "gqa_2bit_s4": (S.LLAMA31_8B_128K.scaled(context=4164, n_tail=64), 2, 4),
    "gqa_4bit_s40": (S.LLAMA31_8B_128K.scaled(context=1064, n_tail=0, bits=4), 4, 40),
    "mha_d64_8bit_s32": (S.TINY.scaled(batch=2, context=288, n_tail=0, bits=8), 8, 32),
    "ragged_2bit_s4": (S.SERVING.scaled(batch=3, context=900, ragged=(36, 900), bits=2), 2, 4),
}


def _inp(name):
    w, bits, sink = CASES[name]
    inp = S.generate(w)
    if w.ragged is not None:  # tail = what is left after the window and whole groups
        inp["n_tail"] = ((inp["seq_len"] - np.minimum(sink, inp["seq_len"])) % 32).astype(np.int32)
    return w, bits, sink, inp


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_with_sinks_bit_exact_and_decode(name):
    w, bits, sink, inp = _inp(name)
    cache = H.device_cache(w, inp, bits, sink_cap=sink)
    torch.cuda.synchronize()
    states = H.oracle_states(inp, bits, sink_cap=sink)
    H.assert_buffers_equal(cache, states)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))
    assert cache.device_errors() == 0


def test_sequences_shorter_than_the_window():
    # every token a sink: exact fp16 attention
    w = S.LLAMA31_8B_128K.scaled(batch=2, context=64, n_tail=0)
    inp = S.generate(w)
    inp["seq_len"][:] = [20, 1]
    cache = H.device_cache(w, inp, 2, sink_cap=32)
    states = H.oracle_states(inp, 2, sink_cap=32)
    H.assert_buffers_equal(cache, states)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))


def test_append_fills_the_window_then_the_tail():
    # start with 2 tokens (window 5), append 130 one at a time: 3 more sinks, then
    # the tail grows, flushes to groups; bit-exact with the oracle after each check
    R, Sw = 32, 5
    w = S.LLAMA31_8B_128K.scaled(batch=2, context=140, n_tail=0)
    inp = S.generate(w)
    inp["seq_len"][:] = 2
    cache = H.device_cache(w, inp, 4, max_tokens=160, tail_cap=R, sink_cap=Sw)
    K = torch.from_numpy(inp["K"]).cuda()
    V = torch.from_numpy(inp["V"]).cuda()
    q = torch.from_numpy(inp["q"]).cuda()
    state = (2, 0, 0)
    for n in range(2, 132):
        cache.append(K[:, n].contiguous(), V[:, n].contiguous())
        state = O.append_lengths_sink(*state, Sw, R)
        if n % 13 == 0 or n == 131:
            torch.cuda.synchronize()
            ns, nq, nt = state
            st_inp = dict(inp, seq_len=np.full(2, n + 1, np.int32), n_tail=np.full(2, nt, np.int32))
            states = H.oracle_states(st_inp, 4, sink_cap=Sw)
            assert states[0]["n_quant"] == nq
            H.assert_buffers_equal(cache, states)
            out = cache.decode(q, w.sm_scale).cpu().numpy()
            H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))
    assert cache.device_errors() == 0
