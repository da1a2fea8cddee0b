"""Parity at the full workload sizes, in the launch configuration the benchmark
times (one stream-K decode launch over every CTA of the GPU): prefill of the
whole cache on the GPU, then a sample of (sequence, KV head) pairs compared
with the oracle -- every packed byte of those pairs bit-exact, and their query
heads' decode outputs within 2e-3 max-abs / 1e-3 mean-abs of the fp64 oracle."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

# workload, bits, sampled (sequence, KV head) pairs
CASES = {
    "llama2_13b_b8_t4096_2bit": (S.LLAMA2_13B, 2, ((0, 0), (3, 17), (7, 39))),
    "llama31_8b_t131072_2bit": (S.LLAMA31_8B_128K, 2, ((0, 0), (0, 5))),
    "llama31_8b_t131072_4bit": (S.LLAMA31_8B_128K_4BIT, 4, ((0, 3), (0, 7))),
    "serving_b16_ragged_4bit": (S.SERVING, 4, ((0, 1), (7, 4), (15, 6))),
}


@pytest.mark.parametrize("name", list(CASES))
def test_full_size_sampled(name):
    w, bits, pairs = CASES[name]
    inp = S.generate(w)
    cache = H.device_cache(w, inp, bits)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    assert cache.device_errors() == 0
    G = w.gqa
    for b, h in pairs:
        st = H.oracle_states(inp, bits, heads=[h], batches=[b])
        H.assert_buffers_equal(cache, st, batches=[b], heads=[h])
        ref = O.sequence_attention(inp["q"][b, h * G:(h + 1) * G], st[0], w.sm_scale)
        H.assert_close(out[b, h * G:(h + 1) * G], ref)
