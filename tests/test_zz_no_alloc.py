"""kvq_decode_attn_static: decode attention for callers that cannot allocate
device memory (an engine whose own pool already holds all of it, a host
program that only reaches the GPU through the C ABI, a decode loop that must
not call cudaMalloc because it can synchronize the device).  Its scratch is a
fixed array inside the library instead of a caller workspace; its results
must match kvq_decode_attn's, call after call.

This file is collected last on purpose: it must pass both on its own in a
fresh process and after every other test has run.
"""
import ctypes

import pytest
import torch

from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu

CASES = {
    "gqa_2bit": (S.LLAMA31_8B_128K.scaled(context=4160), 2),
    "ragged_4bit": (S.SERVING.scaled(batch=5, context=1100, ragged=(1, 1100)), 4),
    "d64_mha_8bit": (S.TINY.scaled(batch=3, context=200, n_tail=8, bits=8), 8),
}


@pytest.mark.parametrize("name", list(CASES))
def test_static_scratch_matches_workspace_decode(name):
    w, bits = CASES[name]
    inp = S.generate(w)
    cache = H.device_cache(w, inp, bits)
    q = torch.from_numpy(inp["q"]).cuda()
    ref = cache.decode(q, w.sm_scale)  # caller-workspace path
    # the same kernel with the same partition: the bits must be identical, on the
    # first call (fresh array) and on the second (the array holds the first call's data)
    for _ in range(2):
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        kvq.kvq_decode_attn_static(cache, q, out, w.sm_scale)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), "static-scratch decode differs from the workspace decode"
    assert cache.device_errors() == 0
    # and both against the fp64 oracle at the decode tolerance
    states = H.oracle_states(inp, bits)
    H.assert_close(out.cpu().numpy(), H.oracle_decode(inp["q"], states, w.sm_scale))


def test_static_scratch_rejects_geometry_beyond_its_size():
    # 512 sequences x 64 KV heads x 8 query heads per KV head would need far more
    # than KVQ_STATIC_SCRATCH_BYTES of partials; the call must refuse up front,
    # before it touches any buffer (the addresses below are never dereferenced).
    d = kvq.kvq_cache(512, 64, 128, 2, 1, 32)
    for i, f in enumerate(("k_codes", "v_codes", "k_meta", "v_meta", "k_tail", "v_tail",
                           "n_quant", "n_tail", "tail_head")):
        setattr(d, f, 0x10000 * (i + 1))
    lib = kvq.load_library()
    st = lib.kvq_decode_attn_static(ctypes.byref(d), 512, 0x200000, 0x300000, 0.088, None)
    assert st == kvq.KVQ_ERR_CAPACITY
