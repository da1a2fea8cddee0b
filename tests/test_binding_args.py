"""Host-side argument checks of the Python binding (no GPU): shapes that would
make the library read or write past a caller's tensors are refused before any
call reaches the C ABI."""
from types import SimpleNamespace

import pytest

from quantized_kv_cache_11_gb300 import kvq

CACHE = SimpleNamespace(batch=2, n_kv_heads=8, head_dim=128)


def test_prefill_args_accept_the_cache_geometry():
    kvq._check_prefill_args(CACHE, (2, 4096, 8, 128), [4096, 100], [32, 4])
    kvq._check_prefill_args(CACHE, (3, 4096, 8, 128), [10, 20], [0, 0])   # extra rows are not read


@pytest.mark.parametrize("shape,seq,tail", [
    ((1, 4096, 8, 128), [1, 1], [0, 0]),      # fewer sequences than the cache
    ((2, 4096, 4, 128), [1, 1], [0, 0]),      # wrong KV heads
    ((2, 4096, 8, 64), [1, 1], [0, 0]),       # wrong head_dim
    ((2, 4096, 8), [1, 1], [0, 0]),           # not 4-d
    ((2, 4096, 8, 128), [1], [0]),            # one length short
    ((2, 4096, 8, 128), [1, 1], [0]),
    ((2, 4096, 8, 128), [4097, 1], [0, 0]),   # longer than the token axis
])
def test_prefill_args_refuse_out_of_bounds(shape, seq, tail):
    with pytest.raises(ValueError):
        kvq._check_prefill_args(CACHE, shape, seq, tail)


def test_decode_args():
    kvq._check_decode_args(CACHE, (2, 32, 128), (2, 32, 128))
    for q, o in (((1, 32, 128), (1, 32, 128)), ((2, 32, 64), (2, 32, 64)), ((2, 32, 128), (2, 16, 128)),
                 ((2, 4096), (2, 4096))):
        with pytest.raises(ValueError):
            kvq._check_decode_args(CACHE, q, o)
