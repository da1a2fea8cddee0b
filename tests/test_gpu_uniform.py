"""GPU parity of the uniform cache path against the oracle, through the C ABI:
prefill codes/scales/zeros bit-exact, decode attention within 2e-3 max-abs /
1e-3 mean-abs of the fp64 oracle, append + flush bit-exact."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu

# Small cases that span several tiles, ragged tails and every compiled variant.
CASES = {
    "tiny_d64_2bit": (S.TINY, 2),
    "mha_2bit": (S.LLAMA2_13B.scaled(batch=2, n_q_heads=4, n_kv_heads=4, context=352), 2),
    "gqa_2bit": (S.LLAMA31_8B_128K.scaled(context=4160), 2),
    "gqa_4bit": (S.LLAMA31_8B_128K.scaled(context=2112, bits=4), 4),
    "gqa_8bit": (S.LLAMA31_8B_128K.scaled(context=1056, n_tail=32, bits=8), 8),
    "ragged_4bit": (S.SERVING.scaled(batch=5, context=1100, ragged=(1, 1100)), 4),
    "d64_gqa2_4bit": (S.LLAMA31_8B_128K.scaled(head_dim=64, n_q_heads=16, context=640,
                                               n_tail=0), 4),
    "gqa8_2bit": (S.LLAMA31_8B_128K.scaled(n_q_heads=64, context=1088), 2),
    "d64_mha_8bit": (S.TINY.scaled(batch=3, context=200, n_tail=8, bits=8), 8),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.load_library()


def _run(name):
    w, bits = CASES[name]
    inp = S.generate(w)
    cache = H.device_cache(w, inp, bits)
    return w, bits, inp, cache


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_bit_exact(name):
    w, bits, inp, cache = _run(name)
    torch.cuda.synchronize()
    H.assert_buffers_equal(cache, H.oracle_states(inp, bits))


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    w, bits, inp, cache = _run(name)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    ref = H.oracle_decode(inp["q"], H.oracle_states(inp, bits), w.sm_scale)
    H.assert_close(out, ref)
    assert cache.device_errors() == 0


def test_decode_repeatable_and_workspace_reset():
    # the last-CTA merge resets its counters: a second call on the same workspace
    # gives the identical result (the merge order does not depend on timing)
    w, bits, inp, cache = _run("gqa_2bit")
    q = torch.from_numpy(inp["q"]).cuda()
    a = cache.decode(q, w.sm_scale).clone()
    b = cache.decode(q, w.sm_scale)
    assert torch.equal(a, b)
    ws = cache.workspace(w.n_q_heads)
    assert int(ws[:4 * w.batch * w.n_kv_heads].count_nonzero()) == 0


def test_same_sequence_in_different_batches_agrees():
    # the split of a sequence's groups across CTAs depends on the whole batch;
    # the result may not (beyond fp32 rounding)
    w = S.SERVING.scaled(batch=4, context=3000, ragged=(500, 3000))
    inp = S.generate(w)
    cache = H.device_cache(w, inp, 4)
    q = torch.from_numpy(inp["q"]).cuda()
    full = cache.decode(q, w.sm_scale).cpu().numpy()
    one = {k: (v[1:2] if isinstance(v, np.ndarray) and v.shape[:1] == (4,) else v)
           for k, v in inp.items()}
    w1 = w.scaled(batch=1)
    c1 = H.device_cache(w1, one, 4)
    single = c1.decode(q[1:2].contiguous(), w.sm_scale).cpu().numpy()
    np.testing.assert_allclose(full[1], single[0], atol=2e-5, rtol=0)


@pytest.mark.parametrize("seq,nt", [(0, 0), (5, 5), (32, 32), (32, 0), (64, 32), (33, 1)])
def test_edge_lengths(seq, nt):
    # empty sequence -> zeros; tail only; a single group; full tail
    w = S.LLAMA31_8B_128K.scaled(context=96, n_tail=nt)
    inp = S.generate(w)
    inp["seq_len"][:] = seq
    cache = H.device_cache(w, inp, 2)
    torch.cuda.synchronize()
    states = H.oracle_states(inp, 2)
    H.assert_buffers_equal(cache, states)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    if seq == 0:
        assert (out == 0).all()
    else:
        H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))


def test_strided_inputs():
    # K/V as a head-slice of a wider tensor: stride_h and stride_t are not the
    # contiguous ones
    w = S.LLAMA31_8B_128K.scaled(n_q_heads=16, n_kv_heads=4, context=320)
    inp = S.generate(w)
    big_k = torch.zeros(1, 320, 8, 128, dtype=torch.float16, device="cuda")
    big_v = torch.zeros_like(big_k)
    big_k[:, :, 2:6] = torch.from_numpy(inp["K"]).cuda()
    big_v[:, :, 2:6] = torch.from_numpy(inp["V"]).cuda()
    cache = H.device_cache(w, inp, 4, k=big_k[:, :, 2:6], v=big_v[:, :, 2:6])
    torch.cuda.synchronize()
    H.assert_buffers_equal(cache, H.oracle_states(inp, 4))


def test_inputs_only_8_byte_aligned():
    # rows that start on 8-byte but not 16-byte boundaries (a 4-element offset and a
    # head stride of 132 elements): the prefill stages them with 8-byte copies
    w = S.LLAMA31_8B_128K.scaled(n_q_heads=8, n_kv_heads=2, context=288, n_tail=32)
    inp = S.generate(w)
    flat_k = torch.zeros(288 * 2 * 132 + 8, dtype=torch.float16, device="cuda")
    flat_v = torch.zeros_like(flat_k)
    big_k = flat_k[4:4 + 288 * 2 * 132].view(1, 288, 2, 132)
    big_v = flat_v[4:4 + 288 * 2 * 132].view(1, 288, 2, 132)
    big_k[..., :128] = torch.from_numpy(inp["K"]).cuda()
    big_v[..., :128] = torch.from_numpy(inp["V"]).cuda()
    k, v = big_k[..., :128], big_v[..., :128]
    assert k.data_ptr() % 16 == 8 and k.stride(2) % 8 == 4
    cache = H.device_cache(w, inp, 2, k=k, v=v)
    torch.cuda.synchronize()
    H.assert_buffers_equal(cache, H.oracle_states(inp, 2))


@pytest.mark.parametrize("bits,R", [(2, 32), (4, 64)])
def test_append_flush_matches_oracle(bits, R):
    # prefill, then append tokens one at a time across several flushes; after
    # every step the cache equals the oracle's quantization of the token list,
    # and decode stays within tolerance
    w = S.LLAMA31_8B_128K.scaled(batch=3, context=400, tail_cap=R, n_tail=None,
                                 ragged=(40, 200))
    inp = S.generate(w)
    inp["n_tail"] = (inp["seq_len"] % 32).astype(np.int32)
    cache = H.device_cache(w, inp, bits, max_tokens=400, tail_cap=R)
    K = torch.from_numpy(inp["K"]).cuda()
    V = torch.from_numpy(inp["V"]).cuda()
    seq = inp["seq_len"].astype(int).copy()
    nq = (inp["seq_len"] - inp["n_tail"]).astype(int)
    ntl = inp["n_tail"].astype(int).copy()
    q = torch.from_numpy(inp["q"]).cuda()
    for step in range(100):
        idx = torch.tensor(seq, device="cuda")
        kn = K[torch.arange(3, device="cuda"), idx].contiguous()
        vn = V[torch.arange(3, device="cuda"), idx].contiguous()
        cache.append(kn, vn)
        for b in range(3):
            nq[b], ntl[b], _ = O.append_lengths(nq[b], ntl[b], R)
        seq += 1
        if step % 9 == 0 or step == 99:
            torch.cuda.synchronize()
            st_inp = dict(inp, seq_len=seq.astype(np.int32), n_tail=ntl.astype(np.int32))
            states = H.oracle_states(st_inp, bits)
            H.assert_buffers_equal(cache, states)
            out = cache.decode(q, w.sm_scale).cpu().numpy()
            H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))
    assert cache.device_errors() == 0


def test_append_flush_at_max_batch():
    # KVQ_MAX_BATCH sequences of ragged lengths, each appended 40 tokens: every
    # sequence crosses at least one flush (tail ring of 32)
    B = kvq.KVQ_MAX_BATCH
    w = S.SERVING.scaled(batch=B, n_kv_heads=1, n_q_heads=4, context=120, tail_cap=32,
                         ragged=(1, 60), bits=2)
    inp = S.generate(w)
    inp["n_tail"] = (inp["seq_len"] % 32).astype(np.int32)
    cache = H.device_cache(w, inp, 2, max_tokens=120, tail_cap=32)
    K = torch.from_numpy(inp["K"]).cuda()
    V = torch.from_numpy(inp["V"]).cuda()
    seq = inp["seq_len"].astype(int).copy()
    nq = (inp["seq_len"] - inp["n_tail"]).astype(int)
    ntl = inp["n_tail"].astype(int).copy()
    rows = torch.arange(B, device="cuda")
    for step in range(40):
        idx = torch.tensor(seq, device="cuda")
        cache.append(K[rows, idx].contiguous(), V[rows, idx].contiguous())
        for b in range(B):
            nq[b], ntl[b], _ = O.append_lengths(nq[b], ntl[b], 32)
        seq += 1
    torch.cuda.synchronize()
    assert cache.device_errors() == 0
    st_inp = dict(inp, seq_len=seq.astype(np.int32), n_tail=ntl.astype(np.int32))
    states = H.oracle_states(st_inp, 2)
    H.assert_buffers_equal(cache, states)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    H.assert_close(out, H.oracle_decode(inp["q"], states, w.sm_scale))


def test_append_past_capacity_sets_error_and_leaves_sequence():
    w = S.LLAMA31_8B_128K.scaled(batch=1, context=64, n_tail=32, tail_cap=32)
    inp = S.generate(w)
    cache = H.device_cache(w, inp, 2, max_tokens=32)  # one group: already full
    before = {k: v.clone() for k, v in cache.views().items()}
    kn = torch.ones(1, 8, 128, dtype=torch.float16, device="cuda")
    cache.append(kn, kn)  # tail full (32 == R) and no room to flush
    assert cache.device_errors() == kvq.KVQ_DEVERR_APPEND_CAPACITY
    after = cache.views()
    for k in before:
        assert torch.equal(before[k], after[k]), k


def test_decode_reports_bad_device_lengths():
    w = S.LLAMA31_8B_128K.scaled(context=128, n_tail=32)
    inp = S.generate(w)
    cache = H.device_cache(w, inp, 2)
    cache.n_tail.fill_(999)  # corrupt: beyond the tail capacity
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale)
    assert cache.device_errors() & kvq.KVQ_DEVERR_BAD_LENGTHS
    assert torch.isfinite(out).all()


def test_bounded_wait_gives_up_and_reports():
    # the mbarrier wait of every staging loop: with nothing arriving it must end
    # after its poll limit, set KVQ_DEVERR_TIMEOUT and leave the context usable
    import time
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    kvq.kvq_selftest_bounded_wait(flags, 1 << 20, arrive=True)
    torch.cuda.synchronize()
    assert int(flags[0]) == 0  # satisfied wait: no error
    t0 = time.perf_counter()
    kvq.kvq_selftest_bounded_wait(flags, 4096, arrive=False)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 5.0
    assert int(flags[0]) == kvq.KVQ_DEVERR_TIMEOUT
    # the context still works
    x = torch.arange(8, device="cuda", dtype=torch.float32)
    assert float(x.sum()) == 28.0


# Geometries with many (sequence, KV head) segments: on a 152-SM GPU the decode
# runs them as 1, 2 and 4 CTAs per SM (the launch picks the smallest grid with a
# CTA per segment); ragged lengths and fp16 tails put several segment pieces and
# chunk items in one CTA.  Every sequence is checked against the oracle.
SHAPES = {
    "seg_100_d128_2bit_gqa4": (S.SERVING.scaled(batch=25, n_kv_heads=4, n_q_heads=16, context=300,
                                                ragged=(1, 300), bits=2), 2),
    "seg_200_d128_2bit_mha": (S.LLAMA2_13B.scaled(batch=25, n_q_heads=8, n_kv_heads=8, context=200,
                                                  n_tail=8), 2),
    "seg_400_d64_4bit_gqa2": (S.SERVING.scaled(batch=50, n_kv_heads=8, n_q_heads=16, head_dim=64, context=260,
                                               ragged=(0, 260), bits=4), 4),
    "seg_320_d128_2bit_gqa8": (S.SERVING.scaled(batch=40, n_kv_heads=8, n_q_heads=64, context=160,
                                                ragged=(30, 160), bits=2), 2),
    # the largest batch one call takes (KVQ_MAX_BATCH sequences): the prefill's
    # per-sequence tables and the decode's shared-memory prefix sums at their limit
    "seg_512_d128_2bit_maxbatch": (S.SERVING.scaled(batch=kvq.KVQ_MAX_BATCH, n_kv_heads=1, n_q_heads=4,
                                                    context=70, ragged=(1, 70), bits=2), 2),
    "seg_1024_d64_4bit_maxbatch": (S.SERVING.scaled(batch=kvq.KVQ_MAX_BATCH, n_kv_heads=2, n_q_heads=4,
                                                    head_dim=64, context=40, ragged=(0, 40), bits=4), 4),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_many_segments_match_oracle(name):
    w, bits = SHAPES[name]
    inp = S.generate(w)
    if w.ragged is not None:
        inp["n_tail"] = (inp["seq_len"] % 32).astype(np.int32)
    cache = H.device_cache(w, inp, bits)
    states = H.oracle_states(inp, bits)
    H.assert_buffers_equal(cache, states)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    assert cache.device_errors() == 0
    ref = H.oracle_decode(inp["q"], states, w.sm_scale)
    H.assert_close(out, ref)
    # a second call gives identical bits (the merge counters were left at zero)
    out2 = cache.decode(q, w.sm_scale).cpu().numpy()
    assert (out2 == out).all()
