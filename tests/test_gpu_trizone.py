"""GPU parity of the mixed-width ("TriZone") cache against the oracle, through
the C ABI: index records, stored token order and every block record bit-exact
with the oracle's packer; decode attention within 2e-3 max-abs / 1e-3 mean-abs
of the fp64 oracle, which attends over the tokens in their ORIGINAL order."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu

W = S.TRIZONE
CASES = {
    # default width mix, several segments, partial blocks in every class
    "mix": W.scaled(batch=2, n_kv_heads=2, n_q_heads=8, context=4168, trizone_fresh=72),
    # all values fp16 (zone B only) / all tokens evicted (fresh only)
    "all_fp16": W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=700, trizone_fresh=40,
                         v_width_probs=(0, 0, 0, 0, 1.0)),
    "all_evicted": W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=300, trizone_fresh=33,
                            v_width_probs=(1.0, 0, 0, 0, 0)),
    # one key class only (k-tiles (8,0,0) and (0,0,8))
    "keys_2bit": W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=1100, trizone_fresh=12,
                          k_width_probs=(1.0, 0, 0)),
    "keys_8bit": W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=1100, trizone_fresh=12,
                          k_width_probs=(0, 0, 1.0)),
    # GQA 8 (two n-tiles), MHA, no fresh tokens
    "gqa8": W.scaled(batch=1, n_kv_heads=2, n_q_heads=16, context=2100, trizone_fresh=5),
    "mha": W.scaled(batch=3, n_kv_heads=4, n_q_heads=4, context=908, trizone_fresh=8),
    # value widths 4 and 8 dominate (their tiles and constant rows)
    "wide_values": W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=1600, trizone_fresh=32,
                            v_width_probs=(0.1, 0.0, 0.45, 0.45, 0.0)),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    kvq.load_library()


def _lengths(w, inp, t_old=None, n_fresh=None):
    B = w.batch
    t_old = np.full(B, w.context - w.trizone_fresh) if t_old is None else np.asarray(t_old)
    n_fresh = np.full(B, w.trizone_fresh) if n_fresh is None else np.asarray(n_fresh)
    return t_old.astype(int), n_fresh.astype(int)


def device_tz(w, inp, t_old, n_fresh, max_old=None, max_fresh=None):
    B, H = w.batch, w.n_kv_heads
    max_old = int(max_old if max_old is not None else inp["v_width"].shape[2])
    max_fresh = int(max_fresh if max_fresh is not None else max(1, n_fresh.max()))
    cache = kvq.TriZoneCache(B, H, max_old, max_fresh)
    vw = np.zeros((B, H, max_old), np.uint8)
    vw[:, :, :inp["v_width"].shape[2]] = inp["v_width"]
    cache.build(torch.from_numpy(inp["K"]).cuda(), torch.from_numpy(inp["V"]).cuda(),
                torch.from_numpy(vw).cuda(), torch.from_numpy(inp["k_width"]).cuda(),
                t_old.tolist(), n_fresh.tolist())
    return cache


def oracle_tz(inp, b, h, t_old, n_fresh):
    k = inp["K"][b, :t_old + n_fresh, h]
    v = inp["V"][b, :t_old + n_fresh, h]
    return O.trizone_quantize(k, v, inp["v_width"][b, h, :t_old], inp["k_width"][b, h])


def assert_segment_equal(views, b, h, pk):
    idx = views["index"][b, h].cpu().numpy()
    if not (idx == pk["index"]).all():
        got = idx[:128].view(np.int32)
        raise AssertionError(f"index of ({b},{h}) differs:\n got {got.tolist()}\n exp "
                             f"{pk['header'].tolist()}")
    n = len(pk["tokens"])
    toks = views["tokens"][b, h, :n].cpu().numpy()
    assert (toks == pk["tokens"]).all(), f"stored token order of ({b},{h}) differs"
    data = views["blocks"][b, h, :len(pk["data"])].cpu().numpy()
    bad = np.nonzero(data != pk["data"])[0]
    if bad.size:
        hdr = pk["header"]
        off = int(bad[0])
        kind = max(i for i in range(5) if hdr[21 + i] <= off)
        blk, within = divmod(off - int(hdr[21 + kind]), int(hdr[16 + kind]))
        raise AssertionError(f"({b},{h}): {bad.size} block bytes differ; first at {off}: kind {kind}, "
                             f"block {blk}, byte {within} of {hdr[16 + kind]} (k-tiles "
                             f"{hdr[13:16].tolist()})")


# cases built with n_fresh = 0 (the drawn fresh tokens are left out)
NO_FRESH = {"mha"}


def run_named(name):
    w = CASES[name]
    return w, *run_case(w, n_fresh=[0] * w.batch if name in NO_FRESH else None)


def run_case(w, t_old=None, n_fresh=None):
    inp = S.generate(w)
    t_old, n_fresh = _lengths(w, inp, t_old, n_fresh)
    cache = device_tz(w, inp, t_old, n_fresh)
    return inp, t_old, n_fresh, cache


@pytest.mark.parametrize("name", list(CASES))
def test_build_bit_exact(name):
    w, inp, t_old, n_fresh, cache = run_named(name)
    torch.cuda.synchronize()
    views = cache.views()
    for b in range(w.batch):
        for h in range(w.n_kv_heads):
            pk = O.trizone_pack(oracle_tz(inp, b, h, t_old[b], n_fresh[b]))
            assert_segment_equal(views, b, h, pk)
    assert cache.device_errors() == 0


def oracle_out(w, inp, t_old, n_fresh):
    out = []
    for b in range(w.batch):
        tzs = [oracle_tz(inp, b, h, t_old[b], n_fresh[b]) for h in range(w.n_kv_heads)]
        out.append(O.trizone_attention(inp["q"][b], tzs, w.sm_scale))
    return np.stack(out)


@pytest.mark.parametrize("name", list(CASES))
def test_decode_matches_oracle(name):
    w, inp, t_old, n_fresh, cache = run_named(name)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    H.assert_close(out, oracle_out(w, inp, t_old, n_fresh))
    assert cache.device_errors() == 0


def test_ragged_lengths_and_empty_sequences():
    # per-sequence old/fresh counts, including an empty sequence (zeros out) and
    # one with fresh tokens only
    w = W.scaled(batch=4, n_kv_heads=2, n_q_heads=8, context=1500, trizone_fresh=60)
    t_old, n_fresh = [1440, 0, 333, 0], [60, 17, 0, 0]
    inp, t_old, n_fresh, cache = run_case(w, t_old, n_fresh)
    torch.cuda.synchronize()
    views = cache.views()
    for b in range(4):
        for h in range(2):
            assert_segment_equal(views, b, h, O.trizone_pack(oracle_tz(inp, b, h, t_old[b], n_fresh[b])))
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    assert (out[3] == 0).all()
    H.assert_close(out, oracle_out(w, inp, t_old, n_fresh))


@pytest.mark.parametrize("case", ["aligned_ragged", "stream_k_many_segments", "max_segments"])
def test_decode_partitions(case):
    # the two partitions of the decode's CTAs: a few segments of unequal length
    # (each gets CTAs of its own, in proportion to its work) and more segments
    # than CTAs (a CTA's range crosses segment boundaries, merged by the split-K
    # counters); every segment against the oracle
    if case == "aligned_ragged":
        w = W.scaled(batch=6, n_kv_heads=2, n_q_heads=8, context=3000, trizone_fresh=20)
        t_old, n_fresh = [2980, 2500, 1200, 400, 2900, 60], [20, 3, 0, 20, 11, 1]
    elif case == "stream_k_many_segments":
        w = W.scaled(batch=40, n_kv_heads=8, n_q_heads=32, context=200, trizone_fresh=8)
        t_old, n_fresh = None, None
    else:  # KVQ_TZ_MAX_SEGMENTS (sequence, KV head) segments
        w = W.scaled(batch=kvq.KVQ_TZ_MAX_SEGMENTS // 8, n_kv_heads=8, n_q_heads=32, context=100,
                     trizone_fresh=4)
        t_old, n_fresh = None, None
    inp, t_old, n_fresh, cache = run_case(w, t_old, n_fresh)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    assert cache.device_errors() == 0
    H.assert_close(out, oracle_out(w, inp, t_old, n_fresh))
    assert torch.equal(torch.from_numpy(out), cache.decode(q, w.sm_scale).cpu())


def test_decode_repeatable_and_workspace_reset():
    # the blocks are dealt to warps the same way on every call: identical results
    w, inp, t_old, n_fresh, cache = run_named("mix")
    q = torch.from_numpy(inp["q"]).cuda()
    a = cache.decode(q, w.sm_scale).clone()
    b = cache.decode(q, w.sm_scale)
    assert torch.equal(a, b)
    ws = cache.workspace(w.n_q_heads)
    assert int(ws[:4 * w.batch * w.n_kv_heads].count_nonzero()) == 0


def test_strided_inputs():
    w = W.scaled(batch=1, n_kv_heads=2, n_q_heads=8, context=800, trizone_fresh=16)
    inp = S.generate(w)
    big_k = torch.zeros(1, 800, 5, 128, dtype=torch.float16, device="cuda")
    big_v = torch.zeros_like(big_k)
    big_k[:, :, 1:3] = torch.from_numpy(inp["K"]).cuda()
    big_v[:, :, 1:3] = torch.from_numpy(inp["V"]).cuda()
    cache = kvq.TriZoneCache(1, 2, 784, 16)
    cache.build(big_k[:, :, 1:3], big_v[:, :, 1:3], torch.from_numpy(inp["v_width"]).cuda(),
                torch.from_numpy(inp["k_width"]).cuda(), [784], [16])
    torch.cuda.synchronize()
    views = cache.views()
    for h in range(2):
        assert_segment_equal(views, 0, h, O.trizone_pack(oracle_tz(inp, 0, h, 784, 16)))


def test_bad_width_sets_error_and_drops_token():
    w = W.scaled(batch=1, n_kv_heads=1, n_q_heads=4, context=200, trizone_fresh=8)
    inp = S.generate(w)
    inp["v_width"][0, 0, 5] = 3  # not a width: the token is dropped
    t_old, n_fresh = _lengths(w, inp)
    cache = device_tz(w, inp, t_old, n_fresh)
    assert cache.device_errors() & kvq.KVQ_DEVERR_BAD_WIDTH
    ref = dict(inp)
    ref["v_width"] = inp["v_width"].copy()
    ref["v_width"][0, 0, 5] = 0
    pk = O.trizone_pack(oracle_tz(ref, 0, 0, t_old[0], n_fresh[0]))
    assert_segment_equal(cache.views(), 0, 0, pk)


# Full-size mixed-width workload (4 sequences x 8 KV heads x 65,408 old + 128 fresh
# tokens, the launch the benchmark times): a sample of segments bit-exact, and
# the output of those segments' query heads against the oracle.
@pytest.mark.slow
def test_full_size_sampled():
    w = W
    inp = S.generate(w)
    t_old, n_fresh = _lengths(w, inp)
    cache = device_tz(w, inp, t_old, n_fresh)
    q = torch.from_numpy(inp["q"]).cuda()
    out = cache.decode(q, w.sm_scale).cpu().numpy()
    views = cache.views()
    G = w.gqa
    for b, h in ((0, 0), (2, 5), (3, 7)):
        tz = oracle_tz(inp, b, h, t_old[b], n_fresh[b])
        assert_segment_equal(views, b, h, O.trizone_pack(tz))
        ref = O.trizone_attention(inp["q"][b, h * G:(h + 1) * G], [tz], w.sm_scale)
        H.assert_close(out[b, h * G:(h + 1) * G], ref)
    assert cache.device_errors() == 0
