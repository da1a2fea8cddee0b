"""The C-ABI library loads, exports every entry point of include/*.h, and its
host-side validation rejects bad arguments before any CUDA call (CPU-only)."""
import ctypes
import os
import re

import pytest

from quantized_kv_cache_11_gb300 import build, kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return kvq.load_library()


def _declared():
    inc = os.path.join(ROOT, "include")
    src = "".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc))
                  if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert names == sorted(kvq.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert kvq.status_string(0) == "ok"
    assert kvq.status_string(-1) == "invalid argument"
    assert kvq.status_string(12345) == "unknown status"
    assert lib.kvq_version().decode().count(".") == 2


def test_cache_bytes_matches_layout(lib):
    d = kvq.kvq_cache(2, 8, 128, 2, 4096 // 32, 64)
    sizes = kvq.kvq_cache_bytes(d)
    groups = 2 * 8 * 128
    assert sizes[kvq.KVQ_BUF_K_CODES] == groups * 32 * 128 * 2 // 8
    assert sizes[kvq.KVQ_BUF_V_CODES] == sizes[kvq.KVQ_BUF_K_CODES]
    assert sizes[kvq.KVQ_BUF_K_META] == groups * 2 * 128 * 2
    assert sizes[kvq.KVQ_BUF_V_META] == groups * 2 * 128 * 2
    assert sizes[kvq.KVQ_BUF_K_TAIL] == 2 * 8 * 64 * 128 * 2
    assert sizes[kvq.KVQ_BUF_LENGTHS] == 2 * 4
    # Llama-3.1-8B 128k, 2-bit: codes + metadata per sequence = 100,663,296 bytes
    d = kvq.kvq_cache(1, 8, 128, 2, 131072 // 32, 64)
    s = kvq.kvq_cache_bytes(d)
    assert sum(s[:4]) == 8 * 4096 * (1024 + 1024 + 512 + 512)


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 96, kvq.KVQ_ERR_UNSUPPORTED), ("bits", 3, kvq.KVQ_ERR_UNSUPPORTED),
    ("tail_cap", 40, kvq.KVQ_ERR_INVALID), ("tail_cap", 0, kvq.KVQ_ERR_INVALID),
    ("batch", 0, kvq.KVQ_ERR_INVALID), ("max_groups", -1, kvq.KVQ_ERR_INVALID),
])
def test_cache_bytes_rejects_bad_geometry(lib, field, value, status):
    d = kvq.kvq_cache(1, 8, 128, 2, 16, 32)
    setattr(d, field, value)
    sizes = (ctypes.c_size_t * kvq.KVQ_NBUF)()
    assert lib.kvq_cache_bytes(ctypes.byref(d), sizes) == status


def _fake_cache(**kw):
    # Host-side validation only: pointers are never dereferenced when a check
    # fails, so aligned fake addresses are enough.
    d = kvq.kvq_cache(2, 4, 128, 2, 8, 32)
    for i, f in enumerate(("k_codes", "v_codes", "k_meta", "v_meta", "k_tail", "v_tail",
                           "n_quant", "n_tail", "tail_head")):
        setattr(d, f, 0x10000 * (i + 1))
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_prefill_validation_fails_before_launch(lib):
    i32 = ctypes.c_int32 * 2
    d = _fake_cache()
    call = lambda d, k=0x100000, sl=(64, 64), nt=(0, 0), st=(1 << 14, 512, 128): \
        lib.kvq_quantize_prefill(ctypes.byref(d), k, k + 0x1000, *st, i32(*sl), i32(*nt), None)
    assert call(_fake_cache(k_codes=None)) == kvq.KVQ_ERR_INVALID
    assert call(_fake_cache(k_meta=0x10008)) == kvq.KVQ_ERR_INVALID  # misaligned
    assert call(d, k=0) == kvq.KVQ_ERR_INVALID
    assert call(d, sl=(65, 64)) == kvq.KVQ_ERR_INVALID  # 65 - 0 not a multiple of 32
    assert call(d, sl=(64, 64), nt=(33, 0)) == kvq.KVQ_ERR_INVALID  # n_tail > R
    assert call(d, sl=(320, 64)) == kvq.KVQ_ERR_CAPACITY  # 10 groups > 8
    assert call(d, st=(1 << 14, 514, 128)) == kvq.KVQ_ERR_INVALID  # stride not multiple of 4
    assert call(d, k=0x100002) == kvq.KVQ_ERR_INVALID  # k not 8-byte aligned
    assert call(_fake_cache(head_dim=80)) == kvq.KVQ_ERR_UNSUPPORTED


def test_decode_and_append_validation_fails_before_launch(lib):
    d = _fake_cache()
    ws = ctypes.c_size_t()
    assert lib.kvq_decode_workspace_bytes(ctypes.byref(d), 6, ctypes.byref(ws)) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_decode_workspace_bytes(ctypes.byref(d), 12, ctypes.byref(ws)) == kvq.KVQ_ERR_UNSUPPORTED
    dec = lambda d, hq=16, q=0x200000, out=0x300000, scale=0.088, w=0x400000, wb=1 << 30: \
        lib.kvq_decode_attn(ctypes.byref(d), hq, q, out, scale, w, wb, None)
    assert dec(d, hq=6) == kvq.KVQ_ERR_INVALID
    assert dec(d, hq=48) == kvq.KVQ_ERR_UNSUPPORTED  # G = 12
    assert dec(d, q=0) == kvq.KVQ_ERR_INVALID
    assert dec(d, out=0x300004) == kvq.KVQ_ERR_INVALID  # out must be 16-byte aligned
    assert dec(d, w=0) == kvq.KVQ_ERR_INVALID
    assert dec(d, scale=0.0) == kvq.KVQ_ERR_INVALID
    assert dec(d, scale=float("nan")) == kvq.KVQ_ERR_INVALID
    assert dec(_fake_cache(n_tail=None)) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_append_token(ctypes.byref(d), 0, 0x1000, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_append_token(ctypes.byref(d), 0x1004, 0x1000, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_append_token(ctypes.byref(_fake_cache(bits=5)), 0x1000, 0x2000, None) == \
        kvq.KVQ_ERR_UNSUPPORTED


# ------------------------------------------------------------- mixed width
def test_trizone_bytes_matches_layout(lib):
    d = kvq.kvq_trizone(4, 8, 128, 65408, 128)
    s = kvq.kvq_trizone_bytes(d)
    assert s[kvq.KVQ_TZ_BUF_INDEX] == 32 * 512
    assert s[kvq.KVQ_TZ_BUF_TOKENS] == 32 * 65408 * 4
    # worst case per (sequence, KV head): ceil(65408/32) + 3 records of 13312 bytes
    # plus 4 fresh blocks of 16384, rounded up to 256
    region = -(-((2044 + 3) * 13312 + 4 * 16384) // 256) * 256
    assert s[kvq.KVQ_TZ_BUF_BLOCKS] == 32 * region


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, kvq.KVQ_ERR_UNSUPPORTED), ("batch", 0, kvq.KVQ_ERR_INVALID),
    ("max_old", -1, kvq.KVQ_ERR_INVALID), ("max_fresh", -5, kvq.KVQ_ERR_INVALID),
])
def test_trizone_bytes_rejects_bad_geometry(lib, field, value, status):
    d = kvq.kvq_trizone(1, 8, 128, 1024, 128)
    setattr(d, field, value)
    sizes = (ctypes.c_size_t * kvq.KVQ_TZ_NBUF)()
    assert lib.kvq_trizone_bytes(ctypes.byref(d), sizes) == status


def _fake_tz(**kw):
    d = kvq.kvq_trizone(2, 4, 128, 1024, 64)
    d.index, d.tokens, d.blocks = 0x10000, 0x20000, 0x100000
    for k, v in kw.items():
        setattr(d, k, v)
    return d


def test_trizone_validation_fails_before_launch(lib):
    i32 = ctypes.c_int32 * 2
    build = lambda d, k=0x1000000, to=(1000, 1000), nf=(64, 64), st=(1 << 14, 512, 128), vw=0x2000000: \
        lib.kvq_trizone_build(ctypes.byref(d), k, k + 0x1000, *st, vw, vw + 0x10000, i32(*to), i32(*nf),
                              None)
    assert build(_fake_tz(index=None)) == kvq.KVQ_ERR_INVALID
    assert build(_fake_tz(blocks=0x100008)) == kvq.KVQ_ERR_INVALID  # blocks 16-byte aligned
    assert build(_fake_tz(), k=0) == kvq.KVQ_ERR_INVALID
    assert build(_fake_tz(), vw=0) == kvq.KVQ_ERR_INVALID
    assert build(_fake_tz(), to=(1025, 0)) == kvq.KVQ_ERR_CAPACITY
    assert build(_fake_tz(), nf=(65, 0)) == kvq.KVQ_ERR_CAPACITY
    assert build(_fake_tz(), to=(-1, 0)) == kvq.KVQ_ERR_INVALID
    assert build(_fake_tz(), st=(1 << 14, 514, 128)) == kvq.KVQ_ERR_INVALID
    assert build(_fake_tz(head_dim=64)) == kvq.KVQ_ERR_UNSUPPORTED
    dec = lambda d, hq=16, q=0x200000, out=0x300000, scale=0.088, w=0x400000, wb=1 << 30: \
        lib.kvq_trizone_decode_attn(ctypes.byref(d), hq, q, out, scale, w, wb, None)
    assert dec(_fake_tz(), hq=6) == kvq.KVQ_ERR_INVALID
    assert dec(_fake_tz(), hq=48) == kvq.KVQ_ERR_UNSUPPORTED
    assert dec(_fake_tz(), out=0x300004) == kvq.KVQ_ERR_INVALID
    assert dec(_fake_tz(), scale=-1.0) == kvq.KVQ_ERR_INVALID
    assert dec(_fake_tz(batch=256, n_kv_heads=8)) == kvq.KVQ_ERR_UNSUPPORTED  # > 1024 segments
    ws = ctypes.c_size_t()
    assert lib.kvq_trizone_decode_workspace_bytes(ctypes.byref(_fake_tz()), 6, ctypes.byref(ws)) == \
        kvq.KVQ_ERR_INVALID


def test_sink_window_bytes_and_validation(lib):
    d = kvq.kvq_cache(2, 8, 128, 2, 16, 32)
    d.sink_cap = 4
    s = kvq.kvq_cache_bytes(d)
    assert s[kvq.KVQ_BUF_K_SINK] == s[kvq.KVQ_BUF_V_SINK] == 2 * 8 * 4 * 128 * 2
    sizes = (ctypes.c_size_t * kvq.KVQ_NBUF)()
    for bad in (-1, 257):
        d.sink_cap = bad
        assert lib.kvq_cache_bytes(ctypes.byref(d), sizes) == kvq.KVQ_ERR_INVALID
    # a window without its buffers is rejected before any launch
    f = _fake_cache(sink_cap=4)
    i32 = ctypes.c_int32 * 2
    st = lib.kvq_quantize_prefill(ctypes.byref(f), 0x100000, 0x101000, 1 << 14, 512, 128,
                                  i32(68, 68), i32(0, 0), None)
    assert st == kvq.KVQ_ERR_INVALID
    f = _fake_cache(sink_cap=4, k_sink=0x900000, v_sink=0x910000, n_sink=0x920000)
    # 68 tokens with a 4-token window: 64 quantized tokens = 2 groups; 67 is ragged
    st = lib.kvq_quantize_prefill(ctypes.byref(f), 0x100000, 0x101000, 1 << 14, 512, 128,
                                  i32(67, 68), i32(0, 0), None)
    assert st == kvq.KVQ_ERR_INVALID


def test_rdkv_workspace_bytes_matches_layout(lib):
    d = kvq.kvq_rdkv(4, 32, 8, 128, 65536)
    n = kvq.kvq_rdkv_workspace_bytes(d)
    lse = 4 * 32 * 65536 * 4                    # per query row, stride rounded up to 64
    wt = 4 * 8 * 65536 * 4
    wc = 4 * 8 * 128 * 4
    part = 4 * 8 * (65536 // 256) * 5 * 128 * 4  # 5 fields per 256-position chunk and channel
    assert n == lse + wt + wc + part
    assert kvq.kvq_rdkv_workspace_bytes(kvq.kvq_rdkv(1, 1, 1, 128, 1)) % 256 == 0


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, kvq.KVQ_ERR_UNSUPPORTED), ("n_q_heads", 24, kvq.KVQ_ERR_UNSUPPORTED),
    ("n_q_heads", 12, kvq.KVQ_ERR_INVALID), ("batch", 0, kvq.KVQ_ERR_INVALID),
    ("batch", kvq.KVQ_MAX_BATCH + 1, kvq.KVQ_ERR_UNSUPPORTED), ("max_tokens", -1, kvq.KVQ_ERR_INVALID),
    ("max_tokens", kvq.KVQ_RDKV_MAX_TOKENS + 1, kvq.KVQ_ERR_UNSUPPORTED),
])
def test_rdkv_rejects_bad_geometry(lib, field, value, status):
    d = kvq.kvq_rdkv(2, 8, 8, 128, 1024)
    setattr(d, field, value)
    out = ctypes.c_size_t()
    assert lib.kvq_rdkv_workspace_bytes(ctypes.byref(d), ctypes.byref(out)) == status


def test_rdkv_validation_fails_before_launch(lib):
    # every call below fails host-side validation, so no CUDA call is made
    d = kvq.kvq_rdkv(2, 8, 2, 128, 1024)
    ws_n = kvq.kvq_rdkv_workspace_bytes(d)
    i32 = ctypes.c_int32 * 2
    q, k, v, w, ws = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000
    qs, ks = (1024 * 8 * 128, 8 * 128, 128), (1024 * 2 * 128, 2 * 128, 128)

    def tw(**kw):
        a = dict(q=q, k=k, n=i32(100, 200), scale=0.088, w=w, ws=ws, wsn=ws_n, qs=qs)
        a.update(kw)
        return lib.kvq_rdkv_token_weights(ctypes.byref(d), a["q"], *a["qs"], a["k"], *ks, a["n"], a["scale"],
                                          a["w"], a["ws"], a["wsn"], None)
    assert tw(q=None) == kvq.KVQ_ERR_INVALID
    assert tw(q=q + 8) == kvq.KVQ_ERR_INVALID                      # not 16-byte aligned
    assert tw(qs=(1024 * 8 * 128, 8 * 128 + 4, 128)) == kvq.KVQ_ERR_INVALID  # stride not a multiple of 8
    assert tw(scale=0.0) == kvq.KVQ_ERR_INVALID
    assert tw(wsn=ws_n - 1) == kvq.KVQ_ERR_INVALID
    assert tw(ws=ws + 16) == kvq.KVQ_ERR_INVALID                   # workspace not 256-byte aligned
    assert tw(n=i32(100, 1025)) == kvq.KVQ_ERR_CAPACITY
    assert tw(n=i32(-1, 5)) == kvq.KVQ_ERR_INVALID

    def al(**kw):
        a = dict(n=i32(100, 200), to=i32(90, 150), vb=3.0, kb=4.0, max_old=512, Wt=None, wsn=ws_n)
        a.update(kw)
        return lib.kvq_rdkv_allocate(ctypes.byref(d), q, *qs, k, v, *ks, a["n"], a["to"], w, a["vb"], a["kb"],
                                     0x600000, a["max_old"], 0x700000, a["Wt"], None, ws, a["wsn"], None)
    assert al(to=i32(101, 150)) == kvq.KVQ_ERR_INVALID             # t_old > n_tokens
    assert al(max_old=120) == kvq.KVQ_ERR_CAPACITY                 # t_old > max_old
    assert al(vb=-1.0) == kvq.KVQ_ERR_INVALID
    assert al(kb=float("inf")) == kvq.KVQ_ERR_INVALID
    assert al(Wt=0x800002) == kvq.KVQ_ERR_INVALID                  # W_t misaligned
    assert al(wsn=100) == kvq.KVQ_ERR_INVALID


def test_rope_table_bytes_and_validation(lib):
    d = kvq.kvq_cache(1, 8, 128, 2, 131072 // 32, 64)
    out = ctypes.c_size_t()
    assert lib.kvq_rope_table_bytes(ctypes.byref(d), ctypes.byref(out)) == kvq.KVQ_OK
    # 64 fp32 offset rows + position blocks, then the fp16 piece part: 56 offset
    # rows of 8 k-tiles x 4 lane columns x 2 pieces x 16 bytes, + 16 bytes of padding
    pieces = 56 * (8 * 4 * 2 * 16 + 16)
    assert out.value == (64 + (131072 + 64) // 32) * 64 * 8 + pieces
    d.sink_cap = 5
    assert lib.kvq_rope_table_bytes(ctypes.byref(d), ctypes.byref(out)) == kvq.KVQ_OK
    assert out.value == (64 + -(-(5 + 131072 + 64) // 32)) * 64 * 8 + pieces
    d64 = kvq.kvq_cache(1, 8, 64, 2, 128, 64)
    assert lib.kvq_rope_table_bytes(ctypes.byref(d64), ctypes.byref(out)) == kvq.KVQ_ERR_UNSUPPORTED
    assert lib.kvq_rope_table(ctypes.byref(d), ctypes.c_float(1.0), 0x100000, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_rope_table(ctypes.byref(d), ctypes.c_float(10000.0), 0x100008, None) == kvq.KVQ_ERR_INVALID


def test_rope_decode_validation_fails_before_launch(lib):
    d = _fake_cache()
    need = ctypes.c_size_t()
    assert lib.kvq_rope_table_bytes(ctypes.byref(d), ctypes.byref(need)) == kvq.KVQ_OK
    dec = lambda tb, table=0x600000, hq=16: lib.kvq_decode_attn_rope(
        ctypes.byref(d), hq, 0x200000, 0x300000, ctypes.c_float(0.088), table, tb, 0x400000, 1 << 30, None)
    assert dec(need.value - 16) == kvq.KVQ_ERR_INVALID   # the table is too small for this cache
    assert dec(0) == kvq.KVQ_ERR_INVALID
    assert dec(need.value, table=0) == kvq.KVQ_ERR_INVALID
    assert dec(need.value, table=0x600008) == kvq.KVQ_ERR_INVALID  # 16-byte aligned
    assert dec(need.value, hq=6) == kvq.KVQ_ERR_INVALID


def test_selftest_validation_fails_before_launch(lib):
    assert lib.kvq_selftest_bounded_wait(None, 16, 0, None) == kvq.KVQ_ERR_INVALID
    assert lib.kvq_selftest_bounded_wait(0x1002, 16, 0, None) == kvq.KVQ_ERR_INVALID  # misaligned
    assert lib.kvq_selftest_bounded_wait(0x1000, 0, 0, None) == kvq.KVQ_ERR_INVALID   # no polls
