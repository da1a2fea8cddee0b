"""Thin Python binding of libkvq.so (the C ABI declared in include/kvq.h,
include/kvq_trizone.h and include/kvq_rdkv.h).

Argument marshalling only: every step of the quantizer and of the decode runs
in the library's CUDA kernels.  Tensors are PyTorch CUDA tensors; PyTorch is
used for device memory and streams only.  There is no CPU fallback: if the
shared library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_ERR_INVALID = -1
KVQ_ERR_UNSUPPORTED = -2
KVQ_ERR_CAPACITY = -3
KVQ_ERR_CUDA = -4
KVQ_DEVERR_APPEND_CAPACITY = 1
KVQ_DEVERR_BAD_LENGTHS = 2
KVQ_DEVERR_TIMEOUT = 4
KVQ_DEVERR_BAD_TABLE = 16
KVQ_GROUP = 32
KVQ_MAX_BATCH = 512
KVQ_NBUF = 9
(KVQ_BUF_K_CODES, KVQ_BUF_V_CODES, KVQ_BUF_K_META, KVQ_BUF_V_META, KVQ_BUF_K_TAIL,
 KVQ_BUF_V_TAIL, KVQ_BUF_LENGTHS, KVQ_BUF_K_SINK, KVQ_BUF_V_SINK) = range(9)

KVQ_DEVERR_BAD_WIDTH = 8
KVQ_TZ_INDEX_BYTES = 512
KVQ_TZ_MAX_BLOCK_BYTES = 13312
KVQ_TZ_FRESH_BLOCK_BYTES = 16384
KVQ_TZ_MAX_SEGMENTS = 1024
KVQ_TZ_NBUF = 3
KVQ_TZ_BUF_INDEX, KVQ_TZ_BUF_TOKENS, KVQ_TZ_BUF_BLOCKS = range(3)
KVQ_RDKV_MAX_TOKENS = 1 << 20

# Every entry point of include/*.h.
EXPORTS = ("kvq_cache_bytes", "kvq_quantize_prefill", "kvq_append_token",
           "kvq_decode_workspace_bytes", "kvq_decode_attn", "kvq_decode_attn_static",
           "kvq_status_string", "kvq_version", "kvq_trizone_bytes", "kvq_trizone_build",
           "kvq_trizone_decode_workspace_bytes", "kvq_trizone_decode_attn",
           "kvq_rdkv_workspace_bytes", "kvq_rdkv_token_weights", "kvq_rdkv_allocate",
           "kvq_rope_table_bytes", "kvq_rope_table", "kvq_decode_attn_rope", "kvq_selftest_bounded_wait")
KVQ_STATIC_SCRATCH_BYTES = 4 << 20


class kvq_cache(ctypes.Structure):
    """Mirror of ``struct kvq_cache``."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("bits", ctypes.c_int32),
        ("max_groups", ctypes.c_int32),
        ("tail_cap", ctypes.c_int32),
        ("k_codes", ctypes.c_void_p),
        ("v_codes", ctypes.c_void_p),
        ("k_meta", ctypes.c_void_p),
        ("v_meta", ctypes.c_void_p),
        ("k_tail", ctypes.c_void_p),
        ("v_tail", ctypes.c_void_p),
        ("n_quant", ctypes.c_void_p),
        ("n_tail", ctypes.c_void_p),
        ("tail_head", ctypes.c_void_p),
        ("error_flags", ctypes.c_void_p),
        ("sink_cap", ctypes.c_int32),
        ("k_sink", ctypes.c_void_p),
        ("v_sink", ctypes.c_void_p),
        ("n_sink", ctypes.c_void_p),
    ]


class kvq_trizone(ctypes.Structure):
    """Mirror of ``struct kvq_trizone``."""

    _fields_ = [
        ("batch", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("max_old", ctypes.c_int32),
        ("max_fresh", ctypes.c_int32),
        ("index", ctypes.c_void_p),
        ("tokens", ctypes.c_void_p),
        ("blocks", ctypes.c_void_p),
        ("error_flags", ctypes.c_void_p),
    ]


class kvq_rdkv(ctypes.Structure):
    """Mirror of ``struct kvq_rdkv``."""

    _fields_ = [("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32)]


class KVQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")
        self.status = status


_lib = None


def load_library() -> ctypes.CDLL:
    """Load libkvq.so (built in-tree).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m quantized_kv_cache_11_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    c_int, c_i64, c_f, c_vp, c_sz = (ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                     ctypes.c_void_p, ctypes.c_size_t)
    cache_p = P(kvq_cache)
    lib.kvq_cache_bytes.argtypes = [cache_p, P(c_sz)]
    lib.kvq_quantize_prefill.argtypes = [cache_p, c_vp, c_vp, c_i64, c_i64, c_i64,
                                         P(ctypes.c_int32), P(ctypes.c_int32), c_vp]
    lib.kvq_append_token.argtypes = [cache_p, c_vp, c_vp, c_vp]
    lib.kvq_decode_workspace_bytes.argtypes = [cache_p, ctypes.c_int32, P(c_sz)]
    lib.kvq_decode_attn.argtypes = [cache_p, ctypes.c_int32, c_vp, c_vp, c_f, c_vp, c_sz, c_vp]
    lib.kvq_decode_attn_static.argtypes = [cache_p, ctypes.c_int32, c_vp, c_vp, c_f, c_vp]
    lib.kvq_rope_table_bytes.argtypes = [cache_p, P(c_sz)]
    lib.kvq_rope_table.argtypes = [cache_p, c_f, c_vp, c_vp]
    lib.kvq_decode_attn_rope.argtypes = [cache_p, ctypes.c_int32, c_vp, c_vp, c_f, c_vp, c_sz, c_vp, c_sz, c_vp]
    lib.kvq_selftest_bounded_wait.argtypes = [c_vp, ctypes.c_uint32, ctypes.c_int32, c_vp]
    tz_p = P(kvq_trizone)
    lib.kvq_trizone_bytes.argtypes = [tz_p, P(c_sz)]
    lib.kvq_trizone_build.argtypes = [tz_p, c_vp, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp,
                                      P(ctypes.c_int32), P(ctypes.c_int32), c_vp]
    lib.kvq_trizone_decode_workspace_bytes.argtypes = [tz_p, ctypes.c_int32, P(c_sz)]
    lib.kvq_trizone_decode_attn.argtypes = [tz_p, ctypes.c_int32, c_vp, c_vp, c_f, c_vp, c_sz,
                                            c_vp]
    rd_p = P(kvq_rdkv)
    i32p = P(ctypes.c_int32)
    lib.kvq_rdkv_workspace_bytes.argtypes = [rd_p, P(c_sz)]
    lib.kvq_rdkv_token_weights.argtypes = [rd_p, c_vp, c_i64, c_i64, c_i64, c_vp, c_i64, c_i64, c_i64,
                                           i32p, c_f, c_vp, c_vp, c_sz, c_vp]
    lib.kvq_rdkv_allocate.argtypes = [rd_p, c_vp, c_i64, c_i64, c_i64, c_vp, c_vp, c_i64, c_i64, c_i64,
                                      i32p, i32p, c_vp, c_f, c_f, c_vp, ctypes.c_int32, c_vp, c_vp, c_vp,
                                      c_vp, c_sz, c_vp]
    lib.kvq_status_string.argtypes = [c_int]
    lib.kvq_status_string.restype = ctypes.c_char_p
    lib.kvq_version.argtypes = []
    lib.kvq_version.restype = ctypes.c_char_p
    for name in ("kvq_cache_bytes", "kvq_quantize_prefill", "kvq_append_token",
                 "kvq_decode_workspace_bytes", "kvq_decode_attn", "kvq_decode_attn_static",
                 "kvq_trizone_bytes", "kvq_trizone_build", "kvq_trizone_decode_workspace_bytes",
                 "kvq_trizone_decode_attn", "kvq_rdkv_workspace_bytes", "kvq_rdkv_token_weights",
                 "kvq_rdkv_allocate", "kvq_rope_table_bytes", "kvq_rope_table", "kvq_decode_attn_rope",
                 "kvq_selftest_bounded_wait"):
        getattr(lib, name).restype = c_int
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load_library().kvq_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != KVQ_OK:
        raise KVQError(fn, status)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def kvq_cache_bytes(desc: kvq_cache) -> list:
    sizes = (ctypes.c_size_t * KVQ_NBUF)()
    _check("kvq_cache_bytes", load_library().kvq_cache_bytes(ctypes.byref(desc), sizes))
    return list(sizes)


def _need(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _check_prefill_args(cache, k_shape, seq_len, n_tail) -> None:
    """k must cover every sequence's tokens with the cache's heads and head_dim:
    the library reads k[b, t] for b < B and t < seq_len[b]."""
    if len(k_shape) != 4 or k_shape[0] < cache.batch or k_shape[2] != cache.n_kv_heads or \
            k_shape[3] != cache.head_dim:
        raise ValueError(f"k and v must be [B >= {cache.batch}, T, {cache.n_kv_heads}, {cache.head_dim}]")
    if len(seq_len) != cache.batch or len(n_tail) != cache.batch:
        raise ValueError("seq_len and n_tail need one entry per sequence")
    if any(int(n) > k_shape[1] for n in seq_len):
        raise ValueError("a sequence is longer than the token axis of k and v")


def _check_decode_args(cache, q_shape, out_shape) -> None:
    """q and out are [B, Hq, D] for the cache's batch and head_dim."""
    if len(q_shape) != 3 or q_shape[0] != cache.batch or q_shape[2] != cache.head_dim:
        raise ValueError(f"q must be [{cache.batch}, Hq, {cache.head_dim}]")
    if tuple(out_shape) != tuple(q_shape):
        raise ValueError("out must have the shape of q")


def kvq_quantize_prefill(cache: "QuantizedKVCache", k: torch.Tensor, v: torch.Tensor,
                         seq_len: Sequence[int], n_tail: Sequence[int], stream=None) -> None:
    """k, v: fp16 CUDA tensors [B, T, Hkv, D] (same strides, D contiguous)."""
    _need(k, torch.float16, "k")
    _need(v, torch.float16, "v")
    if k.shape != v.shape or k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need equal shapes and strides with a contiguous last dim")
    _check_prefill_args(cache, tuple(k.shape), seq_len, n_tail)
    B = cache.batch
    sl = (ctypes.c_int32 * B)(*[int(x) for x in seq_len])
    nt = (ctypes.c_int32 * B)(*[int(x) for x in n_tail])
    st = load_library().kvq_quantize_prefill(
        ctypes.byref(cache.desc), _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2),
        sl, nt, _stream(stream))
    _check("kvq_quantize_prefill", st)


def kvq_append_token(cache: "QuantizedKVCache", k_new: torch.Tensor, v_new: torch.Tensor,
                     stream=None) -> None:
    """k_new, v_new: fp16 CUDA tensors [B, Hkv, D], contiguous."""
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        _need(t, torch.float16, n)
        if not t.is_contiguous() or t.shape != (cache.batch, cache.n_kv_heads, cache.head_dim):
            raise ValueError(f"{n} must be a contiguous [B, Hkv, D] tensor")
    st = load_library().kvq_append_token(ctypes.byref(cache.desc), _ptr(k_new), _ptr(v_new),
                                         _stream(stream))
    _check("kvq_append_token", st)


def kvq_decode_workspace_bytes(cache: "QuantizedKVCache", n_q_heads: int) -> int:
    out = ctypes.c_size_t()
    _check("kvq_decode_workspace_bytes", load_library().kvq_decode_workspace_bytes(
        ctypes.byref(cache.desc), int(n_q_heads), ctypes.byref(out)))
    return out.value


def kvq_decode_attn(cache: "QuantizedKVCache", q: torch.Tensor, out: torch.Tensor,
                    sm_scale: float, workspace: torch.Tensor, stream=None) -> None:
    """q: fp16 [B, Hq, D] contiguous; out: fp32 [B, Hq, D] contiguous;
    workspace: uint8 CUDA tensor, zero-filled before first use."""
    _need(q, torch.float16, "q")
    _need(out, torch.float32, "out")
    _need(workspace, torch.uint8, "workspace")
    if not (q.is_contiguous() and out.is_contiguous()) or q.shape != out.shape:
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    _check_decode_args(cache, tuple(q.shape), tuple(out.shape))
    st = load_library().kvq_decode_attn(ctypes.byref(cache.desc), q.shape[1], _ptr(q), _ptr(out),
                                        float(sm_scale), _ptr(workspace), workspace.numel(),
                                        _stream(stream))
    _check("kvq_decode_attn", st)


def kvq_decode_attn_static(cache: "QuantizedKVCache", q: torch.Tensor, out: torch.Tensor,
                           sm_scale: float, stream=None) -> None:
    """kvq_decode_attn without a workspace: the library's fixed device array holds
    the scratch (see include/kvq.h).  Calls on one device must not overlap."""
    _need(q, torch.float16, "q")
    _need(out, torch.float32, "out")
    if not (q.is_contiguous() and out.is_contiguous()) or q.shape != out.shape:
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    _check_decode_args(cache, tuple(q.shape), tuple(out.shape))
    st = load_library().kvq_decode_attn_static(ctypes.byref(cache.desc), q.shape[1], _ptr(q),
                                               _ptr(out), float(sm_scale), _stream(stream))
    _check("kvq_decode_attn_static", st)


def kvq_rope_table_bytes(cache: "QuantizedKVCache") -> int:
    out = ctypes.c_size_t()
    _check("kvq_rope_table_bytes", load_library().kvq_rope_table_bytes(ctypes.byref(cache.desc), ctypes.byref(out)))
    return out.value


def kvq_rope_table(cache: "QuantizedKVCache", base: float, table: torch.Tensor, stream=None) -> None:
    """table: float32 device tensor of kvq_rope_table_bytes bytes."""
    _need(table, torch.float32, "table")
    if table.numel() * 4 < kvq_rope_table_bytes(cache) or not table.is_contiguous():
        raise ValueError("table too small or not contiguous")
    _check("kvq_rope_table", load_library().kvq_rope_table(ctypes.byref(cache.desc), float(base), _ptr(table),
                                                           _stream(stream)))


def kvq_decode_attn_rope(cache: "QuantizedKVCache", q: torch.Tensor, out: torch.Tensor, sm_scale: float,
                         table: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """Decode over a cache of pre-RoPE keys: q fp16 [B, Hq, D] (rotated to its own
    position), out fp32 [B, Hq, D], table from kvq_rope_table."""
    _need(q, torch.float16, "q")
    _need(out, torch.float32, "out")
    _need(table, torch.float32, "table")
    _need(workspace, torch.uint8, "workspace")
    if not (q.is_contiguous() and out.is_contiguous()) or q.shape != out.shape:
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    _check_decode_args(cache, tuple(q.shape), tuple(out.shape))
    st = load_library().kvq_decode_attn_rope(ctypes.byref(cache.desc), q.shape[1], _ptr(q), _ptr(out),
                                             float(sm_scale), _ptr(table), table.numel() * 4, _ptr(workspace),
                                             workspace.numel(), _stream(stream))
    _check("kvq_decode_attn_rope", st)


def kvq_selftest_bounded_wait(error_flags: torch.Tensor, max_polls: int, arrive: bool, stream=None) -> None:
    """error_flags: int32 device tensor (one element used)."""
    _need(error_flags, torch.int32, "error_flags")
    _check("kvq_selftest_bounded_wait", load_library().kvq_selftest_bounded_wait(
        _ptr(error_flags), int(max_polls), int(bool(arrive)), _stream(stream)))


class QuantizedKVCache:
    """Owns the device buffers of a uniform cache (allocated with PyTorch)."""

    def __init__(self, batch: int, n_kv_heads: int, head_dim: int, bits: int, max_tokens: int,
                 tail_cap: int = 32, device="cuda", sink_cap: int = 0):
        self.batch, self.n_kv_heads, self.head_dim, self.bits = batch, n_kv_heads, head_dim, bits
        self.tail_cap, self.sink_cap = tail_cap, sink_cap
        self.max_groups = math.ceil(max_tokens / KVQ_GROUP)
        d = kvq_cache(batch, n_kv_heads, head_dim, bits, self.max_groups, tail_cap)
        d.sink_cap = sink_cap
        sizes = kvq_cache_bytes(d)
        dev = torch.device(device)

        def buf(n, dtype=torch.uint8):
            return torch.zeros(max(n, 16) // torch.empty((), dtype=dtype).element_size(),
                               dtype=dtype, device=dev)

        self.k_codes = buf(sizes[KVQ_BUF_K_CODES])
        self.v_codes = buf(sizes[KVQ_BUF_V_CODES])
        self.k_meta = buf(sizes[KVQ_BUF_K_META], torch.float16)
        self.v_meta = buf(sizes[KVQ_BUF_V_META], torch.float16)
        self.k_tail = buf(sizes[KVQ_BUF_K_TAIL], torch.float16)
        self.v_tail = buf(sizes[KVQ_BUF_V_TAIL], torch.float16)
        self.k_sink = buf(sizes[KVQ_BUF_K_SINK], torch.float16)
        self.v_sink = buf(sizes[KVQ_BUF_V_SINK], torch.float16)
        lens = torch.zeros(5, (batch + 3) // 4 * 4, dtype=torch.int32, device=dev)
        self._lens = lens
        self.n_quant, self.n_tail, self.tail_head = lens[0, :batch], lens[1, :batch], lens[2, :batch]
        self.error_flags = lens[3, :1]
        self.n_sink = lens[4, :batch]
        for f, t in (("k_codes", self.k_codes), ("v_codes", self.v_codes),
                     ("k_meta", self.k_meta), ("v_meta", self.v_meta),
                     ("k_tail", self.k_tail), ("v_tail", self.v_tail),
                     ("n_quant", self.n_quant), ("n_tail", self.n_tail),
                     ("tail_head", self.tail_head), ("error_flags", self.error_flags),
                     ("k_sink", self.k_sink), ("v_sink", self.v_sink), ("n_sink", self.n_sink)):
            setattr(d, f, t.data_ptr())
        self.desc = d
        self._workspaces = {}

    @property
    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in
                   (self.k_codes, self.v_codes, self.k_meta, self.v_meta, self.k_tail, self.v_tail))

    def views(self) -> dict:
        """The buffers shaped as in include/kvq.h (no copies)."""
        B, H, D, G, R = self.batch, self.n_kv_heads, self.head_dim, self.max_groups, self.tail_cap
        tb = KVQ_GROUP * D * self.bits // 8
        return {
            "k_codes": self.k_codes[:B * H * G * tb].view(B, H, G, tb),
            "v_codes": self.v_codes[:B * H * G * tb].view(B, H, G, tb),
            "k_meta": self.k_meta[:B * H * G * 2 * D].view(B, H, G, 2, D),
            "v_meta": self.v_meta[:B * H * G * 2 * D].view(B, H, G, 2, D // 32, 32),
            "k_tail": self.k_tail[:B * H * R * D].view(B, H, R, D),
            "v_tail": self.v_tail[:B * H * R * D].view(B, H, R, D),
            "k_sink": self.k_sink[:B * H * self.sink_cap * D].view(B, H, self.sink_cap, D),
            "v_sink": self.v_sink[:B * H * self.sink_cap * D].view(B, H, self.sink_cap, D),
            "n_quant": self.n_quant, "n_tail": self.n_tail, "tail_head": self.tail_head,
            "n_sink": self.n_sink,
        }

    def workspace(self, n_q_heads: int) -> torch.Tensor:
        ws = self._workspaces.get(n_q_heads)
        if ws is None:
            ws = torch.zeros(kvq_decode_workspace_bytes(self, n_q_heads), dtype=torch.uint8,
                             device=self.k_codes.device)
            self._workspaces[n_q_heads] = ws
        return ws

    def prefill(self, k, v, seq_len, n_tail, stream=None):
        kvq_quantize_prefill(self, k, v, seq_len, n_tail, stream)

    def append(self, k_new, v_new, stream=None):
        kvq_append_token(self, k_new, v_new, stream)

    def decode(self, q, sm_scale: Optional[float] = None, out=None, stream=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        kvq_decode_attn(self, q, out, sm_scale, self.workspace(q.shape[1]), stream)
        return out

    def rope_table(self, base: float, stream=None) -> torch.Tensor:
        """The cos/sin table of this geometry for pre-RoPE keys (kvq_rope_table)."""
        t = torch.empty(kvq_rope_table_bytes(self) // 4, dtype=torch.float32, device=self.k_codes.device)
        kvq_rope_table(self, base, t, stream)
        return t

    def decode_rope(self, q, table, sm_scale: Optional[float] = None, out=None, stream=None):
        """Decode over pre-RoPE keys rotated to their positions (kvq_decode_attn_rope)."""
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        kvq_decode_attn_rope(self, q, out, sm_scale, table, self.workspace(q.shape[1]), stream)
        return out

    def device_errors(self) -> int:
        """Read (with a sync) the device error bits."""
        return int(self.error_flags.item())


# --------------------------------------------------------------- mixed width
def kvq_trizone_bytes(desc: kvq_trizone) -> list:
    sizes = (ctypes.c_size_t * KVQ_TZ_NBUF)()
    _check("kvq_trizone_bytes", load_library().kvq_trizone_bytes(ctypes.byref(desc), sizes))
    return list(sizes)


def kvq_trizone_build(cache: "TriZoneCache", k: torch.Tensor, v: torch.Tensor,
                      v_width: torch.Tensor, k_width: torch.Tensor, t_old: Sequence[int],
                      n_fresh: Sequence[int], stream=None) -> None:
    """k, v: fp16 [B, T, Hkv, D] (same strides, D contiguous); v_width: uint8
    [B, Hkv, max_old] contiguous; k_width: uint8 [B, Hkv, D] contiguous."""
    _need(k, torch.float16, "k")
    _need(v, torch.float16, "v")
    _need(v_width, torch.uint8, "v_width")
    _need(k_width, torch.uint8, "k_width")
    if k.shape != v.shape or k.stride() != v.stride() or k.stride(3) != 1:
        raise ValueError("k and v need equal shapes and strides with a contiguous last dim")
    B, H = cache.batch, cache.n_kv_heads
    if v_width.shape != (B, H, cache.max_old) or not v_width.is_contiguous():
        raise ValueError("v_width must be a contiguous [B, Hkv, max_old] tensor")
    if k_width.shape != (B, H, cache.head_dim) or not k_width.is_contiguous():
        raise ValueError("k_width must be a contiguous [B, Hkv, D] tensor")
    if len(t_old) != B or len(n_fresh) != B:
        raise ValueError("t_old and n_fresh need one entry per sequence")
    if k.shape[0] != B or k.shape[2] != H or k.shape[3] != cache.head_dim or \
            any(int(a) + int(f) > k.shape[1] for a, f in zip(t_old, n_fresh)):
        raise ValueError("k/v must be [B, T, Hkv, D] with T >= t_old + n_fresh")
    to = (ctypes.c_int32 * B)(*[int(x) for x in t_old])
    nf = (ctypes.c_int32 * B)(*[int(x) for x in n_fresh])
    st = load_library().kvq_trizone_build(
        ctypes.byref(cache.desc), _ptr(k), _ptr(v), k.stride(0), k.stride(1), k.stride(2),
        _ptr(v_width), _ptr(k_width), to, nf, _stream(stream))
    _check("kvq_trizone_build", st)


def kvq_trizone_decode_workspace_bytes(cache: "TriZoneCache", n_q_heads: int) -> int:
    out = ctypes.c_size_t()
    _check("kvq_trizone_decode_workspace_bytes", load_library().kvq_trizone_decode_workspace_bytes(
        ctypes.byref(cache.desc), int(n_q_heads), ctypes.byref(out)))
    return out.value


def kvq_trizone_decode_attn(cache: "TriZoneCache", q: torch.Tensor, out: torch.Tensor,
                            sm_scale: float, workspace: torch.Tensor, stream=None) -> None:
    """q: fp16 [B, Hq, D] contiguous; out: fp32 [B, Hq, D] contiguous."""
    _need(q, torch.float16, "q")
    _need(out, torch.float32, "out")
    _need(workspace, torch.uint8, "workspace")
    if not (q.is_contiguous() and out.is_contiguous()) or q.shape != out.shape:
        raise ValueError("q and out must be contiguous [B, Hq, D] tensors")
    _check_decode_args(cache, tuple(q.shape), tuple(out.shape))
    st = load_library().kvq_trizone_decode_attn(ctypes.byref(cache.desc), q.shape[1], _ptr(q),
                                                _ptr(out), float(sm_scale), _ptr(workspace),
                                                workspace.numel(), _stream(stream))
    _check("kvq_trizone_decode_attn", st)


class TriZoneCache:
    """Owns the device buffers of a mixed-width cache (allocated with PyTorch)."""

    def __init__(self, batch: int, n_kv_heads: int, max_old: int, max_fresh: int,
                 head_dim: int = 128, device="cuda"):
        self.batch, self.n_kv_heads, self.head_dim = batch, n_kv_heads, head_dim
        self.max_old, self.max_fresh = max_old, max_fresh
        d = kvq_trizone(batch, n_kv_heads, head_dim, max_old, max_fresh)
        sizes = kvq_trizone_bytes(d)
        dev = torch.device(device)
        self.region = sizes[KVQ_TZ_BUF_BLOCKS] // (batch * n_kv_heads)
        self.index = torch.zeros(sizes[KVQ_TZ_BUF_INDEX], dtype=torch.uint8, device=dev)
        self.tokens = torch.zeros(max(sizes[KVQ_TZ_BUF_TOKENS] // 4, 4), dtype=torch.int32,
                                  device=dev)
        self.blocks = torch.zeros(sizes[KVQ_TZ_BUF_BLOCKS], dtype=torch.uint8, device=dev)
        self.error_flags = torch.zeros(4, dtype=torch.int32, device=dev)
        d.index, d.tokens, d.blocks = (self.index.data_ptr(), self.tokens.data_ptr(),
                                       self.blocks.data_ptr())
        d.error_flags = self.error_flags.data_ptr()
        self.desc = d
        self._workspaces = {}

    def views(self) -> dict:
        B, H = self.batch, self.n_kv_heads
        return {"index": self.index.view(B, H, KVQ_TZ_INDEX_BYTES),
                "tokens": self.tokens[:B * H * self.max_old].view(B, H, self.max_old),
                "blocks": self.blocks.view(B, H, self.region)}

    def workspace(self, n_q_heads: int) -> torch.Tensor:
        ws = self._workspaces.get(n_q_heads)
        if ws is None:
            ws = torch.zeros(kvq_trizone_decode_workspace_bytes(self, n_q_heads),
                             dtype=torch.uint8, device=self.index.device)
            self._workspaces[n_q_heads] = ws
        return ws

    def build(self, k, v, v_width, k_width, t_old, n_fresh, stream=None):
        kvq_trizone_build(self, k, v, v_width, k_width, t_old, n_fresh, stream)

    def decode(self, q, sm_scale: Optional[float] = None, out=None, stream=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.head_dim)
        kvq_trizone_decode_attn(self, q, out, sm_scale, self.workspace(q.shape[1]), stream)
        return out

    def device_errors(self) -> int:
        return int(self.error_flags[0].item())


def kvq_rdkv_workspace_bytes(desc: kvq_rdkv) -> int:
    out = ctypes.c_size_t()
    _check("kvq_rdkv_workspace_bytes", load_library().kvq_rdkv_workspace_bytes(ctypes.byref(desc),
                                                                                ctypes.byref(out)))
    return out.value


def _check_prompt(t: torch.Tensor, name: str, batch: int, heads: int, d: int):
    _need(t, torch.float16, name)
    if t.dim() != 4 or t.shape[0] < batch or t.shape[2] != heads or t.shape[3] != d or t.stride(3) != 1:
        raise ValueError(f"{name} must be [B >= {batch}, T, {heads}, {d}] with a contiguous last dim")


def kvq_rdkv_token_weights(desc: kvq_rdkv, q: torch.Tensor, k: torch.Tensor, n_tokens: Sequence[int],
                           sm_scale: float, w: torch.Tensor, workspace: torch.Tensor, stream=None) -> None:
    """q: fp16 [B, T, Hq, D]; k: fp16 [B, T, Hkv, D]; w: fp32 [B, Hkv, max_tokens] contiguous."""
    _check_prompt(q, "q", desc.batch, desc.n_q_heads, desc.head_dim)
    _check_prompt(k, "k", desc.batch, desc.n_kv_heads, desc.head_dim)
    _need(w, torch.float32, "w")
    _need(workspace, torch.uint8, "workspace")
    if w.shape != (desc.batch, desc.n_kv_heads, desc.max_tokens) or not w.is_contiguous():
        raise ValueError("w must be a contiguous [B, Hkv, max_tokens] tensor")
    if len(n_tokens) != desc.batch or any(int(n) > min(q.shape[1], k.shape[1]) for n in n_tokens):
        raise ValueError("n_tokens needs one entry per sequence, within the prompt tensors")
    nt = (ctypes.c_int32 * desc.batch)(*[int(x) for x in n_tokens])
    st = load_library().kvq_rdkv_token_weights(
        ctypes.byref(desc), _ptr(q), q.stride(0), q.stride(1), q.stride(2), _ptr(k), k.stride(0),
        k.stride(1), k.stride(2), nt, float(sm_scale), _ptr(w), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check("kvq_rdkv_token_weights", st)


def kvq_rdkv_allocate(desc: kvq_rdkv, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                      n_tokens: Sequence[int], t_old: Sequence[int], w: torch.Tensor, v_avg_bits: float,
                      k_avg_bits: float, v_width: torch.Tensor, k_width: torch.Tensor,
                      workspace: torch.Tensor, W_t: Optional[torch.Tensor] = None,
                      W_c: Optional[torch.Tensor] = None, stream=None) -> None:
    """v_width: uint8 [B, Hkv, max_old] contiguous; k_width: uint8 [B, Hkv, D] contiguous;
    W_t: fp32 [B, Hkv, max_old] or None; W_c: fp32 [B, Hkv, D] or None."""
    _check_prompt(q, "q", desc.batch, desc.n_q_heads, desc.head_dim)
    _check_prompt(k, "k", desc.batch, desc.n_kv_heads, desc.head_dim)
    _check_prompt(v, "v", desc.batch, desc.n_kv_heads, desc.head_dim)
    if k.stride() != v.stride() or k.shape != v.shape:
        raise ValueError("k and v need equal shapes and strides")
    _need(w, torch.float32, "w")
    _need(v_width, torch.uint8, "v_width")
    _need(k_width, torch.uint8, "k_width")
    _need(workspace, torch.uint8, "workspace")
    B, H, D = desc.batch, desc.n_kv_heads, desc.head_dim
    if v_width.dim() != 3 or v_width.shape[:2] != (B, H) or not v_width.is_contiguous():
        raise ValueError("v_width must be a contiguous [B, Hkv, max_old] tensor")
    max_old = v_width.shape[2]
    if k_width.shape != (B, H, D) or not k_width.is_contiguous():
        raise ValueError("k_width must be a contiguous [B, Hkv, D] tensor")
    if W_t is not None:
        _need(W_t, torch.float32, "W_t")
        if W_t.shape != (B, H, max_old) or not W_t.is_contiguous():
            raise ValueError("W_t must be a contiguous [B, Hkv, max_old] tensor")
    if W_c is not None:
        _need(W_c, torch.float32, "W_c")
        if W_c.shape != (B, H, D) or not W_c.is_contiguous():
            raise ValueError("W_c must be a contiguous [B, Hkv, D] tensor")
    if w.shape != (B, H, desc.max_tokens) or not w.is_contiguous():
        raise ValueError("w must be a contiguous [B, Hkv, max_tokens] tensor")
    if len(n_tokens) != B or len(t_old) != B or \
            any(int(n) > min(q.shape[1], k.shape[1]) for n in n_tokens):
        raise ValueError("n_tokens and t_old need one entry per sequence, within the prompt tensors")
    nt = (ctypes.c_int32 * B)(*[int(x) for x in n_tokens])
    to = (ctypes.c_int32 * B)(*[int(x) for x in t_old])
    st = load_library().kvq_rdkv_allocate(
        ctypes.byref(desc), _ptr(q), q.stride(0), q.stride(1), q.stride(2), _ptr(k), _ptr(v),
        k.stride(0), k.stride(1), k.stride(2), nt, to, _ptr(w), float(v_avg_bits), float(k_avg_bits),
        _ptr(v_width), max_old, _ptr(k_width), _ptr(W_t), _ptr(W_c), _ptr(workspace), workspace.numel(),
        _stream(stream))
    _check("kvq_rdkv_allocate", st)


class RDKVAllocator:
    """Workspace and outputs of the RDKV allocation for one geometry (PyTorch
    allocations); ``run`` issues the token weights, then the allocation."""

    def __init__(self, batch: int, n_q_heads: int, n_kv_heads: int, max_tokens: int, max_old: int,
                 head_dim: int = 128, device="cuda"):
        self.desc = kvq_rdkv(batch, n_q_heads, n_kv_heads, head_dim, max_tokens)
        dev = torch.device(device)
        self.workspace = torch.zeros(kvq_rdkv_workspace_bytes(self.desc), dtype=torch.uint8, device=dev)
        self.w = torch.zeros((batch, n_kv_heads, max_tokens), dtype=torch.float32, device=dev)
        self.v_width = torch.zeros((batch, n_kv_heads, max_old), dtype=torch.uint8, device=dev)
        self.k_width = torch.zeros((batch, n_kv_heads, head_dim), dtype=torch.uint8, device=dev)
        self.W_t = torch.zeros((batch, n_kv_heads, max_old), dtype=torch.float32, device=dev)
        self.W_c = torch.zeros((batch, n_kv_heads, head_dim), dtype=torch.float32, device=dev)

    def token_weights(self, q, k, n_tokens, sm_scale: Optional[float] = None, stream=None):
        if sm_scale is None:
            sm_scale = 1.0 / math.sqrt(self.desc.head_dim)
        kvq_rdkv_token_weights(self.desc, q, k, n_tokens, sm_scale, self.w, self.workspace, stream)
        return self.w

    def allocate(self, q, k, v, n_tokens, t_old, v_avg_bits: float, k_avg_bits: float, stream=None):
        kvq_rdkv_allocate(self.desc, q, k, v, n_tokens, t_old, self.w, v_avg_bits, k_avg_bits,
                          self.v_width, self.k_width, self.workspace, self.W_t, self.W_c, stream)
        return self.v_width, self.k_width

    def run(self, q, k, v, n_tokens, t_old, v_avg_bits: float, k_avg_bits: float,
            sm_scale: Optional[float] = None, stream=None):
        self.token_weights(q, k, n_tokens, sm_scale, stream)
        return self.allocate(q, k, v, n_tokens, t_old, v_avg_bits, k_avg_bits, stream)
