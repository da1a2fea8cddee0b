"""Guard bands around every buffer the library writes (a stand-in for a memory
checker): each buffer is allocated with 4 KB of seeded random bytes before and
after it, the entry point runs on small ragged cases (empty sequences, partial
groups, flushes, partial blocks), and the bands must come back byte for byte
unchanged.  A write past a cache tile, a metadata block, the tail ring, the
sink rows, a workspace, an output, a mixed-width record or an allocation output
shows up here even when the values the parity tests read are right."""
import numpy as np
import pytest
import torch

from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

PAD = 4096


class Guarded:
    """A device buffer of `nbytes` bytes (viewed as `dtype`) between two bands of
    PAD seeded random bytes."""

    _seed = 0

    def __init__(self, nbytes: int, dtype=torch.uint8, fill: float = 0):
        Guarded._seed += 1
        g = torch.Generator().manual_seed(1000 + Guarded._seed)
        self.n = int(nbytes)
        self.bands = torch.randint(0, 256, (2, PAD), generator=g, dtype=torch.uint8)
        self.raw = torch.empty(2 * PAD + self.n, dtype=torch.uint8, device="cuda")
        self.raw[:PAD] = self.bands[0].cuda()
        self.raw[PAD + self.n:] = self.bands[1].cuda()
        self.t = self.raw[PAD:PAD + self.n].view(dtype)
        self.t.fill_(fill)

    def intact(self) -> bool:
        torch.cuda.synchronize()
        return torch.equal(self.raw[:PAD].cpu(), self.bands[0]) and \
            torch.equal(self.raw[PAD + self.n:].cpu(), self.bands[1])


def _assert_intact(guards: dict, what: str):
    broken = [name for name, g in guards.items() if not g.intact()]
    assert not broken, f"{what}: guard bands overwritten around {broken}"


def guard_cache(cache: kvq.QuantizedKVCache) -> dict:
    """Move every buffer of a uniform cache into a guarded allocation of exactly
    the size kvq_cache_bytes states (the lengths arrays too)."""
    sizes = kvq.kvq_cache_bytes(cache.desc)
    B = cache.batch
    spec = {"k_codes": (kvq.KVQ_BUF_K_CODES, torch.uint8), "v_codes": (kvq.KVQ_BUF_V_CODES, torch.uint8),
            "k_meta": (kvq.KVQ_BUF_K_META, torch.float16), "v_meta": (kvq.KVQ_BUF_V_META, torch.float16),
            "k_tail": (kvq.KVQ_BUF_K_TAIL, torch.float16), "v_tail": (kvq.KVQ_BUF_V_TAIL, torch.float16),
            "k_sink": (kvq.KVQ_BUF_K_SINK, torch.float16), "v_sink": (kvq.KVQ_BUF_V_SINK, torch.float16)}
    guards = {}
    for name, (idx, dt) in spec.items():
        g = Guarded(sizes[idx], dt)
        guards[name] = g
        setattr(cache, name, g.t)
        setattr(cache.desc, name, g.t.data_ptr() if g.n else g.raw.data_ptr() + PAD)
    for name in ("n_quant", "n_tail", "tail_head", "n_sink"):
        g = Guarded(4 * B, torch.int32)
        guards[name] = g
        setattr(cache, name, g.t)
        setattr(cache.desc, name, g.t.data_ptr())
    g = Guarded(4, torch.int32)
    guards["error_flags"] = g
    cache.error_flags = g.t
    cache.desc.error_flags = g.t.data_ptr()
    return guards


def guard_workspace(cache, n_q_heads: int, guards: dict):
    g = Guarded(kvq.kvq_decode_workspace_bytes(cache, n_q_heads))
    guards["workspace"] = g
    cache._workspaces[n_q_heads] = g.t
    return g.t


def guarded_out(shape, guards: dict, name="out"):
    g = Guarded(int(np.prod(shape)) * 4, torch.float32, fill=float("nan"))
    guards[name] = g
    return g.t.view(*shape)


UNIFORM = {
    # name: (workload, bits, max_tokens, tail_cap, sink_cap)
    "gqa4_d128_2bit_ragged": (S.SERVING.scaled(batch=5, context=700, ragged=(0, 700), bits=2), 2, 768, 64, 0),
    "mha_d128_4bit": (S.LLAMA2_13B.scaled(batch=3, n_q_heads=4, n_kv_heads=4, context=300, n_tail=12), 4, 320, 32, 0),
    "gqa8_d64_8bit": (S.TINY.scaled(batch=2, n_q_heads=8, n_kv_heads=1, context=250, n_tail=26), 8, 256, 32, 0),
    "gqa2_d128_2bit_sinks": (S.SERVING.scaled(batch=3, n_q_heads=4, n_kv_heads=2, context=400, ragged=(2, 400),
                                              bits=2), 2, 448, 32, 5),
}


@pytest.mark.parametrize("name", list(UNIFORM))
def test_uniform_cache_writes_stay_in_bounds(name):
    w, bits, cap, R, sink = UNIFORM[name]
    inp = S.generate(w)
    if w.ragged is not None:
        inp["seq_len"][0] = 0  # one empty sequence
        L = inp["seq_len"].astype(int)
        ns = np.minimum(sink, L)
        inp["n_tail"] = ((L - ns) % 32).astype(np.int32)
    cache = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, bits, cap, R, sink_cap=sink)
    guards = guard_cache(cache)
    k = torch.from_numpy(inp["K"]).cuda()
    v = torch.from_numpy(inp["V"]).cuda()
    q = torch.from_numpy(inp["q"]).cuda()
    cache.prefill(k, v, inp["seq_len"].tolist(), inp["n_tail"].tolist())
    _assert_intact(guards, "prefill")
    hq = w.n_q_heads
    guard_workspace(cache, hq, guards)
    out = guarded_out(q.shape, guards)
    cache.decode(q, w.sm_scale, out=out)
    _assert_intact(guards, "decode")
    assert torch.isfinite(out).all()
    # appends through several flushes (and, for the longest sequences, up to the
    # capacity error, which must leave them unchanged and write nothing else)
    kn = torch.randn(w.batch, w.n_kv_heads, w.head_dim, device="cuda").half()
    vn = torch.randn(w.batch, w.n_kv_heads, w.head_dim, device="cuda").half()
    for i in range(3 * R + 7):
        cache.append(kn, vn)
        if i % R == R - 1:
            _assert_intact(guards, f"append {i}")
    _assert_intact(guards, "append")
    cache.decode(q, w.sm_scale, out=out)
    _assert_intact(guards, "decode after appends")
    out2 = guarded_out(q.shape, guards, "out_static")
    kvq.kvq_decode_attn_static(cache, q, out2, w.sm_scale)
    _assert_intact(guards, "static decode")
    assert torch.equal(out, out2)


def test_prerope_decode_writes_stay_in_bounds():
    w = S.SERVING.scaled(batch=3, context=520, ragged=(1, 520), bits=4)
    inp = S.generate(w)
    inp["n_tail"] = (inp["seq_len"] % 32).astype(np.int32)
    cache = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, 4, 544, 32)
    guards = guard_cache(cache)
    cache.prefill(torch.from_numpy(inp["K"]).cuda(), torch.from_numpy(inp["V"]).cuda(),
                  inp["seq_len"].tolist(), inp["n_tail"].tolist())
    tg = Guarded(kvq.kvq_rope_table_bytes(cache), torch.float32)
    guards["rope_table"] = tg
    kvq.kvq_rope_table(cache, 500000.0, tg.t)
    _assert_intact(guards, "rope table")
    q = torch.from_numpy(inp["q"]).cuda()
    ws = guard_workspace(cache, w.n_q_heads, guards)
    out = guarded_out(q.shape, guards)
    kvq.kvq_decode_attn_rope(cache, q, out, w.sm_scale, tg.t, ws)
    _assert_intact(guards, "pre-RoPE decode")
    assert torch.isfinite(out).all()


def test_mixed_width_writes_stay_in_bounds():
    w = S.TRIZONE.scaled(batch=3, n_q_heads=8, n_kv_heads=2, context=700, trizone_fresh=60)
    inp = S.generate(w)
    t_old = [640, 17, 0]     # a short segment (partial blocks) and one with no old token
    fresh = [60, 33, 5]
    cache = kvq.TriZoneCache(3, 2, 640, 64)
    sizes = kvq.kvq_trizone_bytes(cache.desc)
    guards = {}
    for name, idx, dt in (("index", kvq.KVQ_TZ_BUF_INDEX, torch.uint8), ("tokens", kvq.KVQ_TZ_BUF_TOKENS, torch.int32),
                          ("blocks", kvq.KVQ_TZ_BUF_BLOCKS, torch.uint8)):
        g = Guarded(sizes[idx], dt)
        guards[name] = g
        setattr(cache, name, g.t)
        setattr(cache.desc, name, g.t.data_ptr())
    ef = Guarded(16, torch.int32)
    guards["error_flags"] = ef
    cache.error_flags = ef.t
    cache.desc.error_flags = ef.t.data_ptr()
    vw = torch.from_numpy(np.ascontiguousarray(inp["v_width"][:, :, :640])).cuda()
    kw = torch.from_numpy(inp["k_width"]).cuda()
    cache.build(torch.from_numpy(inp["K"]).cuda(), torch.from_numpy(inp["V"]).cuda(), vw, kw, t_old, fresh)
    _assert_intact(guards, "mixed-width build")
    q = torch.from_numpy(inp["q"]).cuda()
    g = Guarded(kvq.kvq_trizone_decode_workspace_bytes(cache, 8))
    guards["workspace"] = g
    cache._workspaces[8] = g.t
    out = guarded_out(q.shape, guards)
    cache.decode(q, w.sm_scale, out=out)
    _assert_intact(guards, "mixed-width decode")
    assert torch.isfinite(out).all() and cache.device_errors() == 0


def test_rdkv_writes_stay_in_bounds():
    w = S.TRIZONE.scaled(name="rdkv_guard", batch=2, n_q_heads=8, n_kv_heads=2, context=200, seed=77,
                         trizone_fresh=0)
    inp = S.generate(w)
    qn = S.prompt_queries(w)
    a = kvq.RDKVAllocator(2, 8, 2, 200, 160)
    guards = {}
    for name, nbytes, dt in (("workspace", a.workspace.numel(), torch.uint8), ("w", a.w.numel() * 4, torch.float32),
                             ("v_width", a.v_width.numel(), torch.uint8), ("k_width", a.k_width.numel(), torch.uint8),
                             ("W_t", a.W_t.numel() * 4, torch.float32), ("W_c", a.W_c.numel() * 4, torch.float32)):
        old = getattr(a, name)
        g = Guarded(nbytes, dt)
        guards[name] = g
        setattr(a, name, g.t.view(old.shape))
    q, k, v = (torch.from_numpy(x).cuda() for x in (qn, inp["K"], inp["V"]))
    a.run(q, k, v, [200, 131], [160, 100], 3.0, 4.0, w.sm_scale)
    _assert_intact(guards, "RDKV allocation")
