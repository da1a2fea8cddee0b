"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
binding and the oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import kvq_oracle as O
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S

# Decode attention tolerance against the fp64 oracle (the target's own bar).
ATOL_MAX = 2e-3
ATOL_MEAN = 1e-3


def device_cache(w: S.Workload, inp: dict, bits: int, max_tokens: int | None = None,
                 tail_cap: int | None = None, k=None, v=None, sink_cap: int = 0) -> kvq.QuantizedKVCache:
    """Allocate a cache and run kvq_quantize_prefill on the workload's K/V."""
    cap = max_tokens if max_tokens is not None else w.context
    cache = kvq.QuantizedKVCache(w.batch, w.n_kv_heads, w.head_dim, bits, cap,
                                 tail_cap or w.tail_cap, sink_cap=sink_cap)
    if k is None:
        k = torch.from_numpy(inp["K"]).cuda()
        v = torch.from_numpy(inp["V"]).cuda()
    cache.prefill(k, v, inp["seq_len"].tolist(), inp["n_tail"].tolist())
    return cache


def oracle_states(inp: dict, bits: int, heads=None, batches=None, sink_cap: int = 0) -> list:
    out = []
    bs = range(inp["K"].shape[0]) if batches is None else batches
    for b in bs:
        k, v = inp["K"][b], inp["V"][b]
        if heads is not None:
            k, v = k[:, heads], v[:, heads]
        out.append(O.quantize_sequence(k, v, int(inp["seq_len"][b]), int(inp["n_tail"][b]), bits,
                                       n_sink_cap=sink_cap))
    return out


def assert_buffers_equal(cache: kvq.QuantizedKVCache, states: list, batches=None, heads=None,
                         groups=None) -> None:
    """Bit-exact comparison of packed codes, metadata, tail and lengths, plus the
    unpacked logical codes (so a layout slip can't hide a value mismatch)."""
    views = cache.views()
    bs = list(range(len(states))) if batches is None else list(batches)
    nq = views["n_quant"].cpu().numpy()
    nt = views["n_tail"].cpu().numpy()
    th = views["tail_head"].cpu().numpy()
    D, bits = cache.head_dim, cache.bits
    for st, b in zip(states, bs):
        assert nq[b] == st["n_quant"] and nt[b] == st["n_tail"], (b, nq[b], nt[b])
        hs = list(range(cache.n_kv_heads)) if heads is None else list(heads)
        ng = st["n_quant"] // 32
        gs = list(range(ng)) if groups is None else [g for g in groups if g < ng]
        if gs:
            hsel = torch.tensor(hs)
            gsel = torch.tensor(gs)
            kc = views["k_codes"][b][hsel][:, gsel].cpu().numpy()
            vc = views["v_codes"][b][hsel][:, gsel].cpu().numpy()
            km = views["k_meta"][b][hsel][:, gsel].cpu().numpy()
            vm = views["v_meta"][b][hsel][:, gsel].cpu().numpy()
            ek = st["k_codes"].reshape(len(hs), ng, 32, D)[:, gs]
            ev = st["v_codes"].reshape(len(hs), ng, 32, D)[:, gs]
            assert (O.unpack_tiles(kc, "K", D, bits) == ek).all(), "key codes differ"
            assert (O.unpack_tiles(vc, "V", D, bits) == ev).all(), "value codes differ"
            assert (kc == O.pack_tiles(ek, "K", bits)).all(), "packed key bytes differ"
            assert (vc == O.pack_tiles(ev, "V", bits)).all(), "packed value bytes differ"
            ekm = O.pack_key_meta(st["k_scale"][:, gs], st["k_zero"][:, gs])
            assert (km.view(np.uint16) == ekm.view(np.uint16)).all(), "key scales/zeros differ"
            vs = st["v_scale"].reshape(len(hs), ng, 32, D // 32)[:, gs]
            vz = st["v_zero"].reshape(len(hs), ng, 32, D // 32)[:, gs]
            evm = O.pack_value_meta(vs, vz)
            assert (vm.reshape(evm.shape).view(np.uint16) == evm.view(np.uint16)).all(), \
                "value scales/zeros differ"
        # tail in logical order through the ring
        R = cache.tail_cap
        slots = (th[b] + np.arange(st["n_tail"])) % R
        kt = views["k_tail"][b][torch.tensor(hs)].cpu().numpy()[:, slots]
        vt = views["v_tail"][b][torch.tensor(hs)].cpu().numpy()[:, slots]
        assert (kt.view(np.uint16) == st["k_tail"].view(np.uint16)).all(), "key tail differs"
        assert (vt.view(np.uint16) == st["v_tail"].view(np.uint16)).all(), "value tail differs"
        if cache.sink_cap > 0:
            ns = int(views["n_sink"][b])
            assert ns == st["n_sink"], (b, ns, st["n_sink"])
            ks = views["k_sink"][b][torch.tensor(hs)].cpu().numpy()[:, :ns]
            vs = views["v_sink"][b][torch.tensor(hs)].cpu().numpy()[:, :ns]
            assert (ks.view(np.uint16) == st["k_sink"].view(np.uint16)).all(), "key sinks differ"
            assert (vs.view(np.uint16) == st["v_sink"].view(np.uint16)).all(), "value sinks differ"


def oracle_decode(q: np.ndarray, states: list, sm_scale: float, heads=None) -> np.ndarray:
    """[B, Hq, D] float64 for the sequences in states (all query heads of the
    KV heads kept in the states, or of `heads`)."""
    outs = []
    for b, st in enumerate(states):
        outs.append(O.sequence_attention(q[b], st, sm_scale))
    return np.stack(outs)


def assert_close(got: np.ndarray, ref: np.ndarray, atol_max=ATOL_MAX, atol_mean=ATOL_MEAN):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all(), "non-finite output"
    assert err.max() <= atol_max, f"max abs error {err.max():.3e} > {atol_max}"
    assert err.mean() <= atol_mean, f"mean abs error {err.mean():.3e} > {atol_mean}"
    return err.max(), err.mean()
