"""RDKV allocation on the GPU against the oracle (RDKV summary, sections 2.1-2.2):
token weights within 1e-4 relative of the fp64 oracle; the costs W_t within
1e-5 and W_c within 1e-4 relative (fp32 sums); the widths bit-exact, given the GPU's own costs (the
decision procedure is exact float32 arithmetic on both sides)."""
import numpy as np
import pytest
import torch

from oracle import kvq_oracle as O
from oracle import rdkv_oracle as R
from quantized_kv_cache_11_gb300 import kvq
from quantized_kv_cache_11_gb300 import synthetic as S
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _inputs(batch, hq, hkv, T, seed):
    w = S.TRIZONE.scaled(name=f"rdkv_{seed}", batch=batch, n_q_heads=hq, n_kv_heads=hkv, context=T, seed=seed,
                         trizone_fresh=0)
    inp = S.generate(w)
    return w, S.prompt_queries(w), inp["K"], inp["V"]


def _run(w, q, k, v, n_tokens, t_old, v_bits, k_bits, max_old=None):
    dev = torch.device("cuda")
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    max_old = max(t_old) if max_old is None else max_old
    a = kvq.RDKVAllocator(w.batch, w.n_q_heads, w.n_kv_heads, w.context, max(max_old, 1))
    a.run(qd, kd, vd, n_tokens, t_old, v_bits, k_bits, w.sm_scale)
    torch.cuda.synchronize()
    return a


@pytest.mark.parametrize("hq,hkv", [(2, 2), (8, 2), (16, 2)])
def test_token_weights_match_oracle(hq, hkv):
    w, q, k, v = _inputs(2, hq, hkv, 256, seed=20 + hq)
    n_tokens = [201, 256]
    a = _run(w, q, k, v, n_tokens, [150, 200], 3.0, 4.0)
    got = a.w.cpu().numpy()
    G = hq // hkv
    for b in range(2):
        n = n_tokens[b]
        for h in range(hkv):
            ref = R.token_weights(q[b, :n, h * G:(h + 1) * G], k[b, :n, h], w.sm_scale)
            np.testing.assert_allclose(got[b, h, :n], ref, rtol=1e-4, atol=1e-7)
            assert abs(got[b, h, :n].astype(np.float64).sum() - G * n) < 1e-4 * G * n


def test_allocation_bit_exact_given_costs():
    w, q, k, v = _inputs(2, 8, 2, 320, seed=31)
    n_tokens, t_old = [320, 257], [300, 200]
    v_bits, k_bits = 3.0, 4.5
    a = _run(w, q, k, v, n_tokens, t_old, v_bits, k_bits, max_old=304)
    wt, Wt, Wc = a.w.cpu().numpy(), a.W_t.cpu().numpy(), a.W_c.cpu().numpy()
    vw, kw = a.v_width.cpu().numpy(), a.k_width.cpu().numpy()
    G = 4
    for b in range(2):
        to, n = t_old[b], n_tokens[b]
        for h in range(2):
            # costs from the GPU's token weights, in float64
            sig = R.variance(v[b, :to, h].astype(np.float64), axis=1)
            np.testing.assert_allclose(Wt[b, h, :to], wt[b, h, :to].astype(np.float64) * sig, rtol=1e-5, atol=1e-30)
            ref_vw, _ = R.allocate(Wt[b, h, :to], R.V_WIDTHS, R.budget_bits(v_bits, to))
            assert (vw[b, h, :to] == ref_vw).all()
            kept = vw[b, h, :to] != 0
            kk = k[b, :to, h].astype(np.float64)[kept]
            ref_wc = R.channel_weights(q[b, :n, h * G:(h + 1) * G], kk) * R.variance(kk, axis=0)
            np.testing.assert_allclose(Wc[b, h], ref_wc, rtol=1e-4, atol=1e-30)
            ref_kw, _ = R.allocate(Wc[b, h], R.K_WIDTHS, R.budget_bits(k_bits, 128))
            assert (kw[b, h] == ref_kw).all()
            assert int(vw[b, h, :to].astype(int).sum()) <= R.budget_bits(v_bits, to)


def _unexplained(W_ref, x_gpu, x_ref, lam_gpu, lam_ref, rel):
    """Units whose widths differ although no decision threshold separates them.
    A unit takes width a at multiplier lam_a and b > a at lam_b only if its
    switch point W (2^-a - 2^-b) / (b - a) lies in [lam_b, lam_a] (each choice
    minimises W 2^-x + lam x); with the two sides' costs W within a relative
    `rel` of each other, a difference is explained when the reference's switch
    point lies in that band widened by rel."""
    f = lambda bits: float(np.array([bits], np.uint32).view(np.float32)[0])
    lo = min(f(lam_gpu), f(lam_ref)) * (1 - rel)
    hi = max(f(lam_gpu), f(lam_ref)) * (1 + rel)
    bad = []
    for u in np.nonzero(x_gpu != x_ref)[0]:
        a, b = sorted((int(x_gpu[u]), int(x_ref[u])))
        tau = float(W_ref[u]) * (2.0 ** -a - 2.0 ** -b) / (b - a)
        if not lo <= tau <= hi:
            bad.append((int(u), a, b, tau, lo, hi))
    return bad


@pytest.mark.parametrize("seed", [41, 42, 43])
def test_allocation_matches_full_oracle(seed):
    # the whole pipeline against the oracle's own fp64 pipeline: every width
    # equal, except units whose switch point lies between the two sides'
    # multipliers (the GPU's costs are fp32 sums, within 1e-4 relative)
    w, q, k, v = _inputs(1, 4, 1, 192, seed=seed)
    a = _run(w, q, k, v, [192], [160], 2.5, 4.0)
    ref = R.segment_allocation(q[0, :, 0:4], k[0, :, 0], v[0, :, 0], 160, w.sm_scale, 2.5, 4.0)
    vw = a.v_width.cpu().numpy()[0, 0, :160]
    Wt_gpu = a.W_t.cpu().numpy()[0, 0, :160]
    np.testing.assert_allclose(Wt_gpu, ref["W_t"], rtol=1e-4, atol=1e-30)
    budget_v = R.budget_bits(2.5, 160)
    _, lam_ref = R.allocate(ref["W_t"], R.V_WIDTHS, budget_v)
    _, lam_gpu = R.allocate(Wt_gpu, R.V_WIDTHS, budget_v)  # the GPU's decision (bit-exact given its costs)
    assert _unexplained(ref["W_t"], vw, ref["v_width"], lam_gpu, lam_ref, 2e-4) == []
    assert (vw == ref["v_width"]).mean() >= 0.95
    # phase 3 on the same kept set: key widths equal up to switch points in the band
    if ((vw != 0) == ref["kept"]).all():
        kw = a.k_width.cpu().numpy()[0, 0]
        Wc_gpu = a.W_c.cpu().numpy()[0, 0]
        np.testing.assert_allclose(Wc_gpu, ref["W_c"], rtol=1e-4, atol=1e-30)
        _, lk_ref = R.allocate(ref["W_c"], R.K_WIDTHS, R.budget_bits(4.0, 128))
        _, lk_gpu = R.allocate(Wc_gpu, R.K_WIDTHS, R.budget_bits(4.0, 128))
        assert _unexplained(ref["W_c"], kw, ref["k_width"], lk_gpu, lk_ref, 2e-4) == []


@pytest.mark.parametrize("v_bits,k_bits", [(0.0, 0.0), (16.0, 8.0), (1.0, 2.0)])
def test_allocation_budget_extremes(v_bits, k_bits):
    w, q, k, v = _inputs(1, 4, 1, 96, seed=51)
    a = _run(w, q, k, v, [96], [64], v_bits, k_bits)
    vw, kw = a.v_width.cpu().numpy()[0, 0, :64], a.k_width.cpu().numpy()[0, 0]
    if v_bits == 0.0:
        assert (vw == 0).all() and (kw == 2).all()   # nothing kept: K costs are 0, ties to 2 bits
    elif v_bits == 16.0:
        assert (vw == 16).all() and (kw == 8).all()
    else:
        assert int(vw.astype(int).sum()) <= 64 and int(kw.astype(int).sum()) == 256


def test_empty_and_single_token_sequences():
    w, q, k, v = _inputs(3, 4, 1, 64, seed=61)
    n_tokens, t_old = [1, 64, 40], [0, 64, 1]
    a = _run(w, q, k, v, n_tokens, t_old, 3.0, 4.0, max_old=64)
    got = a.w.cpu().numpy()
    assert abs(got[0, 0, 0] - 4.0) < 1e-6                      # one token: all the attention
    ref = R.token_weights(q[2, :40, 0:4], k[2, :40, 0], w.sm_scale)
    np.testing.assert_allclose(got[2, 0, :40], ref, rtol=1e-4)
    assert (a.k_width.cpu().numpy()[0, 0] == 2).all()          # no old token: channel costs 0


def test_allocated_widths_build_and_decode():
    # RDKV widths feed the mixed-width build; decode matches the oracle on that layout
    w, q, k, v = _inputs(2, 8, 2, 288, seed=71)
    n_tokens, t_old, fresh = [288, 250], [224, 200], [64, 50]
    a = _run(w, q, k, v, n_tokens, t_old, 3.0, 4.0, max_old=224)
    dev = torch.device("cuda")
    kd, vd = torch.from_numpy(k).to(dev), torch.from_numpy(v).to(dev)
    cache = kvq.TriZoneCache(2, 2, 224, 64)
    cache.build(kd, vd, a.v_width, a.k_width, t_old, fresh)
    qd = torch.from_numpy(np.ascontiguousarray(q[:, -1])).to(dev)  # one decode query per sequence
    out = cache.decode(qd, w.sm_scale).cpu().numpy()
    assert cache.device_errors() == 0
    vw, kw = a.v_width.cpu().numpy(), a.k_width.cpu().numpy()
    for b in range(2):
        n = t_old[b] + fresh[b]
        tzs = [O.trizone_quantize(k[b, :n, h], v[b, :n, h], vw[b, h, :t_old[b]], kw[b, h]) for h in range(2)]
        ref = O.trizone_attention(q[b, -1], tzs, w.sm_scale)
        H.assert_close(out[b], ref)


@pytest.mark.slow
def test_full_size_sampled():
    # the mixed-width workload's geometry: 4 x 65,536 prompt positions, 32 query
    # heads over 8 KV heads; weights of the last keys (their rows are cheap to
    # recompute), the row-sum identity for every (sequence, KV head), and the
    # widths of two segments bit-exact given the GPU's costs
    w = S.TRIZONE
    inp = S.generate(w)
    q = S.prompt_queries(w)
    T, G = w.context, w.gqa
    t_old = [T - w.trizone_fresh] * w.batch
    a = _run(w, q, inp["K"], inp["V"], [T] * w.batch, t_old, 3.0, 4.0)
    got = a.w.cpu().numpy()
    sums = got.astype(np.float64).sum(axis=2)
    assert np.abs(sums - G * T).max() < 2e-4 * G * T
    for b, h in ((0, 0), (3, 7)):
        kk = inp["K"][b, :, h].astype(np.float64)
        tail = np.zeros(16)
        for tau in range(T - 16, T):
            for g in range(G):
                s = w.sm_scale * (kk[:tau + 1] @ q[b, tau, h * G + g].astype(np.float64))
                p = np.exp(s - s.max())
                p /= p.sum()
                tail[:tau + 1 - (T - 16)] += p[T - 16:tau + 1]
        np.testing.assert_allclose(got[b, h, T - 16:], tail, rtol=1e-4, atol=1e-9)
        Wt = a.W_t.cpu().numpy()[b, h, :t_old[b]]
        ref_vw, _ = R.allocate(Wt, R.V_WIDTHS, R.budget_bits(3.0, t_old[b]))
        assert (a.v_width.cpu().numpy()[b, h, :t_old[b]] == ref_vw).all()
        ref_kw, _ = R.allocate(a.W_c.cpu().numpy()[b, h], R.K_WIDTHS, R.budget_bits(4.0, 128))
        assert (a.k_width.cpu().numpy()[b, h] == ref_kw).all()
