"""Pins of the RDKV allocation oracle to things other than itself: hand-worked
examples (tests/golden), closed forms, brute force on tiny inputs written as
plain loops, and the optimality that defines a Lagrangian solution."""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import rdkv_oracle as R

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rdkv_allocation_examples.txt")


# ------------------------------------------------------------- token weights
def _token_weights_loops(q, k, sm_scale):
    # RDKV summary, section 2.1: w_t = sum over query positions of the attention
    # token t receives; causal: query tau attends keys 0..tau.  Plain loops.
    T, G, _ = q.shape
    w = [0.0] * T
    for g in range(G):
        for tau in range(T):
            s = [sm_scale * sum(float(q[tau, g, d]) * float(k[t, d]) for d in range(k.shape[1]))
                 for t in range(tau + 1)]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for t in range(tau + 1):
                w[t] += e[t] / tot
    return np.array(w)


def test_token_weights_match_loops_on_tiny_input():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((6, 2, 3))
    k = rng.standard_normal((6, 3)) * 2.0
    np.testing.assert_allclose(R.token_weights(q, k, 0.7), _token_weights_loops(q, k, 0.7), rtol=1e-12)


def test_token_weights_sum_to_rows():
    # every query row's attention sums to one: sum_t w_t = G * T
    rng = np.random.default_rng(2)
    q = rng.standard_normal((50, 4, 8))
    k = rng.standard_normal((50, 8)) * 3
    assert abs(R.token_weights(q, k, 0.3).sum() - 200.0) < 1e-9


def test_token_weights_identical_keys_harmonic():
    # all keys equal: a[tau, t] = 1/(tau+1), so w_t = G (H_T - H_t)
    T, G = 20, 3
    rng = np.random.default_rng(3)
    q = rng.standard_normal((T, G, 5))
    k = np.tile(rng.standard_normal(5), (T, 1))
    H = np.concatenate([[0.0], np.cumsum(1.0 / np.arange(1, T + 1))])
    np.testing.assert_allclose(R.token_weights(q, k, 1.0), G * (H[T] - H[:T]), rtol=1e-12)


def test_token_weights_single_token():
    assert R.token_weights(np.ones((1, 4, 2)), np.ones((1, 2)), 1.0).tolist() == [4.0]


def test_row_stats_match_loops():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 2, 3))
    k = rng.standard_normal((5, 3))
    m, l = R.row_stats(q, k, 0.5)
    for g in range(2):
        for tau in range(5):
            s = [0.5 * float(np.dot(q[tau, g], k[t])) for t in range(tau + 1)]
            assert abs(m[tau, g] - max(s)) < 1e-12
            assert abs(l[tau, g] - sum(math.exp(x - max(s)) for x in s)) < 1e-12


# ------------------------------------------------------------- channel weights
def test_channel_weights_constant_columns():
    # Q[:, c] = a, K[:, c] = b everywhere: ||Q_c|| = |a| sqrt(T G), ||K_c|| = |b| sqrt(N)
    T, G, N, D = 7, 2, 5, 4
    a = np.array([1.0, -2.0, 0.5, 3.0])
    b = np.array([2.0, 1.0, -4.0, 0.0])
    q = np.broadcast_to(a, (T, G, D))
    k = np.broadcast_to(b, (N, D))
    expect = np.abs(a) * math.sqrt(T * G) * np.abs(b) * math.sqrt(N) / math.sqrt(D)
    np.testing.assert_allclose(R.channel_weights(q, k), expect, rtol=1e-12)


def test_variance_by_hand():
    assert R.variance(np.array([[1.0, 2.0, 3.0, 4.0]]), axis=1).tolist() == [1.25]
    assert R.variance(np.full((3, 9), 7.5), axis=1).tolist() == [0.0, 0.0, 0.0]
    assert R.variance(np.zeros((0, 4)), axis=0).tolist() == [0.0] * 4


# ------------------------------------------------------------- allocation
def _golden():
    rows = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, widths, W, budget, expect, lam = [f.strip() for f in line.split("|")]
        rows.append((kind, tuple(int(x) for x in widths.split()), np.array([float(x) for x in W.split()],
                     np.float32), int(budget), [int(x) for x in expect.split()], int(lam, 16)))
    return rows


@pytest.mark.parametrize("case", _golden(), ids=lambda c: c[0])
def test_allocation_hand_examples(case):
    _, widths, W, budget, expect, lam = case
    got, lam_bits = R.allocate(W, widths, budget)
    assert got.tolist() == expect
    assert lam_bits == lam


def _exact_cost(W, x):
    return sum(Fraction(float(w)) / 2 ** b for w, b in zip(W, x))


@pytest.mark.parametrize("seed", range(6))
def test_allocation_is_optimal_for_its_bits(seed):
    # A Lagrangian solution x minimises cost + lam * bits, so no assignment using
    # at most bits(x) bits costs less (brute force over all 5^n assignments).
    rng = np.random.default_rng(seed)
    n = 4
    W = (rng.integers(1, 64, n) * 2.0 ** rng.integers(-3, 4, n)).astype(np.float32)
    budget = int(rng.integers(0, 16 * n))
    x, _ = R.allocate(W, R.V_WIDTHS, budget)
    bx = int(x.astype(int).sum())
    assert bx <= budget
    cx = _exact_cost(W, x.tolist())
    for y in itertools.product(R.V_WIDTHS, repeat=n):
        if sum(y) <= bx:
            assert _exact_cost(W, y) >= cx * (1 - Fraction(1, 10 ** 6))


def test_allocation_extremes():
    W = np.array([0.5, 3.0, 100.0], np.float32)
    assert R.allocate(W, R.V_WIDTHS, 48)[0].tolist() == [16, 16, 16]   # lam = 0
    assert R.allocate(W, R.V_WIDTHS, 0)[0].tolist() == [0, 0, 0]
    assert R.allocate(W, R.K_WIDTHS, 5)[0].tolist() == [2, 2, 2]       # below the minimum: all 2


def test_allocation_monotone_in_budget():
    rng = np.random.default_rng(9)
    W = rng.exponential(1.0, 40).astype(np.float32)
    prev = np.zeros(40, np.uint8)
    for budget in range(0, 641, 37):
        x, _ = R.allocate(W, R.V_WIDTHS, budget)
        assert (x >= prev).all() and int(x.astype(int).sum()) <= budget
        prev = x


def test_budget_floor():
    assert R.budget_bits(3.0, 65408) == 196224
    assert R.budget_bits(2.5, 3) == 7


# ------------------------------------------------------------- the three phases together
SEGMENT = os.path.join(os.path.dirname(__file__), "golden", "rdkv_segment_example.txt")


def _segment_example():
    rec = {}
    for line in open(SEGMENT):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, val = (f.strip() for f in line.split("|"))
        rows = [[float(x) if not x.startswith("0x") else int(x, 16) for x in r.split()] for r in val.split(";")]
        rec[key] = rows if len(rows) > 1 else rows[0]
    return rec


def test_segment_allocation_hand_example():
    # phase 2 evicts two tokens; phase 3 must take its statistics over the two
    # kept tokens only (over all four, the key widths would come out reversed)
    ex = _segment_example()
    q = np.array(ex["q_rows"])[:, None, :]        # [T, G = 1, D]
    k, v = np.array(ex["k_rows"]), np.array(ex["v_rows"])
    out = R.segment_allocation(q, k, v, 4, 1.0, ex["v_avg_bits"][0], ex["k_avg_bits"][0],
                               w_tokens=np.array(ex["w_t"]))
    assert out["sigma_t"].tolist() == ex["sigma_t"]
    assert out["v_width"].tolist() == [int(x) for x in ex["v_width"]]
    assert out["kept"].tolist() == [True, True, False, False]
    np.testing.assert_allclose(out["w_c"], ex["w_c"], rtol=1e-15, atol=1e-15)
    assert out["sigma_c"].tolist() == ex["sigma_c"]
    assert out["k_width"].tolist() == [int(x) for x in ex["k_width"]]
    # the multipliers of the hand derivation
    assert R.allocate(out["W_t"], R.V_WIDTHS, 4)[1] == ex["v_lam_bits"][0]
    assert R.allocate(out["W_c"], R.K_WIDTHS, 10)[1] == ex["k_lam_bits"][0]
    # the statistics over all tokens give the reversed key widths (the example
    # separates the two readings)
    W_all = (R.channel_weights(q, k) * R.variance(k, axis=0)).astype(np.float32)
    assert R.allocate(W_all, R.K_WIDTHS, 10)[0].tolist() == [int(x) for x in ex["k_width_all_tokens"]]


@pytest.mark.parametrize("seed", range(3))
def test_segment_allocation_is_the_phases_in_order(seed):
    # phase 1 (token weights over the prompt) -> phase 2 (value widths of the old
    # tokens within floor(v_bits * t_old)) -> phase 3 (channel weights and
    # variances over the kept old tokens, key widths within floor(k_bits * D)),
    # each step called separately
    rng = np.random.default_rng(100 + seed)
    T, G, D, t_old = 48, 2, 8, 40
    q = rng.standard_normal((T, G, D))
    k = rng.standard_normal((T, D)) * np.array([1, 1, 6, 1, 1, 1, 3, 1])
    v = rng.standard_normal((T, D)) * np.exp(rng.standard_normal((T, 1)))
    vb, kb = 2.5, 4.0
    out = R.segment_allocation(q, k, v, t_old, 0.35, vb, kb)
    w = R.token_weights(q, k, 0.35)[:t_old]
    Wt = (w * R.variance(v[:t_old], axis=1)).astype(np.float32)
    vw, _ = R.allocate(Wt, R.V_WIDTHS, R.budget_bits(vb, t_old))
    kept = k[:t_old][vw != 0]
    Wc = (R.channel_weights(q, kept) * R.variance(kept, axis=0)).astype(np.float32)
    kw, _ = R.allocate(Wc, R.K_WIDTHS, R.budget_bits(kb, D))
    assert out["v_width"].tolist() == vw.tolist() and out["k_width"].tolist() == kw.tolist()
    # budgets: the value bits fit floor(2.5 * 40) = 100; the key bits fit floor(4 * 8) = 32
    assert int(out["v_width"].astype(int).sum()) <= 100
    assert int(out["k_width"].astype(int).sum()) <= 32
    assert 0 < out["kept"].sum() < t_old  # the budget evicts some tokens and keeps others
