"""CPU oracle for the RDKV bit allocation that feeds the mixed-width cache.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this module.  It shares no code with the
CUDA path and imports nothing from it.

What it computes follows the RDKV summary (gist.science 2605.08317):

* Section 2.1, V cache: the distortion weight of a token is the total
  attention it receives over every query position, w_t = sum_tau a[tau, t].
* Section 2.1, K cache: the weight of a channel is the product of the norms of
  the matching query and key columns over sqrt(d):
  w_c = ||Q[:, c]||_2 * ||K[:, c]||_2 / sqrt(d).
* Section 2.1, objective: minimise sum_u w_u * sigma_u * 2^(-b_u) subject to
  sum_u b_u <= B.
* Section 2.2, allocation pipeline: weights once after prefill from the
  uncompressed cache (phase 1); a multiple-choice knapsack over token V widths
  {0, 2, 4, 8, 16} (phase 2, width 0 = eviction); then the same over channel
  K widths for the tokens kept in phase 2 (phase 3); solved by Lagrangian
  relaxation (reverse water-filling over the discrete widths).

Readings taken where the pages leave a step open (listed in the design notes):

* Units and budgets are per (sequence, KV head).  A token's weight sums the
  attention of every query head of its GQA group; queries are all prompt
  positions tau, with causal attention (query tau sees keys 0..tau); the
  weight is needed for the old tokens t < t_old only.
* The channel norms run over all prompt positions and the group's query heads
  (Q) and over the kept old tokens (K).
* sigma_u is the unit's population variance: over the D channels of the token's
  V row (phase 2), over the kept old tokens of the channel's keys (phase 3).
* Key widths are {2, 4, 8} (the widths the mixed-width layout stores).
* Budget: floor(average bits per unit * number of units), computed in float64.
* The Lagrangian choice for a multiplier lam is, per unit, the width b that
  minimises cost(b) = fl32(fl32(W * 2^-b) + fl32(lam * b)) with W = w * sigma
  (float32), ties to the smaller width; lam is the smallest float32 >= 0, found
  by binary search over its bit pattern, whose choices fit the budget (the
  largest finite float32 when none does).
"""
from __future__ import annotations

import math

import numpy as np

V_WIDTHS = (0, 2, 4, 8, 16)
K_WIDTHS = (2, 4, 8)
LAMBDA_BITS_MAX = 0x7F7FFFFF  # bit pattern of the largest finite float32


def token_weights(q: np.ndarray, k: np.ndarray, sm_scale: float) -> np.ndarray:
    """w[t] = sum over heads g and query positions tau >= t of the causal
    attention a_g[tau, t] = softmax_t'(sm_scale * q_g[tau] . k[t'])[t], t' <= tau.

    q: [T, G, D] (query heads of one GQA group), k: [T, D].  float64 math.
    Returns w [T] for every key position."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    T = k.shape[0]
    w = np.zeros(T, dtype=np.float64)
    causal = np.tril(np.ones((T, T), dtype=bool))  # [tau, t]: t <= tau
    for g in range(q.shape[1]):
        s = sm_scale * (q[:, g, :] @ k.T)  # [tau, t]
        s = np.where(causal, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        w += p.sum(axis=0)
    return w


def row_stats(q: np.ndarray, k: np.ndarray, sm_scale: float):
    """Per query row of head g: m = max_t<=tau (sm_scale q.k) and
    l = sum_t<=tau exp(sm_scale q.k - m).  Returns (m, l), each [T, G]."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    T = k.shape[0]
    causal = np.tril(np.ones((T, T), dtype=bool))
    m = np.zeros((T, q.shape[1]))
    l = np.zeros((T, q.shape[1]))
    for g in range(q.shape[1]):
        s = np.where(causal, sm_scale * (q[:, g, :] @ k.T), -np.inf)
        m[:, g] = s.max(axis=1)
        l[:, g] = np.exp(s - m[:, g:g + 1]).sum(axis=1)
    return m, l


def channel_weights(q: np.ndarray, k_kept: np.ndarray) -> np.ndarray:
    """w_c = ||Q[:, c]|| * ||K[:, c]|| / sqrt(D); q [T, G, D] (all positions and
    heads of the group are the rows of Q), k_kept [N, D]."""
    q = np.asarray(q, dtype=np.float64).reshape(-1, q.shape[-1])
    k_kept = np.asarray(k_kept, dtype=np.float64)
    d = q.shape[1]
    return np.sqrt((q * q).sum(axis=0)) * np.sqrt((k_kept * k_kept).sum(axis=0)) / math.sqrt(d)


def variance(x: np.ndarray, axis: int) -> np.ndarray:
    """Population variance (mean of squared deviations from the mean); an empty
    axis gives 0."""
    x = np.asarray(x, dtype=np.float64)
    if x.shape[axis] == 0:
        shape = list(x.shape)
        del shape[axis]
        return np.zeros(shape)
    mu = x.mean(axis=axis, keepdims=True)
    return ((x - mu) ** 2).mean(axis=axis)


def budget_bits(avg_bits: float, n_units: int) -> int:
    """Total bits allowed for n units at avg_bits each: floor in float64."""
    return int(math.floor(float(avg_bits) * float(n_units)))


def choose(W: np.ndarray, lam_bits: int, widths) -> np.ndarray:
    """Per unit, the width minimising fl32(fl32(W 2^-b) + fl32(lam b)); ties go to
    the smaller width (widths ascending).  W float32 [N]."""
    W = np.asarray(W, dtype=np.float32)
    lam = np.array([lam_bits], dtype=np.uint32).view(np.float32)[0]

    def cost(b):
        dist = (W * np.float32(2.0 ** -b)).astype(np.float32)
        rate = np.float32(lam * np.float32(b))
        return (dist + rate).astype(np.float32)

    with np.errstate(over="ignore", under="ignore"):
        best = cost(widths[0])
        out = np.full(W.shape, widths[0], dtype=np.uint8)
        for b in widths[1:]:
            c = cost(b)
            take = c < best
            best = np.where(take, c, best)
            out = np.where(take, np.uint8(b), out)
    return out


def allocate(W: np.ndarray, widths, budget: int):
    """Lagrangian allocation: the smallest float32 multiplier (by bit pattern,
    binary search) whose per-unit choices fit the budget.  Returns (widths uint8
    [N], lam_bits)."""
    W = np.asarray(W, dtype=np.float32)

    def total(bits):
        return int(choose(W, bits, widths).astype(np.int64).sum())

    lo, hi = 0, LAMBDA_BITS_MAX
    if total(hi) > budget:
        return choose(W, hi, widths), hi
    while lo < hi:
        mid = (lo + hi) // 2
        if total(mid) <= budget:
            hi = mid
        else:
            lo = mid + 1
    return choose(W, lo, widths), lo


def segment_allocation(q: np.ndarray, k: np.ndarray, v: np.ndarray, t_old: int, sm_scale: float,
                       v_avg_bits: float, k_avg_bits: float, w_tokens=None):
    """The three phases for one (sequence, KV head).

    q [T, G, D], k and v [T, D] (prompt positions 0..T-1; tokens t < t_old are
    old).  w_tokens: token weights to use (default: token_weights over the
    prompt).  Returns a dict with w_t, sigma_t, W_t (float32), v_width, kept,
    w_c, sigma_c, W_c (float32), k_width."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    w_t = token_weights(q, k, sm_scale)[:t_old] if w_tokens is None else np.asarray(w_tokens)[:t_old]
    sigma_t = variance(v[:t_old], axis=1)
    W_t = (np.asarray(w_t, dtype=np.float64) * sigma_t).astype(np.float32)
    v_width, _ = allocate(W_t, V_WIDTHS, budget_bits(v_avg_bits, t_old))
    kept = v_width != 0
    k_kept = k[:t_old][kept]
    w_c = channel_weights(q, k_kept)
    sigma_c = variance(k_kept, axis=0)
    W_c = (w_c * sigma_c).astype(np.float32)
    k_width, _ = allocate(W_c, K_WIDTHS, budget_bits(k_avg_bits, k.shape[1]))
    return {"w_t": w_t, "sigma_t": sigma_t, "W_t": W_t, "v_width": v_width, "kept": kept,
            "w_c": w_c, "sigma_c": sigma_c, "W_c": W_c, "k_width": k_width}
