"""Seeded synthetic KV-cache workloads.

This module only draws random numbers and shapes them; it holds none of the
quantizer or attention arithmetic, so both the CUDA path and the CPU oracle can
consume the same inputs.

Workload recipes follow the geometry of the models the pages measure on:

* "KV-cache quantization axes" article (ihal.it, paragraphs 1, 3-5): Llama-2-13B
  (MHA, 40 heads, head_dim 128), 2-bit groups of 32; key outliers concentrate in
  a few channels that are stable across inputs (max ~7000 vs median ~0.3 in
  Mixtral) and are tied to attention sinks.
* VQKV summary (gist.science 2603.16435, section 4) and RDKV summary
  (gist.science 2605.08317, section 4): LLaMA-3.1-8B (32 query heads over 8 KV
  heads, head_dim 128) at 128K context.
* RDKV summary, sections 2.2 and "2.2 TriZone": per-token V widths and
  per-channel K widths drawn from {0,2,4,8,16} / {2,4,8}.

Every tensor is drawn on the CPU with ``torch.Generator().manual_seed(seed)`` in
float32 and rounded to float16, in this order: K, V, q (standard normals), the
outlier-channel choice, the per-sequence lengths, the widths.  Inputs that
stand in for public benchmarks are shapes only; no dataset item is used.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

GROUP = 32  # group size along the grouping axis (article, paragraph 1)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and distribution of one synthetic decode workload."""

    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    context: int  # tokens per sequence held in the K/V arrays
    tail_cap: int  # R: fp16 tail capacity (tokens), multiple of 32
    bits: int
    seed: int
    recipe: str = "llama"  # "llama" (outlier channels + sink) or "tiny"
    n_tail: Optional[int] = None  # fixed tail length; None -> context mod 32
    ragged: Optional[tuple] = None  # (lo, hi): per-sequence lengths ~ U[lo, hi]
    trizone_fresh: int = 0  # >0: mixed-width layout with this many fresh tokens
    v_width_probs: tuple = (0.5, 0.3, 0.1, 0.05, 0.05)  # widths 0,2,4,8,16
    k_width_probs: tuple = (0.6, 0.3, 0.1)  # widths 2,4,8

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    @property
    def gqa(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


V_WIDTHS = (0, 2, 4, 8, 16)
K_WIDTHS = (2, 4, 8)

# The five workloads, indexed 0..4.
TINY = Workload("tiny_d64_t256_2bit", 1, 1, 1, 64, 256, 32, 2, seed=0,
                recipe="tiny", n_tail=0)
LLAMA2_13B = Workload("llama2_13b_mha_b8_t4096_2bit", 8, 40, 40, 128, 4096, 32, 2,
                      seed=1, n_tail=32)
LLAMA31_8B_128K = Workload("llama31_8b_gqa_b1_t131072_2bit", 1, 32, 8, 128, 131072,
                           64, 2, seed=2, n_tail=64)
LLAMA31_8B_128K_4BIT = LLAMA31_8B_128K.scaled(name="llama31_8b_gqa_b1_t131072_4bit",
                                              bits=4)
SERVING = Workload("llama31_8b_serving_b16_ragged_4bit", 16, 32, 8, 128, 32768, 32, 4,
                   seed=3, ragged=(8192, 32768))
TRIZONE = Workload("llama31_8b_trizone_b4_t65536", 4, 32, 8, 128, 65536, 128, 0,
                   seed=4, trizone_fresh=128)

WORKLOADS = {w.name: w for w in (TINY, LLAMA2_13B, LLAMA31_8B_128K,
                                 LLAMA31_8B_128K_4BIT, SERVING, TRIZONE)}


def _categorical(gen: torch.Generator, shape, probs, values) -> np.ndarray:
    u = torch.rand(shape, generator=gen, dtype=torch.float64).numpy()
    edges = np.cumsum(np.asarray(probs, dtype=np.float64))[:-1]
    idx = np.searchsorted(edges, u, side="right")
    return np.asarray(values, dtype=np.uint8)[idx]


def generate(w: Workload) -> dict:
    """Draw one workload.  Returns numpy arrays.

    K, V: float16 [B, T, Hkv, D]; q: float16 [B, Hq, D]; seq_len, n_tail: int32 [B].
    For the mixed-width layout also v_width uint8 [B, Hkv, T - fresh] and
    k_width uint8 [B, Hkv, D].
    """
    g = torch.Generator().manual_seed(w.seed)
    B, T, H, D = w.batch, w.context, w.n_kv_heads, w.head_dim
    k = torch.randn((B, T, H, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, T, H, D), generator=g, dtype=torch.float32)
    q = torch.randn((B, w.n_q_heads, D), generator=g, dtype=torch.float32)
    if w.recipe == "tiny":
        # K channels 3 and 17 scaled x50 (outlier channels), everything else N(0,1).
        k[..., 3] *= 50.0
        k[..., 17] *= 50.0
    elif w.recipe == "llama":
        # K ~ N(0, 0.3); 4 outlier channels per KV head ~ N(0, 30), fixed per head
        # for every sequence and token; token 0 (attention sink) row x10.
        scale = torch.full((H, D), 0.3)
        for h in range(H):
            ch = torch.randperm(D, generator=g)[:4]
            scale[h, ch] = 30.0
        k *= scale
        k[:, 0] *= 10.0
    else:
        raise ValueError(w.recipe)
    out = {
        "K": k.half().numpy(),
        "V": v.half().numpy(),
        "q": q.half().numpy(),
    }
    del k, v
    if w.ragged is not None:
        lo, hi = w.ragged
        seq_len = torch.randint(lo, hi + 1, (B,), generator=g).numpy().astype(np.int32)
    else:
        seq_len = np.full((B,), T - w.trizone_fresh, dtype=np.int32)
    if w.trizone_fresh:
        n_tail = np.full((B,), w.trizone_fresh, dtype=np.int32)
        t_old = T - w.trizone_fresh
        out["v_width"] = _categorical(g, (B, H, t_old), w.v_width_probs, V_WIDTHS)
        out["k_width"] = _categorical(g, (B, H, D), w.k_width_probs, K_WIDTHS)
        seq_len = np.full((B,), T, dtype=np.int32)
    elif w.n_tail is not None:
        n_tail = np.full((B,), w.n_tail, dtype=np.int32)
    else:
        n_tail = (seq_len % GROUP).astype(np.int32)
    out["seq_len"] = seq_len
    out["n_tail"] = n_tail
    return out


def random_groups(seed: int, n: int, dist: str = "normal", scale: float = 1.0,
                  size: int = GROUP) -> np.ndarray:
    """Random float16 groups [n, size] for quantizer tests."""
    g = torch.Generator().manual_seed(seed)
    if dist == "normal":
        x = torch.randn((n, size), generator=g) * scale
    elif dist == "uniform":
        x = (torch.rand((n, size), generator=g) * 2 - 1) * scale
    elif dist == "lognormal":
        x = torch.exp(torch.randn((n, size), generator=g) * 3.0) * torch.sign(
            torch.randn((n, size), generator=g)) * scale
    else:
        raise ValueError(dist)
    return x.clamp(-60000, 60000).half().numpy()


def prompt_queries(w: Workload, batches=None) -> np.ndarray:
    """Query vectors of every prompt position, float16 [B, T, Hq, D], standard
    normals drawn with their own generator (seed + 1000, one batch row after
    another) so the draws of ``generate`` are unchanged.  ``batches``: the rows
    to return (default all); rows are drawn in order, so a subset matches the
    full draw."""
    g = torch.Generator().manual_seed(w.seed + 1000)
    want = range(w.batch) if batches is None else sorted(batches)
    out = []
    for b in range(max(want) + 1):
        x = torch.randn((w.context, w.n_q_heads, w.head_dim), generator=g, dtype=torch.float32).half()
        if b in want:
            out.append(x.numpy())
    return np.stack(out)
