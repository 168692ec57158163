"""Seeded synthetic inputs for the VerKV hot path.

This module only draws random tensors; it contains none of the method's
arithmetic.  The shapes and distributions stand in for the paper's RULER /
LOFT workloads ("Verify Before You Fetch", Sec. 5.1: Qwen3-4B, GQA 32/8,
d = 128, 32K and 128K contexts, 16x compression, eps0 = 0.05, delta = 0.1).

All arrays are numpy; keys/values are float32 arrays whose values are exactly
representable in the workload's storage dtype (bf16 or fp32).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 values that are exact bf16 -> uint16 bit patterns."""
    return (np.ascontiguousarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


@dataclass
class Workload:
    name: str
    n_kv: int
    n_q: int
    d: int
    n: int
    batch: int
    n_sink: int
    n_local: int
    eta: float
    eps: float
    delta: float
    sketch: str            # "exact" | "int8" | "2bit"
    kv_dtype: str          # "bf16" | "f32"
    seed: int              # Philox key for the Poisson sample
    K: np.ndarray          # [batch, n_kv, n, d] float32
    V: np.ndarray          # [batch, n_kv, n, d] float32
    obs_q: np.ndarray      # [batch, n_q, W, d] float32
    queries: np.ndarray    # [steps, batch, n_q, d] float32
    needles: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int64))  # [batch, n_kv, m]
    notes: str = ""

    @property
    def group(self) -> int:
        return self.n_q // self.n_kv

    def kv_host_layout(self, b: int) -> np.ndarray:
        """[n_kv, n, 2, d] in the storage dtype's bit pattern (uint16 for bf16, float32 otherwise)."""
        kv = np.stack([self.K[b], self.V[b]], axis=2)
        if self.kv_dtype == "bf16":
            return bf16_bits(kv)
        return np.ascontiguousarray(kv, np.float32)


def _needle_positions(rng, n, count, lo=4, hi_pad=128):
    return np.sort(rng.choice(np.arange(lo, n - hi_pad), size=count, replace=False))


def tiny_oracle_case(seed: int = 0, n: int = 1024, d: int = 128, steps: int = 4) -> Workload:
    """1 KV head, 1 query head, fp32 K,V ~ N(0,1), 8 observation queries,
    sink 4 + local 64, eta = 1/8, eps = delta = 0.05, exact sketch.
    Decode query q = 3 k_j + N(0,1) with j uniform over the tokens outside the
    sink/local windows (the candidates for L; L itself is known only after
    compression)."""
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((1, 1, n, d), dtype=np.float32)
    V = rng.standard_normal((1, 1, n, d), dtype=np.float32)
    obs = rng.standard_normal((1, 1, 8, d), dtype=np.float32)
    n_sink, n_local = 4, 64
    js = rng.integers(n_sink, n - n_local, size=steps)
    q = np.zeros((steps, 1, 1, d), np.float32)
    for s, j in enumerate(js):
        q[s, 0, 0] = 3.0 * K[0, 0, j] + rng.standard_normal(d, dtype=np.float32)
    return Workload("tiny-oracle-1kv-n1024", 1, 1, d, n, 1, n_sink, n_local, 1.0 / 8, 0.05, 0.05, "exact", "f32",
                    0, K, V, obs, q, js.reshape(1, 1, -1))


def qwen_layer_case(seed: int = 1, n: int = 32768, n_kv: int = 8, n_q: int = 32, d: int = 128,
                    n_needles: int = 16, W: int = 32, steps: int = 64, sketch: str = "2bit",
                    eta: float = 1.0 / 16, eps: float = 0.05, delta: float = 0.05,
                    n_sink: int = 4, n_local: int = 128, batch: int = 1, query_mode: str = "needle_half",
                    philox_seed: int = 0) -> Workload:
    """Qwen3-4B-shaped attention layer: GQA 32/8, d = 128, bf16 K,V ~ N(0,1),
    `n_needles` random high-norm needle keys (x4) per KV head, an observation
    window of W queries per query head, and decode queries of which the even
    steps aim at a needle of the head's KV group (q = 3 k_needle + N(0,1),
    needles taken round-robin) and the odd steps are N(0,1)."""
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((batch, n_kv, n, d), dtype=np.float32)
    V = rng.standard_normal((batch, n_kv, n, d), dtype=np.float32)
    needles = np.zeros((batch, n_kv, n_needles), np.int64)
    for b in range(batch):
        for h in range(n_kv):
            pos = _needle_positions(rng, n, n_needles)
            needles[b, h] = pos
            K[b, h, pos] *= 4.0
    K = round_to_bf16(K)
    V = round_to_bf16(V)
    obs = rng.standard_normal((batch, n_q, W, d), dtype=np.float32)
    G = n_q // n_kv
    q = rng.standard_normal((steps, batch, n_q, d), dtype=np.float32)
    if query_mode == "needle_half":
        for s in range(0, steps, 2):
            for b in range(batch):
                for h in range(n_q):
                    kv = h // G
                    j = needles[b, kv, (s // 2 + h) % n_needles]
                    q[s, b, h] = 3.0 * K[b, kv, j] + q[s, b, h]
    return Workload(f"qwen3-4b-layer-n{n}-{sketch}", n_kv, n_q, d, n, batch, n_sink, n_local, eta, eps, delta,
                    sketch, "bf16", philox_seed, K, V, obs, q, needles)


def long_context_case(seed: int = 3, n: int = 131072, scale: float = 1.3, steps: int = 4, n_needles: int = 64,
                      W: int = 32) -> Workload:
    """Long context: batch 1, GQA 32/8, d = 128, n = 128K, 64 needles per KV
    head, int8 sketch, eta = 1/16, eps = 0.02, delta = 0.05.  Decode queries are
    scale * N(0,1); the default scale was calibrated with the oracle so that
    about 20% of L must be fetched on average (tests/golden/long_context_query_scale.json)."""
    w = qwen_layer_case(seed=seed, n=n, n_needles=n_needles, W=W, steps=steps, sketch="int8", eta=1.0 / 16,
                        eps=0.02, delta=0.05, query_mode="none")
    rng = np.random.default_rng(seed + 1000)
    w.queries = scale * rng.standard_normal(w.queries.shape, dtype=np.float32)
    w.name = f"long-context-n{n}-int8"
    return w


def stack_layer_case(layer: int, base_seed: int = 2, n: int = 32768, batch: int = 8, steps: int = 128) -> Workload:
    """One layer of the 36-layer decode stack: batch 8, GQA 32/8, bf16 K,V as in
    the Qwen-shaped layer, int8 sketch, eta = 1/32, eps = delta = 0.1, random
    N(0,1) decode queries.  Each layer draws its own tensors (seed = base + layer)."""
    w = qwen_layer_case(seed=base_seed * 1000 + layer, n=n, batch=batch, steps=steps, sketch="int8", eta=1.0 / 32,
                        eps=0.1, delta=0.1, query_mode="random")
    w.name = f"stack36-layer{layer}-b{batch}-n{n}-int8"
    return w


def synthetic_scores(n_kv: int, n: int, seed: int = 7, n_hot: int = 64) -> np.ndarray:
    """Seeded importance scores in (0, 1] standing in for a learned scorer's output (the API takes any
    scorer's scores): a heavy-tailed bulk (lognormal, normalised by its maximum) plus `n_hot` tokens
    per KV head near 1.  [n_kv, n] float32."""
    rng = np.random.default_rng(seed)
    t = np.exp(rng.standard_normal((n_kv, n)) * 1.5)
    for h in range(n_kv):
        t[h, rng.choice(n, n_hot, replace=False)] *= 50.0
    t /= t.max(axis=1, keepdims=True)
    return t.astype(np.float32)
