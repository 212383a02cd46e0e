"""Seeded synthetic inputs for the differential-attention forward.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no scores, no softmax, no lambda). Both the float64 oracle
(through the tests and the benchmark) and the CUDA path are fed from here, so
the two sides see bit-identical inputs.

Shapes follow the exercise specification of the Differential Transformer
attention (paperleet "Differential Transformer Attention", Formula and
conventions): Q1, K1, Q2, K2 are [B, H, T, D]; V is [B, H, T, 2D].  The DIFF
V2 head (aiengineeringfromscratch lesson, "V1 contre V2") keeps the baseline's
head dimension, so its V is [B, H, T, D]: workloads may set the value width.

Recipe (all draws from numpy's PCG64 generator, float32, in this order):
  q1, k1, q2, k2 ~ N(0, 1)      each [B, H, T, D]
  v               ~ N(0, 1)      [B, H, T, Dv]   (Dv = 2D unless stated)
  lq1, lk1, lq2, lk2 ~ N(0, 0.1^2)  each [D]   (the lambda parameter vectors)
  then, per workload:
    planted keys: for each (b, h), 8 distinct key rows j_s ~ U[0, T) and a
      partner query row i_s ~ U[j_s, T); K1[b, h, j_s] = 4 * Q1[b, h, i_s]
      (a causally visible, strongly aligned key in branch 1 only)
    value offset: one vector c ~ N(0, 2^2) of width Dv per (b, h), added to
      every token's value row
The float32 draws are then rounded to the compute dtype (bf16 round to nearest
even, or kept as float32).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic input recipe."""
    name: str
    B: int
    H: int
    T: int
    D: int
    dtype: str               # "bf16" or "f32"
    causal: bool
    seed: int
    layer: Optional[int] = None          # lambda_init from the depth schedule
    lambda_init: Optional[float] = None  # explicit lambda_init
    lambdas: Optional[Sequence[float]] = None  # lambda given directly (swept)
    planted: int = 0                     # planted aligned keys per head
    value_offset_sigma: float = 0.0      # std of the shared per-channel value offset
    kv_heads: Optional[int] = None       # key/value heads (None: H)
    shared_keys: bool = False            # K2 is K1 (one key tensor for both branches)
    value_dim: Optional[int] = None      # V and O width (None: 2D)

    @property
    def Hk(self) -> int:
        return self.H if self.kv_heads is None else self.kv_heads

    @property
    def Dv(self) -> int:
        return 2 * self.D if self.value_dim is None else self.value_dim

    @property
    def pairs_per_head(self) -> int:
        """Unmasked (query, key) pairs of one head."""
        T = self.T
        return T * (T + 1) // 2 if self.causal else T * T

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 2 QK^T (2D each) + 2 PV (2 Dv each) per unmasked
        pair (12 D when Dv = 2D)."""
        return self.B * self.H * self.pairs_per_head * (4 * self.D + 4 * self.Dv)


# The five input recipes.  Sizes, distributions and lambda recipes are the
# ones the workload table fixes; seeds 0..4 in table order.
WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=1, H=2, T=128, D=32, dtype="f32",
                         causal=True, seed=0, layer=1),
    "b4h16t2048": Workload("b4h16t2048", B=4, H=16, T=2048, D=64, dtype="bf16",
                           causal=True, seed=1, layer=12),
    "b2h16t8192": Workload("b2h16t8192", B=2, H=16, T=8192, D=64, dtype="bf16",
                           causal=True, seed=2, layer=24),
    "b1h16t32768_planted": Workload("b1h16t32768_planted", B=1, H=16, T=32768, D=64,
                                    dtype="bf16", causal=True, seed=3,
                                    lambda_init=0.8, planted=8),
    "b8h32t4096_offset": Workload("b8h32t4096_offset", B=8, H=32, T=4096, D=64,
                                  dtype="bf16", causal=False, seed=4,
                                  lambdas=(0.0, 0.5, 1.0), value_offset_sigma=2.0),
}

HEADLINE = "b2h16t8192"

# Grouped key/value heads (the DIFF V2 layout): the headline's 16 differential
# heads over 4 key/value heads, both branches reading one key tensor.  Same
# algorithmic FLOPs as the headline.
GQA_WORKLOADS = {
    "b2h16kv4t8192_shared_k": Workload("b2h16kv4t8192_shared_k", B=2, H=16, T=8192, D=64,
                                       dtype="bf16", causal=True, seed=5, lambda_init=0.8,
                                       kv_heads=4, shared_keys=True),
    # The DIFF V2 head: the baseline's head dimension (128) for Q, K and V, the
    # two branches of a differential head reading one key tensor, 16
    # differential heads (32 query heads) over 8 key/value heads.
    "b2h16kv8t8192_d128_shared_k": Workload("b2h16kv8t8192_d128_shared_k", B=2, H=16, T=8192,
                                            D=128, dtype="bf16", causal=True, seed=6,
                                            lambda_init=0.8, kv_heads=8, shared_keys=True,
                                            value_dim=128),
}
ALL_WORKLOADS = {**WORKLOADS, **GQA_WORKLOADS}


@dataclasses.dataclass
class Inputs:
    """Drawn inputs.  Arrays are float32 holding exactly the values the device
    sees (already rounded to the compute dtype)."""
    q1: np.ndarray
    k1: np.ndarray
    q2: np.ndarray
    k2: np.ndarray
    v: np.ndarray
    lq1: np.ndarray
    lk1: np.ndarray
    lq2: np.ndarray
    lk2: np.ndarray
    planted_keys: Optional[np.ndarray] = None     # [B, H, planted] key rows
    planted_queries: Optional[np.ndarray] = None  # [B, H, planted] query rows
    value_offset: Optional[np.ndarray] = None     # [B, H_kv, Dv]


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bfloat16 (ties to even), returned as float32.

    Pure bit manipulation on the float32 encoding; inputs are finite."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def draw(w: Workload, B: Optional[int] = None, H: Optional[int] = None,
         T: Optional[int] = None, D: Optional[int] = None, seed: Optional[int] = None,
         dtype: Optional[str] = None, kv_heads: Optional[int] = None) -> Inputs:
    """Draw the inputs of workload `w` (optionally overriding its sizes).

    kv_heads: number of key/value heads (default H); K1, K2 and V then have
    that many heads (grouped key/value heads), Q1 and Q2 keep H."""
    B = w.B if B is None else B
    H = w.H if H is None else H
    T = w.T if T is None else T
    D = w.D if D is None else D
    Hk = (w.Hk if H == w.H else H) if kv_heads is None else kv_heads
    if Hk < 1 or H % Hk != 0:
        raise ValueError("kv_heads must divide H")
    if w.planted and Hk != H:
        raise ValueError("planted keys are defined per head; use kv_heads = H")
    dtype = w.dtype if dtype is None else dtype
    rng = np.random.Generator(np.random.PCG64(w.seed if seed is None else seed))
    q1 = rng.standard_normal((B, H, T, D), dtype=np.float32)
    k1 = rng.standard_normal((B, Hk, T, D), dtype=np.float32)
    q2 = rng.standard_normal((B, H, T, D), dtype=np.float32)
    k2 = rng.standard_normal((B, Hk, T, D), dtype=np.float32)
    Dv = 2 * D if w.value_dim is None else w.value_dim
    v = rng.standard_normal((B, Hk, T, Dv), dtype=np.float32)
    lam_vecs = [(0.1 * rng.standard_normal(D)).astype(np.float32) for _ in range(4)]
    planted_keys = planted_queries = offset = None
    if w.planted:
        n = min(w.planted, T)
        planted_keys = np.zeros((B, H, n), dtype=np.int64)
        planted_queries = np.zeros((B, H, n), dtype=np.int64)
        for b in range(B):
            for h in range(H):
                js = rng.choice(T, size=n, replace=False)
                for s, j in enumerate(js):
                    i = int(rng.integers(j, T))
                    planted_keys[b, h, s] = j
                    planted_queries[b, h, s] = i
                    k1[b, h, j] = 4.0 * q1[b, h, i]
    if w.value_offset_sigma:
        offset = (w.value_offset_sigma *
                  rng.standard_normal((B, Hk, Dv), dtype=np.float32)).astype(np.float32)
        v += offset[:, :, None, :]
    if dtype == "bf16":
        q1, k1, q2, k2, v = (round_to_bf16(a) for a in (q1, k1, q2, k2, v))
    elif dtype != "f32":
        raise ValueError(f"unknown dtype {dtype}")
    if w.shared_keys:
        k2 = k1
    return Inputs(q1, k1, q2, k2, v, *lam_vecs, planted_keys=planted_keys,
                  planted_queries=planted_queries, value_offset=offset)


def lambda_init_for(w: Workload) -> float:
    """lambda_init of a workload: explicit, or the depth schedule at its layer
    (0.8 - 0.6 exp(-0.3 (l - 1)), layers counted from 1)."""
    if w.lambda_init is not None:
        return float(w.lambda_init)
    if w.layer is None:
        raise ValueError(f"{w.name}: no lambda_init and no layer")
    return 0.8 - 0.6 * math.exp(-0.3 * (w.layer - 1))


def check_rows(T: int, extra: Sequence[int] = (), n_random: int = 0,
               seed: int = 1234, tile: int = 128) -> np.ndarray:
    """Query rows for sampled parity checks: 0, T-1, both sides of every
    128-row tile boundary, any extra rows, and n_random uniform rows."""
    rows = {0, T - 1}
    for t in range(tile, T, tile):
        rows.add(t - 1)
        rows.add(t)
    rows.update(int(r) for r in extra)
    if n_random:
        rng = np.random.Generator(np.random.PCG64(seed))
        rows.update(int(r) for r in rng.integers(0, T, size=n_random))
    return np.array(sorted(r for r in rows if 0 <= r < T), dtype=np.int64)


@dataclasses.dataclass(frozen=True)
class DecodeWorkload:
    """Tq new queries over a cache of Tk keys (a decode step for small Tq, a
    chunk of a prefill for larger Tq)."""
    name: str
    B: int
    H: int
    Tq: int
    Tk: int
    D: int
    dtype: str
    causal: bool
    seed: int
    lambda_value: float = 0.8
    kv_heads: Optional[int] = None      # key/value heads (None: H)
    value_dim: Optional[int] = None     # V and O width (None: 2D)
    shared_keys: bool = False           # K2 is K1 (one key tensor for both branches)

    @property
    def Dv(self) -> int:
        return 2 * self.D if self.value_dim is None else self.value_dim

    @property
    def Hk(self) -> int:
        return self.H if self.kv_heads is None else self.kv_heads

    @property
    def bytes(self) -> int:
        """Algorithmic HBM bytes: K1, K2 (one tensor when shared), V of every
        key/value head read once; Q1, Q2 read and O written for every query
        head."""
        el = 2 if self.dtype == "bf16" else 4
        k_tensors = 1 if self.shared_keys else 2
        return (self.B * self.Hk * self.Tk * (k_tensors * self.D + self.Dv) +
                self.B * self.H * self.Tq * (2 * self.D + self.Dv)) * el

    @property
    def pairs_per_head(self) -> int:
        """Unmasked (query, key) pairs of one head: query i sees keys
        j <= Tk - Tq + i under the causal mask."""
        if not self.causal:
            return self.Tq * self.Tk
        return self.Tq * (self.Tk - self.Tq) + self.Tq * (self.Tq + 1) // 2

    @property
    def flops(self) -> int:
        """Algorithmic FLOPs: 4 D + 4 Dv per unmasked pair."""
        return self.B * self.H * self.pairs_per_head * (4 * self.D + 4 * self.Dv)


# Decode workloads: 16 sequences with 16 heads (the V1 layout halves the heads
# of a 32-head model), D = 64, an 8192-token cache; one query, and four
# (speculative decoding).
DECODE_WORKLOADS = {
    "decode_b16h16q1k8192": DecodeWorkload("decode_b16h16q1k8192", 16, 16, 1, 8192, 64, "bf16", True, 20),
    "decode_b16h16q4k8192": DecodeWorkload("decode_b16h16q4k8192", 16, 16, 4, 8192, 64, "bf16", True, 21),
    # grouped key/value heads: 32 differential heads over 8 key/value heads
    # (the 32-query / 8-key-value-head grouping of the GQA exercise)
    "decode_b16h32kv8q1k8192": DecodeWorkload("decode_b16h32kv8q1k8192", 16, 32, 1, 8192, 64,
                                              "bf16", True, 22, kv_heads=8),
    # the same grouping with four speculative tokens: 16 query rows per
    # key/value head
    "decode_b16h32kv8q4k8192": DecodeWorkload("decode_b16h32kv8q4k8192", 16, 32, 4, 8192, 64,
                                              "bf16", True, 26, kv_heads=8),
    # the DIFF V2 head: 16 differential heads over 8 key/value heads, D = Dv =
    # 128, one key tensor for both branches
    "decode_b16h16kv8q1k8192_d128_shared_k": DecodeWorkload(
        "decode_b16h16kv8q1k8192_d128_shared_k", 16, 16, 1, 8192, 128, "bf16", True, 25,
        kv_heads=8, value_dim=128, shared_keys=True),
}

# Chunked prefill: the next 1024 tokens of 4 sequences (16 heads, D = 64)
# against their cache of 8192 keys (the chunk's own keys at its end), and the
# same with the DIFF V2 head (D = Dv = 128, 16 differential heads over 8
# key/value heads, shared keys).  Compute-bound: timed in TFLOP/s.
PREFILL_WORKLOADS = {
    "prefill_b4h16q1024k8192": DecodeWorkload("prefill_b4h16q1024k8192", 4, 16, 1024, 8192, 64,
                                              "bf16", True, 23),
    "prefill_b4h16kv8q1024k8192_d128_shared_k": DecodeWorkload(
        "prefill_b4h16kv8q1024k8192_d128_shared_k", 4, 16, 1024, 8192, 128, "bf16", True, 24,
        kv_heads=8, value_dim=128, shared_keys=True),
}


def draw_kv(w: DecodeWorkload, **override) -> Inputs:
    """Decode inputs: q1, q2 [B, H, Tq, D]; k1, k2 [B, H_kv, Tk, D]; v [B, H_kv,
    Tk, Dv] (H_kv = w.kv_heads, default H; Dv = w.Dv); i.i.d. N(0, 1) float32
    drawn in the order q1, k1, q2, k2, v from PCG64(seed), rounded to the
    dtype.  The lambda vectors are left zero (lambda is given directly for
    decode workloads)."""
    f = dict(B=w.B, H=w.H, Tq=w.Tq, Tk=w.Tk, D=w.D, dtype=w.dtype, seed=w.seed,
             kv_heads=w.kv_heads, value_dim=w.value_dim)
    f.update(override)
    rng = np.random.Generator(np.random.PCG64(f["seed"]))
    B, H, Tq, Tk, D = f["B"], f["H"], f["Tq"], f["Tk"], f["D"]
    Hk = H if f["kv_heads"] is None else f["kv_heads"]
    if Hk < 1 or H % Hk != 0:
        raise ValueError("kv_heads must divide H")
    q1 = rng.standard_normal((B, H, Tq, D), dtype=np.float32)
    k1 = rng.standard_normal((B, Hk, Tk, D), dtype=np.float32)
    q2 = rng.standard_normal((B, H, Tq, D), dtype=np.float32)
    k2 = rng.standard_normal((B, Hk, Tk, D), dtype=np.float32)
    Dv = 2 * D if f["value_dim"] is None else f["value_dim"]
    v = rng.standard_normal((B, Hk, Tk, Dv), dtype=np.float32)
    if f["dtype"] == "bf16":
        q1, k1, q2, k2, v = (round_to_bf16(a) for a in (q1, k1, q2, k2, v))
    z = np.zeros(D, dtype=np.float32)
    return Inputs(q1, k1, q2, k2, v, z, z, z, z)
