"""Float64 CPU oracle for the Differential Transformer attention forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  The product path (the C-ABI library
and its Python binding) never imports, calls or links it, and shares no code
with it.

What it computes (plain definition, written out; no blocking beyond a loop over
query rows, no fusion, no reordering):

  S_b   = Q_b K_b^T / sqrt(D) + M                       b = 1, 2
  A_b   = softmax over keys of S_b (max-subtracted, two passes)
  O     = (A_1 - lambda A_2) V
  lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init

Sources:
  * paperleet "Differential Transformer Attention" -- Formula and conventions:
    the two masked maps, the signed combination, the [B,H,T,D] / [B,H,T,2D]
    shapes, the scale 1/sqrt(D) with D the Q/K width, the causal mask (0 on
    allowed positions, -inf on future ones, applied to both branches), and the
    lambda parameterisation.  Per-head normalisation and its fixed multiplier
    are outside this operation and are not applied.
  * aifetchly "Differential Transformer: Canceling LLM Attention Noise" --
    section 1 (the DiffAttn formula), section 3 (the lambda re-parameterisation
    and the lambda_init depth schedule), and the numerically stable softmax
    (subtract the row maximum before exponentiating).
  * ultralytics glossary "Differential Transformer" -- "So funktioniert
    differentielle Aufmerksamkeit": each map sums to 1 per row, so the signed
    map's rows sum to 1 - lambda and can hold negative entries.

Readings where the pages leave a step open:
  * A masked position contributes exactly zero weight (exp(-inf) = 0); with
    the causal mask, key j is visible to query i iff j <= i, so no row is
    ever fully masked.
  * lambda is any finite real (not clamped to [0, 1]).
  * The value width Dv is 2D in the operation's own shape (paperleet, Formula
    and conventions).  The DIFF V2 head of the aiengineeringfromscratch lesson
    ("V1 contre V2": the head dimension stays that of the baseline) has V as
    wide as Q and K, Dv = D.  O = (A_1 - lambda A_2) V holds for any V width,
    so every function here takes V of any width Dv >= 1 and returns O of that
    width.

The step that follows the operation in the model (per-head normalisation,
GroupNorm or RMSNorm, then x (1 - lambda_init)) is `head_norm`, pinned
against torch's group_norm and rms_norm.

The backward (`differential_attention_backward`, `differential_lambda_backward`)
is the chain rule through the same steps (paperleet, Return requirements:
gradients through both Q/K branches, the value, the coefficient and the four
lambda vectors), pinned against torch autograd, finite differences and closed
forms in tests/test_oracle_backward.py.

Parity is pinned by tests/test_oracle.py (brute-force scalar softmax on tiny
inputs, a library attention routine at lambda = 0, row sums, the identical-map
and value-offset identities, closed forms, and the printed worked example).
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "lambda_init_schedule",
    "differential_lambda",
    "softmax_maps",
    "signed_map",
    "differential_attention",
    "head_norm",
    "differential_attention_kv",
]


def lambda_init_schedule(layer: int) -> float:
    """lambda_init = 0.8 - 0.6 exp(-0.3 (l - 1)) for layer l >= 1
    (aifetchly, section 3; paperleet, Formula and conventions)."""
    if layer < 1:
        raise ValueError("layers are counted from 1")
    return 0.8 - 0.6 * math.exp(-0.3 * (layer - 1))


def differential_lambda(lq1, lk1, lq2, lk2, lambda_init: float = 0.2) -> float:
    """lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init, in float64
    (aifetchly, section 3; paperleet, Formula and conventions: equal-length,
    non-empty vectors, the result is not restricted to [0, 1])."""
    vecs = [np.asarray(x, dtype=np.float64).reshape(-1) for x in (lq1, lk1, lq2, lk2)]
    n = vecs[0].size
    if n == 0 or any(x.size != n for x in vecs):
        raise ValueError("lambda vectors must be non-empty and of equal length")
    dot1 = float(np.dot(vecs[0], vecs[1]))
    dot2 = float(np.dot(vecs[2], vecs[3]))
    return math.exp(dot1) - math.exp(dot2) + float(lambda_init)


# ---------------------------------------------------------------------------
# The steps of one head, on float64 arrays.  Kept separate so that each can be
# read against the formula on its own.
# ---------------------------------------------------------------------------

def _scores(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """S = Q K^T / sqrt(D) for query rows q [R, D] and all keys k [T, D]."""
    D = q.shape[-1]
    return (q @ k.T) / math.sqrt(D)


def _mask(s: np.ndarray, rows: np.ndarray, causal: bool, offset: int = 0) -> np.ndarray:
    """Add M: -inf where key j > query i + offset (causal), nothing otherwise.
    offset = Tk - Tq places the queries at the end of the key sequence (a KV
    cache); it is 0 when queries and keys are the same sequence."""
    if not causal:
        return s
    keys = np.arange(s.shape[-1])
    future = keys[None, :] > rows[:, None] + offset
    out = s.copy()
    out[future] = -np.inf
    return out


def _softmax(s: np.ndarray) -> np.ndarray:
    """Row softmax over keys: subtract the row max, exponentiate, divide by the
    row sum (two passes).  exp(-inf) is exactly 0."""
    m = np.max(s, axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=-1, keepdims=True)


def _combine(a1: np.ndarray, a2: np.ndarray, lam: float) -> np.ndarray:
    """The signed map A_1 - lambda A_2."""
    return a1 - lam * a2


def _head_rows(q1, k1, q2, k2, rows, lam, causal, offset=0):
    """Signed-map rows of one head for the given query rows."""
    a1 = _softmax(_mask(_scores(q1[rows], k1), rows, causal, offset))
    a2 = _softmax(_mask(_scores(q2[rows], k2), rows, causal, offset))
    return _combine(a1, a2, lam)


def _as64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _check_shapes(q1, k1, q2, k2, v=None):
    """Q1, Q2: [B, H, T, D]; K1, K2: [B, H_kv, T, D]; V: [B, H_kv, T, Dv] (Dv =
    2D for the operation's own shape, Dv = D for the DIFF V2 head) with H a
    multiple of H_kv (query heads share key/value heads in groups of H / H_kv,
    the grouped layout of DIFF V2; H_kv = H is the plain layout).  Returns the
    group size H / H_kv."""
    if q1.shape != q2.shape or k1.shape != k2.shape:
        raise ValueError("Q1, Q2 must share one shape, and K1, K2 another")
    if q1.ndim != 4 or k1.ndim != 4 or min(q1.shape) < 1 or min(k1.shape) < 1:
        raise ValueError("expected non-empty [B, H, T, D] tensors")
    B, H, T, D = q1.shape
    Hk = k1.shape[1]
    if k1.shape[0] != B or k1.shape[2:] != (T, D) or H % Hk != 0:
        raise ValueError("K1/K2 must be [B, H_kv, T, D] with H a multiple of H_kv")
    if v is not None and (v.ndim != 4 or v.shape[:3] != (B, Hk, T) or v.shape[3] < 1):
        raise ValueError("V must be [B, H_kv, T, Dv] with Dv >= 1")
    return H // Hk


def softmax_maps(q1, k1, q2, k2, causal: bool = True):
    """The two attention maps A_1, A_2 as [B, H, T, T] float64 (small inputs)."""
    q1, k1, q2, k2 = (_as64(x) for x in (q1, k1, q2, k2))
    g = _check_shapes(q1, k1, q2, k2)
    B, H, T, _ = q1.shape
    rows = np.arange(T)
    a1 = np.empty((B, H, T, T))
    a2 = np.empty((B, H, T, T))
    for b in range(B):
        for h in range(H):
            a1[b, h] = _softmax(_mask(_scores(q1[b, h], k1[b, h // g]), rows, causal))
            a2[b, h] = _softmax(_mask(_scores(q2[b, h], k2[b, h // g]), rows, causal))
    return a1, a2


def signed_map(q1, k1, q2, k2, lam: float, causal: bool = True) -> np.ndarray:
    """The signed map A_1 - lambda A_2 as [B, H, T, T] float64 (small inputs)."""
    a1, a2 = softmax_maps(q1, k1, q2, k2, causal)
    return _combine(a1, a2, float(lam))


def differential_attention(q1, k1, q2, k2, v, lam: float, causal: bool = True,
                           rows: Optional[Sequence[int]] = None,
                           heads: Optional[Sequence[tuple]] = None,
                           block: int = 256) -> np.ndarray:
    """O = (A_1 - lambda A_2) V in float64.

    q1, q2: [B, H, T, D]; k1, k2: [B, H_kv, T, D]; v: [B, H_kv, T, Dv] (any
    real dtype, upcast to float64; Dv = 2D in the operation's own shape), H a
    multiple of H_kv: query head h uses key/value head h // (H / H_kv).  lam:
    the scalar lambda.  causal: apply the causal mask to both branches.

    rows: optional query rows to evaluate (every row when None).  Every output
    row depends only on its own query row and all keys/values of its head, so
    a row subset is exact, not an approximation.
    heads: optional list of (b, h) to evaluate (every head when None).

    Returns [B, H, R, Dv] for all heads, or [len(heads), R, Dv] when heads is
    given.  Query rows are processed `block` at a time only to bound memory.
    """
    g = _check_shapes(q1, k1, q2, k2, v)
    B, H, T, D = q1.shape
    Dv = v.shape[3]
    lam = float(lam)
    row_idx = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    if row_idx.size and (row_idx.min() < 0 or row_idx.max() >= T):
        raise ValueError("row index out of range")
    head_list = [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)
    out = np.empty((len(head_list), row_idx.size, Dv))
    for n, (b, h) in enumerate(head_list):
        hq1, hq2 = _as64(q1[b, h]), _as64(q2[b, h])
        hk1, hk2, hv = (_as64(x[b, h // g]) for x in (k1, k2, v))
        for r0 in range(0, row_idx.size, block):
            r = row_idx[r0:r0 + block]
            out[n, r0:r0 + block] = _head_rows(hq1, hk1, hq2, hk2, r, lam, causal) @ hv
    if heads is None:
        out = out.reshape(B, H, row_idx.size, Dv)
    return out


# ---------------------------------------------------------------------------
# Per-head output normalisation and the fixed multiplier (the step after the
# operation: aifetchly section 4 and the ultralytics glossary describe a
# per-head GroupNorm followed by x (1 - lambda_init); the aiengineeringfromscratch
# lesson describes the per-head normalisation of DIFF V1 as an RMSNorm).
# ---------------------------------------------------------------------------

def head_norm(o, kind: str, eps: float = 1e-5, weight=None, bias=None,
              out_scale: float = 1.0) -> np.ndarray:
    """Y = out_scale * (norm(O) * weight + bias), per (b, h, t) over the head's
    2D output channels, in float64.

    kind "rms":   norm(x) = x / sqrt(mean(x^2) + eps)
    kind "group": norm(x) = (x - mean(x)) / sqrt(var(x) + eps), var the mean
                  squared deviation (one group per head, as GroupNorm with
                  num_groups = H over the H * 2D channels of a token)
    kind "none":  norm(x) = x
    weight, bias: optional [H, 2D] per-channel affine parameters.
    """
    o = np.asarray(o, dtype=np.float64)
    if kind == "rms":
        y = o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    elif kind == "group":
        mu = np.mean(o, axis=-1, keepdims=True)
        var = np.mean((o - mu) ** 2, axis=-1, keepdims=True)
        y = (o - mu) / np.sqrt(var + eps)
    elif kind == "none":
        y = o.copy()
    else:
        raise ValueError(f"unknown norm {kind!r}")
    H = o.shape[1]
    if weight is not None:
        y = y * np.asarray(weight, dtype=np.float64).reshape(1, H, 1, -1)
    if bias is not None:
        y = y + np.asarray(bias, dtype=np.float64).reshape(1, H, 1, -1)
    return out_scale * y


def differential_attention_kv(q1, k1, q2, k2, v, lam: float, causal: bool = True) -> np.ndarray:
    """O = (A_1 - lambda A_2) V for Tq queries against Tk >= Tq keys (decode
    over a KV cache), in float64.

    q1, q2: [B, H, Tq, D]; k1, k2: [B, H_kv, Tk, D]; v: [B, H_kv, Tk, Dv], H a
    multiple of H_kv (query head h reads key/value head h // (H / H_kv)).  With
    the causal mask, query i sits at position Tk - Tq + i of the key sequence and
    sees keys j <= Tk - Tq + i (the usual KV-cache alignment; for Tq = Tk it is
    the causal mask of differential_attention).  Returns [B, H, Tq, Dv].
    """
    q1, k1, q2, k2, v = (_as64(x) for x in (q1, k1, q2, k2, v))
    if q1.shape != q2.shape or k1.shape != k2.shape or q1.ndim != 4 or k1.ndim != 4:
        raise ValueError("Q1/Q2 must be [B, H, Tq, D] and K1/K2 [B, H_kv, Tk, D]")
    B, H, Tq, D = q1.shape
    Hk, Tk = k1.shape[1], k1.shape[2]
    if (k1.shape[0] != B or Hk < 1 or H % Hk != 0 or k1.shape[3] != D
            or v.ndim != 4 or v.shape[:3] != (B, Hk, Tk) or v.shape[3] < 1):
        raise ValueError("inconsistent shapes")
    g = H // Hk
    if min(B, H, Tq, D, Tk) < 1 or (causal and Tk < Tq):
        raise ValueError("need non-empty tensors and Tk >= Tq for the causal mask")
    rows = np.arange(Tq)
    out = np.empty((B, H, Tq, v.shape[3]))
    for b in range(B):
        for h in range(H):
            w = _head_rows(q1[b, h], k1[b, h // g], q2[b, h], k2[b, h // g], rows, float(lam),
                           causal, Tk - Tq)
            out[b, h] = w @ v[b, h // g]
    return out


# ---------------------------------------------------------------------------
# Backward: the vector-Jacobian product of the operation.  paperleet
# "Differential Transformer Attention", Return requirements: gradients flow
# through both Q/K branches, the value and a tensor coefficient, and
# differential_lambda passes gradients to all four parameter vectors; its Toy
# experiment section checks all of them with analytic vector-Jacobian products.
# The steps below are the chain rule through the forward's own steps, for one
# head, given dO = dL/dO:
#
#   W      = A_1 - lambda A_2                     (the signed map)
#   dV     = W^T dO                               (O = W V)
#   dW     = dO V^T
#   dA_1   = dW,   dA_2 = -lambda dW,   dlambda = -sum(dW * A_2)
#   dS_b   = A_b * (dA_b - rowsum(dA_b * A_b))    (row softmax; masked entries
#                                                  have A_b = 0, so dS_b = 0)
#   dQ_b   = dS_b K_b / sqrt(D),   dK_b = dS_b^T Q_b / sqrt(D)
#
# With grouped key/value heads, dK_b and dV of a key/value head sum the
# contributions of every query head that reads it.
# ---------------------------------------------------------------------------

def _head_backward(q1, k1, q2, k2, v, dout, lam, causal, block=256):
    """Gradients of one query head (float64 arrays of that head) for all rows:
    returns dq1, dk1, dq2, dk2, dv, dlam.  Query rows go `block` at a time;
    each row's softmax is complete within its block, so blocking is exact."""
    T, D = q1.shape
    scale = 1.0 / math.sqrt(D)
    dq1, dq2 = np.zeros_like(q1), np.zeros_like(q2)
    dk1, dk2 = np.zeros_like(k1), np.zeros_like(k2)
    dv = np.zeros_like(v)
    dlam = 0.0
    for r0 in range(0, T, block):
        rows = np.arange(r0, min(T, r0 + block))
        a1 = _softmax(_mask(_scores(q1[rows], k1), rows, causal))
        a2 = _softmax(_mask(_scores(q2[rows], k2), rows, causal))
        w = _combine(a1, a2, lam)
        g = dout[rows]
        dv += w.T @ g
        dw = g @ v.T
        dlam += -float(np.sum(dw * a2))
        for a, da, q, k, dq, dk in ((a1, dw, q1, k1, dq1, dk1),
                                    (a2, -lam * dw, q2, k2, dq2, dk2)):
            ds = a * (da - np.sum(da * a, axis=-1, keepdims=True))
            dq[rows] = scale * (ds @ k)
            dk += scale * (ds.T @ q[rows])
    return dq1, dk1, dq2, dk2, dv, dlam


def differential_attention_backward(q1, k1, q2, k2, v, lam: float, dout, causal: bool = True,
                                    kv_heads: Optional[Sequence[tuple]] = None):
    """Gradients of L with dL/dO = dout through O = (A_1 - lambda A_2) V, in
    float64.

    Shapes as differential_attention (q1, q2 [B, H, T, D]; k1, k2 [B, H_kv, T,
    D]; v [B, H_kv, T, Dv], Dv = 2D in the operation's own shape); dout [B, H,
    T, Dv].  Returns dq1, dk1, dq2, dk2, dv with the shapes of their inputs, and
    dlambda (a float).

    kv_heads: optional list of (b, hk) key/value heads to evaluate; then every
    query head that reads them is processed, the gradients of the other heads
    are left zero, and dlambda sums only the processed query heads.
    """
    g = _check_shapes(q1, k1, q2, k2, v)
    B, H, T, D = q1.shape
    Hk = H // g
    dout = _as64(dout)
    Dv = v.shape[3]
    if dout.shape != (B, H, T, Dv):
        raise ValueError("dout must be [B, H, T, Dv], Dv the width of V")
    lam = float(lam)
    dq1 = np.zeros((B, H, T, D))
    dq2 = np.zeros((B, H, T, D))
    dk1 = np.zeros((B, Hk, T, D))
    dk2 = np.zeros((B, Hk, T, D))
    dv = np.zeros((B, Hk, T, Dv))
    dlam = 0.0
    todo = [(b, hk) for b in range(B) for hk in range(Hk)] if kv_heads is None else list(kv_heads)
    for b, hk in todo:
        hk1, hk2, hv = (_as64(x[b, hk]) for x in (k1, k2, v))
        for h in range(hk * g, (hk + 1) * g):
            r = _head_backward(_as64(q1[b, h]), hk1, _as64(q2[b, h]), hk2, hv, dout[b, h], lam,
                               causal)
            dq1[b, h], dq2[b, h] = r[0], r[2]
            dk1[b, hk] += r[1]
            dk2[b, hk] += r[3]
            dv[b, hk] += r[4]
            dlam += r[5]
    return dq1, dk1, dq2, dk2, dv, dlam


def differential_lambda_backward(lq1, lk1, lq2, lk2, dlam: float):
    """Gradients of lambda = exp(lq1 . lk1) - exp(lq2 . lk2) + lambda_init with
    respect to the four vectors, given dL/dlambda (float64):
    d/dlq1 = dlam e1 lk1, d/dlk1 = dlam e1 lq1, d/dlq2 = -dlam e2 lk2,
    d/dlk2 = -dlam e2 lq2, with e_b = exp(lq_b . lk_b)."""
    vecs = [np.asarray(x, dtype=np.float64).reshape(-1) for x in (lq1, lk1, lq2, lk2)]
    e1 = math.exp(float(np.dot(vecs[0], vecs[1])))
    e2 = math.exp(float(np.dot(vecs[2], vecs[3])))
    d = float(dlam)
    return d * e1 * vecs[1], d * e1 * vecs[0], -d * e2 * vecs[3], -d * e2 * vecs[2]


def branch_logsumexp(q, k, causal: bool = True) -> np.ndarray:
    """log sum_j exp(S_ij) per query row of one branch, S = Q K^T / sqrt(D) + M
    (natural log, float64): the normaliser of the row softmax of the
    Formula-and-conventions maps, which the backward reuses.

    q: [B, H, T, D]; k: [B, H_kv, T, D].  Returns [B, H, T]."""
    q, k = _as64(q), _as64(k)
    B, H, T, D = q.shape
    g = H // k.shape[1]
    out = np.empty((B, H, T))
    rows = np.arange(T)
    for b in range(B):
        for h in range(H):
            s = _mask(_scores(q[b, h], k[b, h // g]), rows, causal)
            m = np.max(s, axis=-1)
            out[b, h] = m + np.log(np.sum(np.exp(s - m[:, None]), axis=-1))
    return out
