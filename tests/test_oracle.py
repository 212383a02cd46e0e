"""Pins for the float64 oracle, independent of the oracle's own code.

Each pin checks the oracle against something the pages or the mathematics fix:
  * a brute-force scalar softmax written with plain Python loops (the
    "independent scalar softmax" the paperleet exercise names for verification);
  * torch's scaled_dot_product_attention at lambda = 0 (paperleet, Formula and
    conventions: "At lambda=0 it becomes ordinary attention");
  * row sums 1 - lambda (paperleet; ultralytics "So funktioniert ...");
  * identical maps cancel exactly at lambda = 1 (paperleet);
  * a value offset shared by every token responds by exactly (1 - lambda)
    (paperleet, Toy experiment);
  * closed forms on two-token inputs and for the causal first row;
  * the worked example printed on the ultralytics page (row sum 0.20, 13 of 36
    negative weights);
  * lambda: zero vectors give lambda_init (aifetchly, section 3), the depth
    schedule gives 0.2 at layer 1.
The mutation tests at the end plant a plausible mistake in one oracle step and
check that some pin fails.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import diffattn_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_inputs(B, H, T, D, seed):
    rng = np.random.default_rng(seed)
    q1, k1, q2, k2 = (rng.standard_normal((B, H, T, D)) for _ in range(4))
    v = rng.standard_normal((B, H, T, 2 * D))
    return q1, k1, q2, k2, v


def brute_force(q1, k1, q2, k2, v, lam, causal):
    """Per-element scalar evaluation with Python floats and math.exp."""
    B, H, T, D = q1.shape
    Dv = v.shape[-1]
    out = np.zeros((B, H, T, Dv))
    for b in range(B):
        for h in range(H):
            for i in range(T):
                weights = [0.0] * T
                for q, k, sign in ((q1, k1, 1.0), (q2, k2, -lam)):
                    visible = [j for j in range(T) if (not causal) or j <= i]
                    logits = {}
                    for j in visible:
                        dot = 0.0
                        for c in range(D):
                            dot += float(q[b, h, i, c]) * float(k[b, h, j, c])
                        logits[j] = dot / math.sqrt(D)
                    top = max(logits.values())
                    ex = {j: math.exp(x - top) for j, x in logits.items()}
                    z = sum(ex.values())
                    for j in visible:
                        weights[j] += sign * ex[j] / z
                for c in range(Dv):
                    acc = 0.0
                    for j in range(T):
                        acc += weights[j] * float(v[b, h, j, c])
                    out[b, h, i, c] = acc
    return out


# ---------------------------------------------------------------------------
# Pins (plain functions so the mutation tests can rerun them)
# ---------------------------------------------------------------------------

def pin_brute_force():
    for (B, H, T, D, seed) in [(1, 2, 5, 3, 0), (2, 1, 8, 4, 1), (1, 1, 1, 2, 2), (1, 1, 7, 6, 3)]:
        q1, k1, q2, k2, v = rand_inputs(B, H, T, D, seed)
        for lam in (0.0, 0.2, 0.8, 1.0, -0.35, 1.7):
            for causal in (True, False):
                got = oracle.differential_attention(q1, k1, q2, k2, v, lam, causal)
                ref = brute_force(q1, k1, q2, k2, v, lam, causal)
                assert np.max(np.abs(got - ref)) <= 1e-12, (B, H, T, D, lam, causal)


def pin_sdpa_lambda0():
    for causal in (True, False):
        q1, k1, q2, k2, v = rand_inputs(2, 3, 37, 16, 7)
        got = oracle.differential_attention(q1, k1, q2, k2, v, 0.0, causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q1), torch.from_numpy(k1), torch.from_numpy(v),
            is_causal=causal).numpy()
        assert np.max(np.abs(got - ref)) <= 1e-12


def pin_row_sums():
    q1, k1, q2, k2, _ = rand_inputs(1, 2, 33, 8, 11)
    for lam in (0.0, 0.5, 0.8, 1.3, -2.0):
        for causal in (True, False):
            m = oracle.signed_map(q1, k1, q2, k2, lam, causal)
            assert np.max(np.abs(m.sum(-1) - (1.0 - lam))) <= 1e-12
            ones = np.ones((1, 2, 33, 16))
            o = oracle.differential_attention(q1, k1, q2, k2, ones, lam, causal)
            assert np.max(np.abs(o - (1.0 - lam))) <= 1e-12


def pin_identical_maps():
    q1, k1, _, _, v = rand_inputs(1, 2, 29, 8, 12)
    for causal in (True, False):
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q1), torch.from_numpy(k1), torch.from_numpy(v),
            is_causal=causal).numpy()
        for lam in (0.0, 0.3, 0.8):
            got = oracle.differential_attention(q1, k1, q1, k1, v, lam, causal)
            assert np.max(np.abs(got - (1.0 - lam) * ref)) <= 1e-12
        got1 = oracle.differential_attention(q1, k1, q1, k1, v, 1.0, causal)
        assert np.all(got1 == 0.0)


def pin_value_offset():
    q1, k1, q2, k2, v = rand_inputs(2, 2, 24, 8, 13)
    c = np.random.default_rng(5).normal(0.0, 2.0, size=(2, 2, 1, 16))
    for lam in (0.0, 0.25, 0.5, 1.0, 1.5):
        for causal in (True, False):
            base = oracle.differential_attention(q1, k1, q2, k2, v, lam, causal)
            shifted = oracle.differential_attention(q1, k1, q2, k2, v + c, lam, causal)
            assert np.max(np.abs((shifted - base) - (1.0 - lam) * c)) <= 1e-12


def pin_closed_forms():
    # Two tokens, D = 4 (scale 1/2).  Branch 1: q = (a,0,0,0), k0 = (b,0,0,0),
    # k1 = 0, so w0 = sigmoid(a b / 2).  Branch 2: q = 0, uniform weights 1/2.
    a, b, lam = 1.3, -0.7, 0.6
    q1 = np.zeros((1, 1, 2, 4)); q1[0, 0, :, 0] = a
    k1 = np.zeros((1, 1, 2, 4)); k1[0, 0, 0, 0] = b
    q2 = np.zeros((1, 1, 2, 4)); k2 = np.random.default_rng(0).standard_normal((1, 1, 2, 4))
    v = np.random.default_rng(1).standard_normal((1, 1, 2, 8))
    w0 = 1.0 / (1.0 + math.exp(-a * b / 2.0))
    expect_last = (w0 - lam / 2) * v[0, 0, 0] + ((1 - w0) - lam / 2) * v[0, 0, 1]
    got = oracle.differential_attention(q1, k1, q2, k2, v, lam, causal=False)
    assert np.max(np.abs(got[0, 0, 1] - expect_last)) <= 1e-14
    assert np.max(np.abs(got[0, 0, 0] - expect_last)) <= 1e-14  # same query, same keys
    got_c = oracle.differential_attention(q1, k1, q2, k2, v, lam, causal=True)
    # Causal first row sees only key 0 in both branches: (1 - lambda) v0.
    assert np.max(np.abs(got_c[0, 0, 0] - (1 - lam) * v[0, 0, 0])) <= 1e-15
    assert np.max(np.abs(got_c[0, 0, 1] - expect_last)) <= 1e-14
    # Causal row 0 on random data: (1 - lambda) v0 for every head.
    q1, k1, q2, k2, v = rand_inputs(2, 3, 17, 5, 21)
    o = oracle.differential_attention(q1, k1, q2, k2, v, 0.37, True)
    assert np.max(np.abs(o[:, :, 0] - 0.63 * v[:, :, 0])) <= 1e-15
    # The last causal row sees every key: equal to the non-causal last row.
    onc = oracle.differential_attention(q1, k1, q2, k2, v, 0.37, False)
    assert np.max(np.abs(o[:, :, -1] - onc[:, :, -1])) <= 1e-13


def pin_worked_example():
    with open(os.path.join(GOLDEN, "p4_worked_example.json")) as f:
        g = json.load(f)
    torch.manual_seed(0)
    n, d, lam = g["n"], g["d"], g["lambda"]
    q1, k1, q2, k2 = torch.randn(4, n, d).double()
    m = oracle.signed_map(*(x.numpy()[None, None] for x in (q1, k1, q2, k2)), lam, causal=False)
    assert f"{m[0, 0, 0].sum():.2f}" == g["printed_row_sum"]
    assert int((m < 0).sum()) == g["printed_negative_weights"]
    assert m[0, 0].size == g["printed_total_weights"]


def pin_lambda():
    z = np.zeros(16)
    assert oracle.differential_lambda(z, z, z, z, 0.37) == 0.37
    assert oracle.lambda_init_schedule(1) == pytest.approx(0.2, abs=1e-15)
    assert oracle.lambda_init_schedule(12) == pytest.approx(0.8 - 0.6 * math.exp(-3.3), abs=1e-15)
    e = np.zeros(4); e[0] = 1.0
    two = np.zeros(4); two[0] = 2.0
    # exp(1*2) - exp(0) + 0.2
    assert oracle.differential_lambda(e, two, z[:4], z[:4], 0.2) == pytest.approx(math.exp(2) - 1 + 0.2, abs=1e-13)
    # exp(0) - exp(1*2) + 0.2  (second term subtracts; negative result allowed)
    assert oracle.differential_lambda(z[:4], z[:4], e, two, 0.2) == pytest.approx(1 - math.exp(2) + 0.2, abs=1e-13)
    # Dot product, not elementwise mismatch: (1,2).(3,4) = 11 -> exp(11)
    assert oracle.differential_lambda([1, 2], [3, 4], [0, 0], [0, 0], 0.0) == pytest.approx(math.exp(11) - 1, rel=1e-14)
    with pytest.raises(ValueError):
        oracle.differential_lambda([], [], [], [])
    with pytest.raises(ValueError):
        oracle.differential_lambda([1, 2], [1], [1, 2], [1, 2])


def pin_kv_decode():
    test_kv_decode_brute_force()


ALL_PINS = [pin_brute_force, pin_sdpa_lambda0, pin_row_sums, pin_identical_maps,
            pin_value_offset, pin_closed_forms, pin_worked_example, pin_kv_decode]


@pytest.mark.parametrize("pin", ALL_PINS + [pin_lambda], ids=lambda f: f.__name__)
def test_pin(pin):
    pin()


def test_row_subset_is_exact():
    q1, k1, q2, k2, v = rand_inputs(2, 2, 300, 8, 31)
    full = oracle.differential_attention(q1, k1, q2, k2, v, 0.7, True)
    rows = [0, 5, 127, 128, 255, 256, 299]
    sub = oracle.differential_attention(q1, k1, q2, k2, v, 0.7, True, rows=rows)
    assert np.array_equal(sub, full[:, :, rows])
    one = oracle.differential_attention(q1, k1, q2, k2, v, 0.7, True, rows=rows, heads=[(1, 0)])
    assert np.array_equal(one[0], full[1, 0, rows])


def test_block_size_does_not_matter():
    q1, k1, q2, k2, v = rand_inputs(1, 1, 70, 8, 32)
    a = oracle.differential_attention(q1, k1, q2, k2, v, 0.7, True, block=256)
    b = oracle.differential_attention(q1, k1, q2, k2, v, 0.7, True, block=7)
    assert np.array_equal(a, b)


def test_noncausal_key_permutation_invariance():
    q1, k1, q2, k2, v = rand_inputs(1, 2, 19, 8, 33)
    perm = np.random.default_rng(3).permutation(19)
    a = oracle.differential_attention(q1, k1, q2, k2, v, 0.8, False)
    b = oracle.differential_attention(q1, k1[:, :, perm], q2, k2[:, :, perm], v[:, :, perm], 0.8, False)
    assert np.max(np.abs(a - b)) <= 1e-12


def test_shape_validation():
    q1, k1, q2, k2, v = rand_inputs(1, 1, 4, 4, 0)
    with pytest.raises(ValueError):
        oracle.differential_attention(q1, k1, q2, k2, v[..., :0], 0.5)
    with pytest.raises(ValueError):
        oracle.differential_attention(q1, k1, q2, k2, v[:, :, :3], 0.5)
    with pytest.raises(ValueError):
        oracle.differential_attention(q1, k1[:, :, :3], q2, k2, v, 0.5)
    with pytest.raises(ValueError):
        oracle.differential_attention_kv(q1, k1, q2, k2, v[:, :, :3], 0.5)


# ---------------------------------------------------------------------------
# The DIFF V2 head (aiengineeringfromscratch lesson, "V1 contre V2": the head
# dimension stays that of the baseline): V as wide as Q and K, Dv = D, with
# the two branches sharing a key/value head.
# ---------------------------------------------------------------------------

def test_value_width_d_lambda0_matches_torch_gqa():
    # lambda = 0 is ordinary attention (paperleet, Formula and conventions);
    # torch's attention routine takes a value width of its own and grouped heads
    rng = np.random.default_rng(70)
    q1, q2 = rng.standard_normal((2, 2, 6, 33, 16))
    k1, k2 = rng.standard_normal((2, 2, 3, 33, 16))
    for dv in (16, 5, 40):
        v = rng.standard_normal((2, 3, 33, dv))
        for causal in (True, False):
            got = oracle.differential_attention(q1, k1, q2, k2, v, 0.0, causal)
            assert got.shape == (2, 6, 33, dv)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q1), torch.from_numpy(k1), torch.from_numpy(v), is_causal=causal,
                enable_gqa=True).numpy()
            assert np.max(np.abs(got - ref)) <= 1e-12


def test_value_width_d_brute_force_and_identities():
    rng = np.random.default_rng(71)
    q1, k1, q2, k2 = rng.standard_normal((4, 1, 2, 7, 4))
    v = rng.standard_normal((1, 2, 7, 4))          # Dv = D
    for lam in (0.0, 0.8, -0.35, 1.7):
        for causal in (True, False):
            got = oracle.differential_attention(q1, k1, q2, k2, v, lam, causal)
            ref = brute_force(q1, k1, q2, k2, v, lam, causal)
            assert np.max(np.abs(got - ref)) <= 1e-12
    # shared keys (K1 = K2) and identical queries cancel exactly at lambda = 1
    assert np.all(oracle.differential_attention(q1, k1, q1, k1, v, 1.0, True) == 0.0)
    # rows of O through ones of width D are 1 - lambda
    o = oracle.differential_attention(q1, k1, q2, k1, np.ones((1, 2, 7, 4)), 0.3, True)
    assert np.max(np.abs(o - 0.7)) <= 1e-12
    # queries over a cache with Dv = D equal the last rows of the full pass
    full = oracle.differential_attention(q1, k1, q2, k2, v, 0.6, True)
    tail = oracle.differential_attention_kv(q1[:, :, -3:], k1, q2[:, :, -3:], k2, v, 0.6, True)
    assert np.max(np.abs(full[:, :, -3:] - tail)) <= 1e-12


# ---------------------------------------------------------------------------
# Mutation tests: a mistake planted in one step of the oracle must fail a pin.
# ---------------------------------------------------------------------------

def _wrong_sign(a1, a2, lam):
    return a1 + lam * a2


def _lambda_on_first(a1, a2, lam):
    return lam * a1 - a2


def _scale_by_D(q, k):
    return (q @ k.T) / q.shape[-1]


def _no_scale(q, k):
    return q @ k.T


def _transposed_scores(q, k):
    # S^T in place of S (only expressible when every query row is evaluated).
    if q.shape[0] != k.shape[0]:
        return (q @ k.T) / math.sqrt(q.shape[-1])
    return (k @ q.T) / math.sqrt(q.shape[-1])


def _mask_diag_off(s, rows, causal, offset=0):
    if not causal:
        return s
    keys = np.arange(s.shape[-1])
    out = s.copy()
    out[keys[None, :] >= rows[:, None] + offset] = -np.inf
    out[np.all(np.isinf(out), axis=-1)] = 0.0
    return out


def _mask_upper_kept(s, rows, causal, offset=0):
    if not causal:
        return s
    keys = np.arange(s.shape[-1])
    out = s.copy()
    out[keys[None, :] < rows[:, None] + offset] = -np.inf
    return out


def _mask_branch1_only(q1, k1, q2, k2, rows, lam, causal, offset=0):
    a1 = O._softmax(O._mask(O._scores(q1[rows], k1), rows, causal, offset))
    a2 = O._softmax(O._scores(q2[rows], k2))
    return O._combine(a1, a2, lam)


def _softmax_wrong_axis(s):
    m = np.max(s, axis=0, keepdims=True)
    e = np.exp(s - m)
    return e / np.sum(e, axis=0, keepdims=True)


def _softmax_unnormalised(s):
    m = np.max(s, axis=-1, keepdims=True)
    return np.exp(s - m)


MUTANTS = [
    ("_combine", _wrong_sign),
    ("_combine", _lambda_on_first),
    ("_scores", _scale_by_D),
    ("_scores", _no_scale),
    ("_scores", _transposed_scores),
    ("_mask", _mask_diag_off),
    ("_mask", _mask_upper_kept),
    ("_softmax", _softmax_wrong_axis),
    ("_softmax", _softmax_unnormalised),
    ("_head_rows", _mask_branch1_only),
]


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m[1].__name__ for m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(O, name, mutant)
    failures = 0
    for pin in ALL_PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, IndexError, FloatingPointError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake in {name}"


def test_planted_lambda_sign_is_caught(monkeypatch):
    def bad(lq1, lk1, lq2, lk2, lambda_init=0.2):
        return math.exp(np.dot(lq1, lk1)) + math.exp(np.dot(lq2, lk2)) + lambda_init
    monkeypatch.setattr(oracle, "differential_lambda", bad)
    with pytest.raises(AssertionError):
        pin_lambda()


# ---------------------------------------------------------------------------
# Per-head norm and multiplier (the step after the operation)
# ---------------------------------------------------------------------------

def test_head_norm_group_matches_torch_group_norm():
    rng = np.random.default_rng(40)
    B, H, T, C = 2, 3, 5, 16
    o = rng.normal(1.5, 2.0, size=(B, H, T, C))
    w = rng.normal(size=(H, C))
    b = rng.normal(size=(H, C))
    got = oracle.head_norm(o, "group", 1e-5, w, b, out_scale=0.37)
    x = torch.from_numpy(o).permute(0, 2, 1, 3).reshape(B * T, H * C)   # a token's channels
    ref = torch.nn.functional.group_norm(x, H, torch.from_numpy(w.reshape(-1)),
                                         torch.from_numpy(b.reshape(-1)), eps=1e-5)
    ref = (0.37 * ref).reshape(B, T, H, C).permute(0, 2, 1, 3).numpy()
    assert np.max(np.abs(got - ref)) <= 1e-12


def test_head_norm_rms_matches_torch_rms_norm():
    rng = np.random.default_rng(41)
    o = rng.normal(0.3, 1.7, size=(2, 4, 6, 32))
    w = rng.normal(size=(4, 32))
    got = oracle.head_norm(o, "rms", 1e-6, w, None, out_scale=0.8)
    ref = np.stack([torch.nn.functional.rms_norm(torch.from_numpy(o[:, h]), (32,),
                                                 torch.from_numpy(w[h]), eps=1e-6).numpy()
                    for h in range(4)], axis=1)
    assert np.max(np.abs(got - 0.8 * ref)) <= 1e-12


def test_head_norm_invariants():
    rng = np.random.default_rng(42)
    o = rng.normal(size=(1, 2, 7, 8))
    g = oracle.head_norm(o, "group", 0.0)
    assert np.max(np.abs(g.mean(-1))) <= 1e-12 and np.max(np.abs(g.var(-1) - 1)) <= 1e-12
    r = oracle.head_norm(o, "rms", 0.0)
    assert np.max(np.abs(np.mean(r * r, -1) - 1)) <= 1e-12
    # scale invariance (eps = 0) and the multiplier
    assert np.max(np.abs(oracle.head_norm(3.5 * o, "rms", 0.0) - r)) <= 1e-12
    assert np.max(np.abs(oracle.head_norm(o, "none", out_scale=0.25) - 0.25 * o)) <= 0
    with pytest.raises(ValueError):
        oracle.head_norm(o, "layer")


# ---------------------------------------------------------------------------
# Decode over a KV cache (Tq queries at the end of Tk keys)
# ---------------------------------------------------------------------------

def brute_force_kv(q1, k1, q2, k2, v, lam, causal):
    B, H, Tq, D = q1.shape
    Tk = k1.shape[2]
    out = np.zeros((B, H, Tq, v.shape[-1]))
    for b in range(B):
        for h in range(H):
            for i in range(Tq):
                pos = Tk - Tq + i
                visible = [j for j in range(Tk) if (not causal) or j <= pos]
                weights = [0.0] * Tk
                for q, k, sign in ((q1, k1, 1.0), (q2, k2, -lam)):
                    logit = {j: sum(float(q[b, h, i, c]) * float(k[b, h, j, c]) for c in range(D)) / math.sqrt(D)
                             for j in visible}
                    top = max(logit.values())
                    z = sum(math.exp(x - top) for x in logit.values())
                    for j in visible:
                        weights[j] += sign * math.exp(logit[j] - top) / z
                for c in range(v.shape[-1]):
                    out[b, h, i, c] = sum(weights[j] * float(v[b, h, j, c]) for j in range(Tk))
    return out


def test_kv_decode_brute_force():
    rng = np.random.default_rng(50)
    for (Tq, Tk) in [(1, 7), (2, 9), (3, 3), (1, 1)]:
        q1, q2 = rng.standard_normal((2, 1, 2, Tq, 4))
        k1, k2 = rng.standard_normal((2, 1, 2, Tk, 4))
        v = rng.standard_normal((1, 2, Tk, 8))
        for lam in (0.0, 0.8, -0.4):
            for causal in (True, False):
                got = oracle.differential_attention_kv(q1, k1, q2, k2, v, lam, causal)
                ref = brute_force_kv(q1, k1, q2, k2, v, lam, causal)
                assert np.max(np.abs(got - ref)) <= 1e-12, (Tq, Tk, lam, causal)


def test_kv_decode_rows_match_full_sequence():
    """Decode of the last Tq positions equals those rows of the full causal pass."""
    q1, k1, q2, k2, v = rand_inputs(1, 2, 40, 8, 51)
    full = oracle.differential_attention(q1, k1, q2, k2, v, 0.6, True)
    dec = oracle.differential_attention_kv(q1[:, :, -3:], k1, q2[:, :, -3:], k2, v, 0.6, True)
    assert np.max(np.abs(dec - full[:, :, -3:])) <= 1e-13
    with pytest.raises(ValueError):
        oracle.differential_attention_kv(q1, k1[:, :, :5], q2, k2[:, :, :5], v[:, :, :5], 0.6, True)


# ---------------------------------------------------------------------------
# Grouped key/value heads (DIFF V2 layout: H query heads over H_kv KV heads)
# ---------------------------------------------------------------------------

def test_grouped_heads_lambda0_matches_torch_gqa():
    rng = np.random.default_rng(60)
    q1, q2 = rng.standard_normal((2, 2, 6, 20, 8))
    k1, k2 = rng.standard_normal((2, 2, 2, 20, 8))
    v = rng.standard_normal((2, 2, 20, 16))
    for causal in (True, False):
        got = oracle.differential_attention(q1, k1, q2, k2, v, 0.0, causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q1), torch.from_numpy(k1), torch.from_numpy(v), is_causal=causal,
            enable_gqa=True).numpy()
        assert np.max(np.abs(got - ref)) <= 1e-12


def test_grouped_heads_brute_force():
    rng = np.random.default_rng(61)
    q1, q2 = rng.standard_normal((2, 1, 4, 6, 4))
    k1, k2 = rng.standard_normal((2, 1, 2, 6, 4))
    v = rng.standard_normal((1, 2, 6, 8))
    for causal in (True, False):
        got = oracle.differential_attention(q1, k1, q2, k2, v, 0.8, causal)
        # brute force per query head on the key/value head it shares
        for h in range(4):
            ref = brute_force(q1[:, h:h + 1], k1[:, h // 2:h // 2 + 1], q2[:, h:h + 1],
                              k2[:, h // 2:h // 2 + 1], v[:, h // 2:h // 2 + 1], 0.8, causal)
            assert np.max(np.abs(got[:, h:h + 1] - ref)) <= 1e-12
    with pytest.raises(ValueError):
        oracle.differential_attention(q1[:, :3], k1, q2[:, :3], k2, v, 0.8)


def test_grouped_heads_kv_cache_matches_full_sequence_rows():
    # Tq queries at the end of Tk keys with grouped heads equal the last Tq rows
    # of the full-sequence forward with the same grouping
    rng = np.random.default_rng(62)
    q1, q2 = rng.standard_normal((2, 1, 6, 12, 4))
    k1, k2 = rng.standard_normal((2, 1, 3, 12, 4))
    v = rng.standard_normal((1, 3, 12, 8))
    full = oracle.differential_attention(q1, k1, q2, k2, v, 0.6, True)
    tail = oracle.differential_attention_kv(q1[:, :, -3:], k1, q2[:, :, -3:], k2, v, 0.6, True)
    assert np.max(np.abs(full[:, :, -3:] - tail)) <= 1e-12
