"""Pins for the float64 oracle's backward, independent of the oracle's code.

The paperleet exercise ("Differential Transformer Attention", Return
requirements and Toy experiment) asks for gradients through both Q/K branches,
the value, the coefficient and the four lambda vectors, verified against
analytic vector-Jacobian products.  The oracle writes the chain rule out by
hand; these tests check it against:
  * torch autograd (float64) of a plain torch statement of the forward;
  * central finite differences of the float64 forward oracle;
  * torch's scaled_dot_product_attention backward at lambda = 0;
  * closed forms: gradients of the keys sum to zero over keys (softmax rows
    are shift-invariant), the value gradients sum to (1 - lambda) sum(dO),
    dlambda = -sum(dO * A_2 V), identical branches at lambda = 1 have zero
    gradient for V and for a shared Q/K.
Mutation tests plant one mistake at a time in a copy of the oracle's
per-head backward and check that a pin fails.
"""
import inspect
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import diffattn_oracle as O


def inputs(B, H, Hk, T, D, seed, Dv=None):
    rng = np.random.default_rng(seed)
    Dv = 2 * D if Dv is None else Dv
    q1, q2 = rng.standard_normal((2, B, H, T, D))
    k1, k2 = rng.standard_normal((2, B, Hk, T, D))
    v = rng.standard_normal((B, Hk, T, Dv))
    dout = rng.standard_normal((B, H, T, Dv))
    return q1, k1, q2, k2, v, dout


def torch_forward(q1, k1, q2, k2, v, lam, causal):
    """The operation in plain torch (float64), for autograd."""
    H, Hk = q1.shape[1], k1.shape[1]
    g = H // Hk
    k1, k2, v = (x.repeat_interleave(g, dim=1) for x in (k1, k2, v))
    T, D = q1.shape[2], q1.shape[3]
    mask = torch.zeros(T, T, dtype=torch.float64)
    if causal:
        mask = mask.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    a1 = torch.softmax(q1 @ k1.transpose(-1, -2) / math.sqrt(D) + mask, dim=-1)
    a2 = torch.softmax(q2 @ k2.transpose(-1, -2) / math.sqrt(D) + mask, dim=-1)
    return (a1 - lam * a2) @ v


def autograd_grads(q1, k1, q2, k2, v, dout, lam, causal):
    ts = [torch.tensor(x, dtype=torch.float64, requires_grad=True) for x in (q1, k1, q2, k2, v)]
    lt = torch.tensor(float(lam), dtype=torch.float64, requires_grad=True)
    out = torch_forward(*ts, lt, causal)
    out.backward(torch.from_numpy(dout))
    return [t.grad.numpy() for t in ts] + [float(lt.grad)]


CASES = [  # B, H, Hk, T, D, lam, causal
    (1, 2, 2, 7, 4, 0.8, True),
    (2, 2, 2, 9, 3, -0.35, False),
    (1, 4, 2, 6, 5, 1.7, True),
    (1, 3, 1, 5, 2, 0.0, False),
    (1, 1, 1, 1, 4, 0.5, True),
    (2, 2, 1, 33, 8, 0.6, True),
]


@pytest.mark.parametrize("case", CASES)
def test_backward_matches_torch_autograd(case):
    B, H, Hk, T, D, lam, causal = case
    q1, k1, q2, k2, v, dout = inputs(B, H, Hk, T, D, seed=T * 10 + D)
    got = oracle.differential_attention_backward(q1, k1, q2, k2, v, lam, dout, causal)
    ref = autograd_grads(q1, k1, q2, k2, v, dout, lam, causal)
    for name, a, b in zip(("dq1", "dk1", "dq2", "dk2", "dv"), got[:5], ref[:5]):
        assert a.shape == b.shape, name
        assert np.max(np.abs(a - b)) <= 1e-10, name
    assert abs(got[5] - ref[5]) <= 1e-10 * max(1.0, abs(ref[5]))


@pytest.mark.parametrize("case", [(1, 4, 2, 9, 4, 4, 0.7, True), (2, 2, 1, 7, 3, 3, -0.4, False),
                                  (1, 2, 2, 6, 4, 5, 1.2, True)])
def test_backward_value_width_matches_torch_autograd(case):
    # the DIFF V2 head's value width (Dv = D) and another width: the chain
    # rule is the same for any width of V
    B, H, Hk, T, D, Dv, lam, causal = case
    q1, k1, q2, k2, v, dout = inputs(B, H, Hk, T, D, seed=T * 7 + Dv, Dv=Dv)
    got = oracle.differential_attention_backward(q1, k1, q2, k2, v, lam, dout, causal)
    ref = autograd_grads(q1, k1, q2, k2, v, dout, lam, causal)
    for name, a, b in zip(("dq1", "dk1", "dq2", "dk2", "dv"), got[:5], ref[:5]):
        assert a.shape == b.shape, name
        assert np.max(np.abs(a - b)) <= 1e-10, name
    assert abs(got[5] - ref[5]) <= 1e-10 * max(1.0, abs(ref[5]))
    with pytest.raises(ValueError):
        oracle.differential_attention_backward(q1, k1, q2, k2, v, lam, dout[..., :-1], causal)


def test_backward_finite_differences():
    q1, k1, q2, k2, v, dout = inputs(1, 2, 1, 5, 3, seed=7)
    lam, causal, eps = 0.7, True, 1e-6
    got = oracle.differential_attention_backward(q1, k1, q2, k2, v, lam, dout, causal)
    base = [q1, k1, q2, k2, v]

    def loss(xs, lm):
        return float(np.sum(oracle.differential_attention(*xs, lm, causal) * dout))

    rng = np.random.default_rng(8)
    for t in range(5):
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in base[t].shape)
            plus = [x.copy() for x in base]
            minus = [x.copy() for x in base]
            plus[t][idx] += eps
            minus[t][idx] -= eps
            fd = (loss(plus, lam) - loss(minus, lam)) / (2 * eps)
            assert abs(fd - got[t][idx]) <= 1e-6 * max(1.0, abs(fd)), (t, idx)
    fd = (loss(base, lam + eps) - loss(base, lam - eps)) / (2 * eps)
    assert abs(fd - got[5]) <= 1e-6 * max(1.0, abs(fd))


@pytest.mark.parametrize("causal", [True, False])
def test_backward_lambda0_is_sdpa_backward(causal):
    q1, k1, q2, k2, v, dout = inputs(1, 2, 2, 10, 4, seed=9)
    got = oracle.differential_attention_backward(q1, k1, q2, k2, v, 0.0, dout, causal)
    ts = [torch.tensor(x, requires_grad=True) for x in (q1, k1, v)]
    out = torch.nn.functional.scaled_dot_product_attention(*ts, is_causal=causal)
    out.backward(torch.from_numpy(dout))
    for a, t in zip((got[0], got[1], got[4]), ts):
        assert np.max(np.abs(a - t.grad.numpy())) <= 1e-10
    assert np.max(np.abs(got[2])) == 0.0 and np.max(np.abs(got[3])) == 0.0


@pytest.mark.parametrize("lam,causal", [(0.8, True), (-0.4, False), (1.3, True)])
def test_backward_closed_forms(lam, causal):
    q1, k1, q2, k2, v, dout = inputs(2, 4, 2, 12, 4, seed=11)
    dq1, dk1, dq2, dk2, dv, dlam = oracle.differential_attention_backward(
        q1, k1, q2, k2, v, lam, dout, causal)
    # softmax rows are invariant to a shift of the scores, so key gradients sum to 0
    assert np.max(np.abs(dk1.sum(axis=2))) <= 1e-10
    assert np.max(np.abs(dk2.sum(axis=2))) <= 1e-10
    # sum over keys of dV = W^T dO summed = (1 - lambda) * sum over rows of dO
    g = 2
    douts = dout.reshape(2, 2, g, 12, 8).sum(axis=2)      # per key/value head
    assert np.max(np.abs(dv.sum(axis=2) - (1 - lam) * douts.sum(axis=2))) <= 1e-10
    # dlambda = -sum(dO * (A_2 V)); A_2 V is the forward at lambda 0 with branch 2 alone
    a2v = oracle.differential_attention(q2, k2, q2, k2, v, 0.0, causal)
    assert abs(dlam + float(np.sum(dout * a2v))) <= 1e-10 * max(1.0, abs(dlam))


def test_backward_identical_branches_cancel_at_lambda1():
    q, k, _, _, v, dout = inputs(1, 2, 2, 8, 4, seed=12)
    dq1, dk1, dq2, dk2, dv, _ = oracle.differential_attention_backward(q, k, q, k, v, 1.0, dout, True)
    assert np.max(np.abs(dv)) <= 1e-12
    assert np.max(np.abs(dq1 + dq2)) <= 1e-12      # a shared Q sees no change in O
    assert np.max(np.abs(dk1 + dk2)) <= 1e-12


def test_backward_kv_head_subset():
    q1, k1, q2, k2, v, dout = inputs(2, 4, 2, 9, 3, seed=13)
    full = oracle.differential_attention_backward(q1, k1, q2, k2, v, 0.6, dout, True)
    part = oracle.differential_attention_backward(q1, k1, q2, k2, v, 0.6, dout, True,
                                                  kv_heads=[(1, 0)])
    assert np.array_equal(part[0][1, 0:2], full[0][1, 0:2])
    assert np.array_equal(part[4][1, 0], full[4][1, 0])
    assert np.max(np.abs(part[0][0])) == 0.0


def test_lambda_vector_gradients():
    rng = np.random.default_rng(14)
    vecs = [0.3 * rng.standard_normal(6) for _ in range(4)]
    dlam = -1.7
    got = oracle.differential_lambda_backward(*vecs, dlam)
    ts = [torch.tensor(x, requires_grad=True) for x in vecs]
    lam = torch.exp(ts[0] @ ts[1]) - torch.exp(ts[2] @ ts[3]) + 0.8
    lam.backward(torch.tensor(dlam, dtype=torch.float64))
    for a, t in zip(got, ts):
        assert np.max(np.abs(a - t.grad.numpy())) <= 1e-12
    eps = 1e-6
    for i in range(4):
        p = [x.copy() for x in vecs]
        m = [x.copy() for x in vecs]
        p[i][2] += eps
        m[i][2] -= eps
        fd = dlam * (oracle.differential_lambda(*p, 0.8) - oracle.differential_lambda(*m, 0.8)) / (2 * eps)
        assert abs(fd - got[i][2]) <= 1e-7


# ---------------------------------------------------------------------------
# Mutation tests: one planted mistake in a copy of the per-head backward
# ---------------------------------------------------------------------------
MUTANTS = {
    "no_rowsum_term": ("ds = a * (da - np.sum(da * a, axis=-1, keepdims=True))", "ds = a * da"),
    "dA2_sign": ("(a2, -lam * dw, q2, k2, dq2, dk2)", "(a2, lam * dw, q2, k2, dq2, dk2)"),
    "dlam_sign": ("dlam += -float(np.sum(dw * a2))", "dlam += float(np.sum(dw * a2))"),
    "w_without_lambda": ("w = _combine(a1, a2, lam)", "w = _combine(a1, a2, 0.0)"),
    "dq_no_scale": ("dq[rows] = scale * (ds @ k)", "dq[rows] = ds @ k"),
    "dk_uses_other_q": ("dk += scale * (ds.T @ q[rows])", "dk += scale * (ds.T @ q1[rows])"),
    "dw_uses_dout_T": ("dw = g @ v.T", "dw = g @ v[::-1].T"),
    "mask_off": ("a1 = _softmax(_mask(_scores(q1[rows], k1), rows, causal))",
                 "a1 = _softmax(_mask(_scores(q1[rows], k1), rows, False))"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_backward_mistake_is_caught(monkeypatch, name):
    old, new = MUTANTS[name]
    src = inspect.getsource(O._head_backward)
    assert old in src, name
    ns = dict(O.__dict__)
    exec(src.replace(old, new), ns)
    monkeypatch.setattr(O, "_head_backward", ns["_head_backward"])
    caught = False
    for case in CASES:
        B, H, Hk, T, D, lam, causal = case
        if lam == 0.0 and name in ("dA2_sign", "dlam_sign"):
            continue
        q1, k1, q2, k2, v, dout = inputs(B, H, Hk, T, D, seed=T * 10 + D)
        got = oracle.differential_attention_backward(q1, k1, q2, k2, v, lam, dout, causal)
        ref = autograd_grads(q1, k1, q2, k2, v, dout, lam, causal)
        err = max([float(np.max(np.abs(a - b))) for a, b in zip(got[:5], ref[:5])] +
                  [abs(got[5] - ref[5])])
        if err > 1e-6:
            caught = True
            break
    assert caught, name


def test_branch_logsumexp_matches_scipy_and_closed_forms():
    from scipy.special import logsumexp
    rng = np.random.default_rng(15)
    q = rng.standard_normal((1, 4, 9, 5))
    k = rng.standard_normal((1, 2, 9, 5))
    for causal in (True, False):
        got = oracle.branch_logsumexp(q, k, causal)
        for h in range(4):
            s = q[0, h] @ k[0, h // 2].T / math.sqrt(5)
            if causal:
                s = np.where(np.tril(np.ones((9, 9), dtype=bool)), s, -np.inf)
            assert np.max(np.abs(got[0, h] - logsumexp(s, axis=-1))) <= 1e-12
    # first causal row sees one key: lse = q0 . k0 / sqrt(D)
    got = oracle.branch_logsumexp(q, k, True)
    assert abs(got[0, 0, 0] - float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(5)) <= 1e-12
    # equal scores over n visible keys: lse = s + log n
    qz = np.zeros((1, 1, 6, 3))
    assert np.allclose(oracle.branch_logsumexp(qz, qz, True)[0, 0], np.log(np.arange(1, 7)), atol=1e-14)
