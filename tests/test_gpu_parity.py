"""GPU parity: the CUDA path against the float64 oracle on the five seeded
workloads, through the C ABI (via the Python binding).

The small workloads are compared on every output element; the large ones on
every element of two whole heads plus sampled query rows of every head (the
oracle is row-separable, so a sampled row is exact).  The sampled rows include
row 0, row T-1, both sides of tile boundaries, and the planted query rows.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import assert_close, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def lambda32(w, inp):
    """lambda from the oracle's float64 formula, rounded once to float32; both
    sides then use this same value."""
    lam = oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2, W.lambda_init_for(w))
    return float(np.float32(lam))


def run_gpu(inp, w, lam, causal):
    dev = [to_device(x, w.dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    kern = da.select_kernel(*dev)
    out = da.differential_attention(*dev, lam, causal=causal)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    return out, kern


def sampled_check(w, inp, out, lam, causal, full_heads, rows):
    """Whole heads `full_heads` plus `rows` of every head."""
    B, H = inp.q1.shape[:2]
    for (b, h) in full_heads:
        ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal,
                                            heads=[(b, h)])[0]
        assert_close(to_numpy(out[b, h]), ref, w.dtype, f"{w.name} head ({b},{h})")
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal, rows=rows)
    got = to_numpy(out[:, :, torch.as_tensor(rows, device=out.device)])
    return assert_close(got, ref, w.dtype, f"{w.name} sampled rows")


def test_tiny_f32_full():
    w = W.WORKLOADS["tiny_f32"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    out, kern = run_gpu(inp, w, lam, w.causal)
    assert kern == da.DIFFATTN_KERNEL_SIMT
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, w.causal)
    assert_close(to_numpy(out), ref, "f32", "tiny fp32")


def test_tiny_shape_bf16_full():
    w = W.WORKLOADS["tiny_f32"]
    inp = W.draw(w, dtype="bf16")
    lam = lambda32(w, inp)
    out, _ = run_gpu(inp, W.Workload(**{**w.__dict__, "dtype": "bf16"}), lam, w.causal)
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, w.causal)
    assert_close(to_numpy(out), ref, "bf16", "tiny bf16")


def test_b4h16t2048_full():
    w = W.WORKLOADS["b4h16t2048"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    out, kern = run_gpu(inp, w, lam, w.causal)
    assert kern == da.DIFFATTN_KERNEL_TCGEN05
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, w.causal)
    assert_close(to_numpy(out), ref, "bf16", w.name)


def test_headline_b2h16t8192_sampled():
    w = W.WORKLOADS["b2h16t8192"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    out, kern = run_gpu(inp, w, lam, w.causal)
    assert kern == da.DIFFATTN_KERNEL_TCGEN05
    rows = W.check_rows(w.T, n_random=32, seed=2)
    rows = rows[::4] if rows.size > 160 else rows
    sampled_check(w, inp, out, lam, w.causal, [(0, 0), (1, 15)], rows)


def test_planted_b1h16t32768_sampled():
    w = W.WORKLOADS["b1h16t32768_planted"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    out, kern = run_gpu(inp, w, lam, w.causal)
    assert kern == da.DIFFATTN_KERNEL_TCGEN05
    planted = np.unique(inp.planted_queries)
    rows = np.unique(np.concatenate([W.check_rows(w.T, n_random=16, seed=3)[::16], planted,
                                     np.unique(inp.planted_keys)]))
    # one whole head (every one of its 32768 rows, its 8 planted keys among them)
    sampled_check(w, inp, out, lam, w.causal, [(0, 9)], rows)


@pytest.mark.parametrize("lam", [0.0, 0.5, 1.0])
def test_offset_b8h32t4096_sweep(lam):
    w = W.WORKLOADS["b8h32t4096_offset"]
    inp = _offset_inputs()
    out, kern = run_gpu(inp, w, lam, w.causal)
    assert kern == da.DIFFATTN_KERNEL_TCGEN05
    rows = W.check_rows(w.T, n_random=8, seed=4)[::8]
    sampled_check(w, inp, out, lam, w.causal, [(0, 0), (7, 31)], rows)


_OFFSET_CACHE = {}


def _offset_inputs():
    if "x" not in _OFFSET_CACHE:
        _OFFSET_CACHE["x"] = W.draw(W.WORKLOADS["b8h32t4096_offset"])
    return _OFFSET_CACHE["x"]


def test_offset_response_is_one_minus_lambda():
    """O(V + 1c^T) - O(V) = (1 - lambda) c for a value offset shared by every
    token (paperleet, Toy experiment), on the GPU, per head."""
    w = W.Workload("offset_small", B=2, H=4, T=1000, D=64, dtype="bf16", causal=False, seed=40)
    inp = W.draw(w)
    c = np.round(np.random.default_rng(9).normal(0, 2, size=(2, 4, 1, 128)) * 4) / 4  # exact in bf16
    v0 = inp.v
    v1 = W.round_to_bf16((v0 + c).astype(np.float32))
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2)]
    for causal in (False, True):
        for lam in (0.0, 0.5, 1.0, 1.5):
            o0 = to_numpy(da.differential_attention(*dev, to_device(v0, "bf16"), lam, causal=causal))
            o1 = to_numpy(da.differential_attention(*dev, to_device(v1, "bf16"), lam, causal=causal))
            # exact inputs give O(v1) - O(v0) = A (v1 - v0); compare with the oracle of that
            ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, v1 - v0, lam, causal)
            assert np.max(np.abs((o1 - o0) - ref)) <= 2 * 2e-2
            # and v1 - v0 is c up to the rounding of v0 + c, so the response is ~ (1 - lambda) c
            assert np.mean(np.abs((o1 - o0) - (1 - lam) * c)) <= 2e-2


def test_lambda_kernel_matches_oracle():
    for w in W.WORKLOADS.values():
        inp = W.draw(w, T=1, B=1, H=1)
        vecs = [torch.from_numpy(x).cuda() for x in (inp.lq1, inp.lk1, inp.lq2, inp.lk2)]
        got = da.differential_lambda(*vecs, lambda_init=W.lambda_init_for(w) if w.lambdas is None else 0.8)
        ref = oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2,
                                         W.lambda_init_for(w) if w.lambdas is None else 0.8)
        assert got.shape == () and got.dtype == torch.float32
        assert abs(float(got) - ref) <= 1e-6 * max(1.0, abs(ref))
    z = torch.zeros(64, device="cuda")
    assert float(da.differential_lambda(z, z, z, z, 0.37)) == np.float32(0.37)
    e = torch.zeros(8, device="cuda"); e[0] = 1.0
    t = torch.zeros(8, device="cuda"); t[0] = 2.0
    assert abs(float(da.differential_lambda(e, t, z[:8], z[:8], 0.2)) - (np.exp(2) - 1 + 0.2)) <= 1e-6


def test_grouped_shared_keys_b2h16kv4t8192_sampled():
    # the DIFF V2 layout at the headline size: 16 heads over 4 key/value heads,
    # one key tensor for both branches
    w = W.GQA_WORKLOADS["b2h16kv4t8192_shared_k"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    dev = [to_device(x, w.dtype) for x in (inp.q1, inp.k1, inp.q2, inp.v)]
    q1, k, q2, v = dev
    assert da.select_kernel(q1, k, q2, k, v) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(q1, k, q2, k, v, lam, causal=w.causal)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    rows = W.check_rows(w.T, n_random=32, seed=5)[::4]
    sampled_check(w, inp, out, lam, w.causal, [(0, 3), (1, 12)], rows)


def test_headline_backward_sampled_heads():
    # the backward at the headline size, from the training forward's saved
    # results (the launch configuration of bench.py --mode backward); the
    # oracle's backward for two key/value heads (query heads (0,0) and (1,15))
    from tests.helpers import SAVED_PATH_SLACK, assert_grad_close
    w = W.WORKLOADS["b2h16t8192"]
    inp = W.draw(w)
    lam = lambda32(w, inp)
    rng = np.random.Generator(np.random.PCG64(w.seed + 1000))
    dout = W.round_to_bf16(rng.standard_normal((w.B, w.H, w.T, w.Dv), dtype=np.float32))
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    saved = da.differential_attention_train(*dev, lam, causal=True)
    got = da.differential_attention_backward(*dev, lam, to_device(dout, "bf16"), True, saved=saved)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    heads = [(0, 0), (1, 15)]
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, dout,
                                                 True, kv_heads=heads)
    for b, h in heads:
        for name, g, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), got[:5], ref[:5]):
            assert_grad_close(to_numpy(g[b, h]), r[b, h], "bf16", f"headline backward ({b},{h}) {name}",
                              slack=SAVED_PATH_SLACK)
