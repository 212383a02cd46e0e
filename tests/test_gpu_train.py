"""GPU parity of the training forward (diffattn_fwd_train: O, A_2 V and the
per-branch log-sum-exp) and of the backward from its saved results
(diffattn_bwd_saved), against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import (SAVED_PATH_SLACK, assert_close, assert_dlambda_close, assert_grad_close,
                           to_device, to_numpy)

pytestmark = pytest.mark.gpu
NAMES = ("dq1", "dk1", "dq2", "dk2", "dv")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def draw(B, H, Hk, T, D, dtype, seed):
    w = W.Workload("train", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed)
    inp = W.draw(w, kv_heads=Hk)
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    dout = rng.standard_normal((B, H, T, 2 * D), dtype=np.float32)
    if dtype == "bf16":
        dout = W.round_to_bf16(dout)
    return inp, dout


CASES = [("bf16", 64, 2, 2, 300), ("bf16", 64, 8, 2, 513), ("bf16", 64, 2, 2, 1),
         ("f32", 32, 2, 1, 130), ("bf16", 48, 2, 2, 77)]


@pytest.mark.parametrize("dtype,D,H,Hk,T", CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_train_forward_outputs(dtype, D, H, Hk, T, causal):
    inp, _ = draw(1, H, Hk, T, D, dtype, seed=T + D)
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out, out2, lse = da.differential_attention_train(*dev, 0.6, causal=causal)
    # the output is the plain forward's, bit for bit
    assert torch.equal(out, da.differential_attention(*dev, 0.6, causal=causal))
    ref2 = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, causal)
    assert_close(to_numpy(out2), ref2, dtype, f"train out2 {dtype} T={T} causal={causal}")
    lse_ref = np.stack([oracle.branch_logsumexp(inp.q1, inp.k1, causal),
                        oracle.branch_logsumexp(inp.q2, inp.k2, causal)], axis=-1)
    assert lse.shape == (1, H, T, 2) and lse.dtype == torch.float32
    tol = 1e-4 if dtype == "f32" else 1e-3
    assert np.max(np.abs(to_numpy(lse) - lse_ref)) <= tol * max(1.0, float(np.max(np.abs(lse_ref))))


@pytest.mark.parametrize("dtype,D,H,Hk,T", CASES)
@pytest.mark.parametrize("causal", [True, False])
def test_backward_from_saved_results(dtype, D, H, Hk, T, causal):
    inp, dout = draw(1, H, Hk, T, D, dtype, seed=T + D + 1)
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    saved = da.differential_attention_train(*dev, -0.4, causal=causal)
    g = to_device(dout, dtype)
    got = da.differential_attention_backward(*dev, -0.4, g, causal, saved=saved)
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, -0.4,
                                                 dout, causal)
    for name, a, r in zip(NAMES, got[:5], ref[:5]):
        assert_grad_close(to_numpy(a), r, dtype, f"saved bwd {dtype} T={T} causal={causal} {name}",
                          slack=SAVED_PATH_SLACK)
    a2v = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, causal)
    assert_dlambda_close(float(got[5]), ref[5], np.sum(dout * a2v, axis=-1), dtype,
                         f"saved bwd {dtype} T={T} causal={causal} dlambda")


def test_autograd_bf16_tensor_core_end_to_end():
    inp, dout = draw(2, 4, 2, 700, 64, "bf16", seed=77)
    dev = [to_device(x, "bf16").requires_grad_() for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    lam = torch.tensor(0.55, device="cuda", requires_grad=True)
    out = da.differential_attention(*dev, lam, causal=True)
    out.backward(to_device(dout, "bf16"))
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v,
                                                 float(np.float32(0.55)), dout, True)
    for name, t, r in zip(NAMES, dev, ref[:5]):
        assert_grad_close(to_numpy(t.grad), r, "bf16", f"autograd bf16 {name}",
                          slack=SAVED_PATH_SLACK)
    a2v = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, True)
    assert_dlambda_close(float(lam.grad), ref[5], np.sum(dout * a2v, axis=-1), "bf16",
                         "autograd bf16 dlambda")


def test_saved_and_recomputed_backward_agree():
    inp, dout = draw(1, 4, 4, 1024, 64, "bf16", seed=78)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    g = to_device(dout, "bf16")
    saved = da.differential_attention_train(*dev, 0.7, causal=True)
    a = da.differential_attention_backward(*dev, 0.7, g, True, saved=saved)
    b = da.differential_attention_backward(*dev, 0.7, g, True)
    for x, y in zip(a[:5], b[:5]):
        assert float((x.float() - y.float()).abs().max()) <= 2e-2 * max(1.0, float(y.float().abs().max()))
    assert abs(float(a[5]) - float(b[5])) <= 1e-2 * max(1.0, abs(float(b[5])))
