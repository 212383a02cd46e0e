"""GPU parity of the backward (diffattn_bwd, diffattn_lambda_backward and the
autograd nodes of the binding) against the float64 oracle's backward."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import assert_dlambda_close, assert_grad_close, to_device, to_numpy

pytestmark = pytest.mark.gpu

NAMES = ("dq1", "dk1", "dq2", "dk2", "dv")


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def draw(B, H, Hk, T, D, dtype, seed):
    w = W.Workload("bwd", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed)
    inp = W.draw(w, kv_heads=Hk)
    rng = np.random.Generator(np.random.PCG64(seed + 1000))
    dout = rng.standard_normal((B, H, T, 2 * D), dtype=np.float32)
    if dtype == "bf16":
        dout = W.round_to_bf16(dout)
    return inp, dout


def check(inp, dout, dtype, lam, causal, what, dev_inputs=None):
    dev = dev_inputs or [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    got = da.differential_attention_backward(*dev, lam, to_device(dout, dtype), causal)
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v,
                                                 float(lam), dout, causal)
    for name, g, r in zip(NAMES, got[:5], ref[:5]):
        assert_grad_close(to_numpy(g), r, dtype, f"{what} {name}")
    # dlambda: a sum over every row, held to the output bound in units of the
    # L2 norm of its row terms dO . (A_2 V)
    a2v = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, causal)
    assert_dlambda_close(float(got[5]), ref[5], np.sum(dout * a2v, axis=-1), dtype, f"{what} dlambda")
    return got


@pytest.mark.parametrize("T", [1, 7, 33, 130, 257])
@pytest.mark.parametrize("causal", [True, False])
def test_backward_f32(T, causal):
    inp, dout = draw(1, 2, 2, T, 32, "f32", seed=T)
    check(inp, dout, "f32", 0.8, causal, f"f32 T={T} causal={causal}")


@pytest.mark.parametrize("D", [64, 128, 48])
@pytest.mark.parametrize("lam", [0.7, -0.3, 0.0])
def test_backward_bf16(D, lam):
    inp, dout = draw(2, 2, 2, 200, D, "bf16", seed=D)
    for causal in (True, False):
        check(inp, dout, "bf16", lam, causal, f"bf16 D={D} lam={lam} causal={causal}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_backward_grouped_heads(dtype):
    inp, dout = draw(1, 6, 2, 150, 64, dtype, seed=21)
    check(inp, dout, dtype, 0.5, True, f"{dtype} grouped 6/2")


def test_backward_shared_keys_and_device_lambda():
    inp, dout = draw(1, 4, 2, 120, 64, "bf16", seed=22)
    inp.k2 = inp.k1
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.v)]
    q1, k, q2, v = dev
    lam = torch.tensor(0.6, device="cuda")
    check(inp, dout, "bf16", lam, True, "shared keys", dev_inputs=[q1, k, q2, k, v])


def test_backward_strided_token_major_views():
    inp, dout = draw(1, 3, 3, 90, 64, "f32", seed=23)
    # token-major storage [B, T, H, *] seen through a [B, H, T, *] view
    dev = [to_device(np.ascontiguousarray(x.transpose(0, 2, 1, 3)), "f32").transpose(1, 2)
           for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    check(inp, dout, "f32", 0.4, True, "token-major", dev_inputs=dev)


def test_backward_is_reproducible():
    inp, dout = draw(1, 2, 2, 300, 64, "bf16", seed=24)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    g = to_device(dout, "bf16")
    a = da.differential_attention_backward(*dev, 0.5, g, True)
    b = da.differential_attention_backward(*dev, 0.5, g, True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_autograd_end_to_end_with_lambda_vectors():
    inp, dout = draw(1, 2, 2, 64, 32, "f32", seed=25)
    dev = [to_device(x, "f32").requires_grad_() for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    vecs = [torch.from_numpy(x).cuda().requires_grad_() for x in (inp.lq1, inp.lk1, inp.lq2, inp.lk2)]
    lam = da.differential_lambda(*vecs, lambda_init=0.8)
    out = da.differential_attention(*dev, lam, causal=True)
    out.backward(to_device(dout, "f32"))
    lam_ref = oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2, 0.8)
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v,
                                                 float(np.float32(lam_ref)), dout, True)
    for name, t, r in zip(NAMES, dev, ref[:5]):
        assert_grad_close(to_numpy(t.grad), r, "f32", f"autograd {name}")
    vref = oracle.differential_lambda_backward(inp.lq1, inp.lk1, inp.lq2, inp.lk2, ref[5])
    for t, r in zip(vecs, vref):
        assert np.max(np.abs(to_numpy(t.grad) - r)) <= 1e-4 * max(1.0, float(np.max(np.abs(r))))


def test_autograd_rejects_epilogue():
    inp, _ = draw(1, 2, 2, 16, 32, "f32", seed=26)
    dev = [to_device(x, "f32").requires_grad_() for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    with pytest.raises(ValueError):
        da.differential_attention(*dev, 0.5, norm="rms")


def test_backward_rejects_bad_arguments():
    inp, dout = draw(1, 2, 2, 16, 32, "f32", seed=27)
    dev = [to_device(x, "f32") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    with pytest.raises(ValueError):
        da.differential_attention_backward(*dev, 0.5, to_device(dout[:, :, :8], "f32"))


# ---------------------------------------------------------------------------
# The tensor-core backward (bf16, D = 64, aligned): ragged lengths, both masks,
# grouped heads, shared keys, several tiles per item
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 200, 257, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_backward_tensor_core_ragged(T, causal):
    inp, dout = draw(1, 2, 2, T, 64, "bf16", seed=100 + T)
    check(inp, dout, "bf16", 0.8, causal, f"tc bwd T={T} causal={causal}")


@pytest.mark.parametrize("H,Hk", [(8, 2), (4, 1), (6, 3)])
def test_backward_tensor_core_grouped(H, Hk):
    inp, dout = draw(2, H, Hk, 700, 64, "bf16", seed=H * 10 + Hk)
    for causal in (True, False):
        check(inp, dout, "bf16", -0.4, causal, f"tc bwd grouped {H}/{Hk} causal={causal}")


def test_backward_tensor_core_long_and_reproducible():
    inp, dout = draw(1, 4, 4, 2048, 64, "bf16", seed=200)
    got = check(inp, dout, "bf16", 0.6, True, "tc bwd T=2048")
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    again = da.differential_attention_backward(*dev, 0.6, to_device(dout, "bf16"), True)
    for x, y in zip(got, again):
        assert torch.equal(x, y)


def test_backward_unaligned_view_runs_on_cuda_cores():
    # a view that starts 2 bytes past a 16-byte boundary cannot use TMA; the
    # CUDA-core backward takes it and must agree with the oracle as well
    inp, dout = draw(1, 2, 2, 150, 64, "bf16", seed=201)
    base = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    shifted = []
    for t in base:
        buf = torch.empty(t.numel() + 1, dtype=t.dtype, device=t.device)
        view = buf[1:].view(t.shape)
        view.copy_(t)
        shifted.append(view)
    assert shifted[0].data_ptr() % 16 != 0
    check(inp, dout, "bf16", 0.7, True, "simt bwd unaligned bf16", dev_inputs=shifted)
