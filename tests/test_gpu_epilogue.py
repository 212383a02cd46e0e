"""GPU parity of the fused output epilogue (per-head RMSNorm or GroupNorm,
affine weight/bias, then the (1 - lambda_init) multiplier) against the float64
oracle's head_norm applied to its differential_attention, on both kernels."""
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


def case(B, H, T, D, dtype, seed):
    return W.draw(W.Workload("epi", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed))


@pytest.mark.parametrize("norm", ["rms", "group"])
@pytest.mark.parametrize("affine", [False, True])
@pytest.mark.parametrize("dtype,D,T", [("bf16", 64, 300), ("bf16", 64, 1000), ("f32", 32, 130),
                                       ("bf16", 32, 200)])
def test_norm_epilogue(norm, affine, dtype, D, T):
    inp = case(2, 3, T, D, dtype, seed=T + D)
    H, Dv = 3, 2 * D
    rng = np.random.default_rng(7)
    w = (1 + 0.1 * rng.standard_normal((H, Dv))).astype(np.float32) if affine else None
    b = (0.1 * rng.standard_normal((H, Dv))).astype(np.float32) if affine else None
    lam_init = oracle.lambda_init_schedule(12)
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    for causal in (True, False):
        out = da.differential_attention(
            *dev, 0.7, causal=causal, norm=norm, norm_eps=1e-5,
            norm_weight=torch.from_numpy(w).cuda() if affine else None,
            norm_bias=torch.from_numpy(b).cuda() if affine else None, out_scale=1 - lam_init)
        o = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.7, causal)
        ref = oracle.head_norm(o, norm, 1e-5, w, b, out_scale=1 - lam_init)
        assert_close(to_numpy(out), ref, dtype, f"{norm} affine={affine} {dtype} D={D}")


def test_out_scale_only():
    inp = case(1, 2, 257, 64, "bf16", seed=3)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out = da.differential_attention(*dev, 0.6, causal=True, out_scale=0.25)
    ref = 0.25 * oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, True)
    assert_close(to_numpy(out), ref, "bf16", "out_scale")


def test_headline_shape_group_norm_sampled():
    w = W.WORKLOADS["b2h16t8192"]
    inp = W.draw(w)
    lam = float(np.float32(oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2,
                                                      W.lambda_init_for(w))))
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out = da.differential_attention(*dev, lam, causal=True, norm="group",
                                    out_scale=1 - W.lambda_init_for(w))
    rows = W.check_rows(w.T, n_random=16, seed=5)[::16]
    o = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, True, rows=rows)
    ref = oracle.head_norm(o, "group", 1e-5, out_scale=1 - W.lambda_init_for(w))
    assert_close(to_numpy(out[:, :, torch.as_tensor(rows, device="cuda")]), ref, "bf16",
                 "headline group norm")
    assert da.get_device_error() == 0
