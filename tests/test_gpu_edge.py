"""GPU edge cases against the float64 oracle: ragged and tiny T, lambda
outside [0, 1], exact cancellation of identical branches, strided layouts,
the CUDA-core path's shapes, device-resident lambda, output guard regions,
determinism and the device status word."""
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


def inputs(B, H, T, D, dtype="bf16", seed=0):
    w = W.Workload("edge", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed)
    return W.draw(w)


def gpu(inp, dtype, lam, causal, **kw):
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    return da.differential_attention(*dev, lam, causal=causal, **kw), dev


def ref(inp, lam, causal):
    return oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal)


@pytest.mark.parametrize("T", [1, 2, 3, 64, 127, 128, 129, 200, 255, 256, 257, 384, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_ragged_T_tensor_core(T, causal):
    inp = inputs(1, 2, T, 64, seed=T)
    out, dev = gpu(inp, "bf16", 0.8, causal)
    assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_TCGEN05
    assert_close(to_numpy(out), ref(inp, 0.8, causal), "bf16", f"T={T} causal={causal}")


@pytest.mark.parametrize("lam", [-0.7, 0.0, 1.0, 1.9])
def test_lambda_outside_unit_interval(lam):
    inp = inputs(2, 2, 300, 64, seed=5)
    for causal in (True, False):
        out, _ = gpu(inp, "bf16", lam, causal)
        assert_close(to_numpy(out), ref(inp, lam, causal), "bf16", f"lam={lam}")


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 32), ("f32", 64), ("f32", 32)])
def test_identical_branches_cancel_exactly(dtype, D):
    inp = inputs(2, 3, 333, D, dtype=dtype, seed=6)
    q = to_device(inp.q1, dtype)
    k = to_device(inp.k1, dtype)
    v = to_device(inp.v, dtype)
    for causal in (True, False):
        out = da.differential_attention(q, k, q.clone(), k.clone(), v, 1.0, causal=causal)
        assert torch.count_nonzero(out).item() == 0
        out = da.differential_attention(q, k, q, k, v, 0.25, causal=causal)
        r = oracle.differential_attention(inp.q1, inp.k1, inp.q1, inp.k1, inp.v, 0.25, causal)
        assert_close(to_numpy(out), r, dtype, "identical branches lambda=0.25")


def test_v1_head_split_layout():
    """Q = [Q1, Q2] and K = [K1, K2] as halves of one [B, H, T, 2D] tensor
    (aifetchly, section 1: the head dimension is split in two)."""
    inp = inputs(2, 2, 260, 64, seed=7)
    Q = to_device(np.concatenate([inp.q1, inp.q2], -1), "bf16")
    K = to_device(np.concatenate([inp.k1, inp.k2], -1), "bf16")
    v = to_device(inp.v, "bf16")
    q1, q2, k1, k2 = Q[..., :64], Q[..., 64:], K[..., :64], K[..., 64:]
    assert da.select_kernel(q1, k1, q2, k2, v) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(q1, k1, q2, k2, v, 0.6, causal=True)
    assert_close(to_numpy(out), ref(inp, 0.6, True), "bf16", "split-head views")


def test_token_major_layout_and_strided_output():
    """Tensors stored [B, T, H, *] and viewed as [B, H, T, *]; output written
    through a strided view."""
    inp = inputs(2, 3, 190, 64, seed=8)
    dev = [to_device(np.ascontiguousarray(x.transpose(0, 2, 1, 3)), "bf16").transpose(1, 2)
           for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out_buf = torch.empty(2, 190, 3, 128, dtype=torch.bfloat16, device="cuda")
    out = out_buf.transpose(1, 2)
    assert da.select_kernel(*dev, out=out) == da.DIFFATTN_KERNEL_TCGEN05
    da.differential_attention(*dev, 0.45, causal=False, out=out)
    assert_close(to_numpy(out), ref(inp, 0.45, False), "bf16", "token-major")


def test_non_contiguous_inner_dim_is_marshalled():
    inp = inputs(1, 2, 100, 64, seed=9)
    dev = [to_device(np.repeat(x, 2, axis=-1), "bf16")[..., ::2] for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out = da.differential_attention(*dev, 0.3, causal=True)
    assert_close(to_numpy(out), ref(inp, 0.3, True), "bf16", "inner stride 2")


@pytest.mark.parametrize("dtype,D,T", [("bf16", 16, 150), ("bf16", 100, 77), ("bf16", 128, 129),
                                       ("f32", 64, 300), ("f32", 128, 70), ("f32", 1, 5),
                                       ("f32", 32, 1)])
def test_cuda_core_path(dtype, D, T):
    inp = inputs(2, 2, T, D, dtype=dtype, seed=D + T)
    for causal in (True, False):
        out, dev = gpu(inp, dtype, 0.7, causal)
        assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_SIMT
        assert_close(to_numpy(out), ref(inp, 0.7, causal), dtype, f"simt {dtype} D={D} T={T}")


def test_unaligned_bf16_d64_falls_back_to_cuda_cores():
    inp = inputs(1, 2, 140, 64, seed=10)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    buf = torch.empty(dev[2].numel() + 1, dtype=torch.bfloat16, device="cuda")
    q2 = buf[1:].view(dev[2].shape)
    q2.copy_(dev[2])
    dev[2] = q2
    assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_SIMT
    # the slower kernel is not chosen silently: the binding warns (once)
    da._WARNED_SLOW.discard("differential_attention")
    with pytest.warns(RuntimeWarning, match="CUDA-core kernel"):
        out = da.differential_attention(*dev, 0.8, causal=True)
    assert_close(to_numpy(out), ref(inp, 0.8, True), "bf16", "unaligned q2")


def test_device_lambda_matches_host_lambda():
    inp = inputs(1, 4, 500, 64, seed=11)
    vecs = [torch.from_numpy(x).cuda() for x in (inp.lq1, inp.lk1, inp.lq2, inp.lk2)]
    lam_t = da.differential_lambda(*vecs, lambda_init=0.5)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    a = da.differential_attention(*dev, lam_t, causal=True)
    b = da.differential_attention(*dev, float(lam_t.item()), causal=True)
    assert torch.equal(a, b)
    assert_close(to_numpy(a), ref(inp, float(lam_t.item()), True), "bf16", "device lambda")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_output_guard_regions_untouched(dtype):
    inp = inputs(2, 2, 257, 64, dtype=dtype, seed=12)
    n = 2 * 2 * 257 * 128
    guard = 4096
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    buf = torch.full((n + 2 * guard,), -12345.0, dtype=tdt, device="cuda")
    out = buf[guard:guard + n].view(2, 2, 257, 128)
    gpu(inp, dtype, 0.8, True, out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:guard] == -12345.0) and torch.all(buf[guard + n:] == -12345.0)
    assert_close(to_numpy(out), ref(inp, 0.8, True), dtype, "guarded output")


def test_deterministic_and_status_clean():
    inp = inputs(2, 4, 1111, 64, seed=13)
    a, dev = gpu(inp, "bf16", 0.8, True)
    b = da.differential_attention(*dev, 0.8, causal=True)
    assert torch.equal(a, b)
    assert da.get_device_error() == 0


def test_many_items_multiple_waves():
    # More work items than SMs, and heads of unequal causal cost.
    inp = inputs(3, 40, 640, 64, seed=14)
    out, _ = gpu(inp, "bf16", 0.8, True)
    rows = [0, 1, 127, 128, 300, 511, 512, 639]
    r = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.8, True, rows=rows)
    assert_close(to_numpy(out[:, :, rows]), r, "bf16", "multi-wave")


def test_empty_and_mismatched_inputs_rejected():
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(1, 1, 4, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):          # V with another sequence length
        da.differential_attention(x, x, x, x, v[:, :, :3], 0.5)
    with pytest.raises(ValueError):          # V wider than 256
        da.differential_attention(x, x, x, x, torch.zeros(1, 1, 4, 300, dtype=torch.bfloat16,
                                                          device="cuda"), 0.5)
    with pytest.raises(ValueError):
        da.differential_attention(x, x, x, x.float(), v, 0.5)
    e = torch.zeros(1, 1, 0, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(da.DiffattnError):
        da.differential_attention(e, e, e, e, torch.zeros(1, 1, 0, 128, dtype=torch.bfloat16, device="cuda"), 0.5)


@pytest.mark.parametrize("causal", [True, False])
def test_static_and_dynamic_schedules_agree(causal):
    inp = inputs(3, 20, 700, 64, seed=15)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    a = da.differential_attention(*dev, 0.8, causal=causal, dynamic_schedule=False)
    b = da.differential_attention(*dev, 0.8, causal=causal, dynamic_schedule=True)
    c = da.differential_attention(*dev, 0.8, causal=causal, dynamic_schedule=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(b, c)
    ws = da.workspace_for(dev[0].device, torch.cuda.current_stream())
    assert torch.count_nonzero(ws).item() == 0      # left zeroed for the next call
    rows = [0, 127, 128, 699]
    r = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.8, causal, rows=rows)
    assert_close(to_numpy(b[:, :, rows]), r, "bf16", "dynamic schedule")


def test_dynamic_schedule_on_a_side_stream():
    inp = inputs(2, 8, 1000, 64, seed=16)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    ref = da.differential_attention(*dev, 0.5, causal=True, dynamic_schedule=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs = [da.differential_attention(*dev, 0.5, causal=True) for _ in range(3)]
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert all(torch.equal(o, ref) for o in outs)
    assert da.get_device_error() == 0
