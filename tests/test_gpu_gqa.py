"""GPU parity of grouped key/value heads (the DIFF V2 layout: H query heads
over H_kv = H / g key/value heads, query head h reading key/value head h // g)
against the float64 oracle, for the tensor-core, CUDA-core and decode paths;
also the two branches sharing one key tensor."""
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


def grouped(B, H, Hk, T, D, dtype="bf16", seed=0):
    w = W.Workload("gqa", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed)
    return W.draw(w, kv_heads=Hk)


def dev_all(inp, dtype):
    return [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]


@pytest.mark.parametrize("H,Hk,T", [(8, 2, 700), (4, 1, 513), (6, 3, 128), (8, 8, 300),
                                    (16, 4, 1100)])
@pytest.mark.parametrize("causal", [True, False])
def test_tensor_core_grouped_heads(H, Hk, T, causal):
    inp = grouped(2, H, Hk, T, 64, seed=H * 100 + Hk + T)
    dev = dev_all(inp, "bf16")
    assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(*dev, 0.8, causal=causal)
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.8, causal)
    assert_close(to_numpy(out), ref, "bf16", f"tc gqa H={H} Hk={Hk} T={T} causal={causal}")


@pytest.mark.parametrize("causal", [True, False])
def test_tensor_core_shared_keys_v2_layout(causal):
    # DIFF V2: 2H query heads in one tensor, the two branches of differential
    # head i are query heads 2i and 2i + 1, and both read the same key head.
    B, H, Hk, T, D = 2, 8, 2, 777, 64
    rng = np.random.default_rng(70)
    q = W.round_to_bf16(rng.standard_normal((B, 2 * H, T, D), dtype=np.float32))
    k = W.round_to_bf16(rng.standard_normal((B, Hk, T, D), dtype=np.float32))
    v = W.round_to_bf16(rng.standard_normal((B, Hk, T, 2 * D), dtype=np.float32))
    qd, kd, vd = (to_device(x, "bf16") for x in (q, k, v))
    q1, q2 = qd[:, 0::2], qd[:, 1::2]           # strided views, no copies
    assert da.select_kernel(q1, kd, q2, kd, vd) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(q1, kd, q2, kd, vd, 0.6, causal=causal)
    ref = oracle.differential_attention(q[:, 0::2], k, q[:, 1::2], k, v, 0.6, causal)
    assert_close(to_numpy(out), ref, "bf16", f"tc v2 shared keys causal={causal}")
    # the shared-key load path gives the same bits as passing two copies
    out2 = da.differential_attention(q1, kd, q2, kd.clone(), vd, 0.6, causal=causal)
    assert torch.equal(out, out2)


def test_tensor_core_grouped_schedules_agree_and_epilogue():
    inp = grouped(2, 8, 2, 1000, 64, seed=71)
    dev = dev_all(inp, "bf16")
    a = da.differential_attention(*dev, 0.5, causal=True, dynamic_schedule=True)
    b = da.differential_attention(*dev, 0.5, causal=True, dynamic_schedule=False)
    assert torch.equal(a, b)
    rng = np.random.default_rng(72)
    wt = (1 + 0.1 * rng.standard_normal((8, 128))).astype(np.float32)
    bs = (0.1 * rng.standard_normal((8, 128))).astype(np.float32)
    out = da.differential_attention(*dev, 0.5, causal=True, norm="group",
                                    norm_weight=torch.from_numpy(wt).cuda(),
                                    norm_bias=torch.from_numpy(bs).cuda(), out_scale=0.2)
    o = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.5, True)
    assert_close(to_numpy(out), oracle.head_norm(o, "group", 1e-5, wt, bs, 0.2), "bf16",
                 "tc gqa group norm")


@pytest.mark.parametrize("dtype,D", [("f32", 32), ("f32", 64), ("bf16", 32), ("bf16", 128)])
def test_cuda_core_grouped_heads(dtype, D):
    inp = grouped(1, 6, 2, 150, D, dtype=dtype, seed=D)
    dev = dev_all(inp, dtype)
    assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_SIMT
    for causal in (True, False):
        out = da.differential_attention(*dev, -0.4, causal=causal)
        ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, -0.4, causal)
        assert_close(to_numpy(out), ref, dtype, f"simt gqa {dtype} D={D} causal={causal}")


@pytest.mark.parametrize("dtype,D,H,Hk,Tq,Tk", [
    ("bf16", 64, 8, 2, 1, 3000),      # 4 rows per key/value head: one CTA
    ("bf16", 64, 8, 2, 2, 1025),      # 8 rows: one CTA
    ("bf16", 64, 8, 2, 3, 700),       # 12 rows: two CTAs of 6 (bucket 8)
    ("bf16", 64, 9, 3, 3, 513),       # 9 rows: two CTAs
    ("bf16", 64, 16, 1, 1, 4096),     # one key/value head for 16 query heads
    ("f32", 128, 8, 2, 1, 900),       # 4 rows at the D = 128 cap
    ("f32", 128, 8, 1, 2, 600),       # 16 rows: four CTAs of 4
    ("bf16", 32, 4, 2, 5, 800),
])
@pytest.mark.parametrize("causal", [True, False])
def test_decode_grouped_heads(dtype, D, H, Hk, Tq, Tk, causal):
    w = W.DecodeWorkload("t", 2, H, Tq, Tk, D, dtype, causal, seed=H + Hk + Tq + Tk, kv_heads=Hk)
    inp = W.draw_kv(w)
    dev = dev_all(inp, dtype)
    out = da.differential_attention_decode(*dev, 0.7, causal=causal)
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.7, causal)
    assert_close(to_numpy(out), ref, dtype, f"decode gqa {dtype} D={D} H={H} Hk={Hk} Tq={Tq}")


def test_decode_grouped_matches_forward_last_rows():
    inp = grouped(1, 8, 2, 640, 64, seed=73)
    dev = dev_all(inp, "bf16")
    full = da.differential_attention(*dev, 0.5, causal=True)
    dec = da.differential_attention_decode(dev[0][:, :, -2:], dev[1], dev[2][:, :, -2:], dev[3],
                                           dev[4], 0.5, causal=True)
    assert float((full[:, :, -2:].float() - dec.float()).abs().max()) <= 2e-2
    want = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.5, True,
                                         rows=[638, 639])
    assert_close(to_numpy(dec), want, "bf16", "grouped decode last rows vs oracle")
    assert_close(to_numpy(full[:, :, -2:]), want, "bf16", "grouped forward last rows vs oracle")


def test_grouped_heads_rejected_shapes():
    inp = grouped(1, 6, 6, 64, 64, seed=74)
    dev = dev_all(inp, "bf16")
    bad_k = dev[1][:, :4].contiguous()           # 4 key heads do not divide 6 query heads
    with pytest.raises(ValueError):
        da.differential_attention(dev[0], bad_k, dev[2], bad_k, dev[4][:, :4].contiguous(), 0.5)
    with pytest.raises(ValueError):
        da.differential_attention_decode(dev[0][:, :, :1], bad_k, dev[2][:, :, :1], bad_k,
                                         dev[4][:, :4].contiguous(), 0.5)
    with pytest.raises(ValueError):               # value heads must match key heads
        da.differential_attention(dev[0], dev[1], dev[2], dev[3], dev[4][:, :1].contiguous(), 0.5)
