"""GPU parity of queries over a key/value cache beyond a decode step (a chunk
of a prefill): Tq new queries at the end of a Tk-key sequence, query i seeing
keys j <= Tk - Tq + i, against the float64 oracle's differential_attention_kv.
More query rows than the split-key decode takes run on the forward kernels
(tensor cores for bf16 with value width 128)."""
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


def case(B, H, Tq, Tk, D, seed, dtype="bf16", kv_heads=None, Dv=None):
    w = W.DecodeWorkload("prefill", B, H, Tq, Tk, D, dtype, True, seed, kv_heads=kv_heads,
                         value_dim=Dv)
    return W.draw_kv(w)


def check(inp, lam, causal, dtype="bf16", shared=False, what=""):
    q1, k1, q2, k2, v = (to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v))
    if shared:
        k2 = k1
        inp.k2 = inp.k1
    out = da.differential_attention_decode(q1, k1, q2, k2, v, lam, causal=causal)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    want = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal)
    return assert_close(to_numpy(out), want, dtype, what)


@pytest.mark.parametrize("Tq", [9, 128, 1000])
@pytest.mark.parametrize("mult", [1, 4])
@pytest.mark.parametrize("causal", [True, False])
def test_chunk_over_cache_tensor_cores(Tq, mult, causal):
    inp = case(2, 3, Tq, mult * Tq, 64, seed=400 + Tq + mult)
    check(inp, 0.6, causal, what=f"prefill Tq={Tq} Tk={mult * Tq} causal={causal}")


@pytest.mark.parametrize("Tq,Tk", [(9, 70), (200, 1000), (129, 129), (64, 8000)])
def test_chunk_over_cache_v2_head(Tq, Tk):
    # D = Dv = 128, grouped heads with shared keys: the tensor-core kernel's
    # second head shape
    inp = case(1, 4, Tq, Tk, 128, seed=410 + Tq, kv_heads=2, Dv=128)
    for causal in (True, False):
        check(inp, -0.3, causal, shared=True, what=f"prefill V2 Tq={Tq} Tk={Tk} causal={causal}")


@pytest.mark.parametrize("dtype,D", [("f32", 32), ("bf16", 48), ("f32", 128)])
def test_chunk_over_cache_cuda_cores(dtype, D):
    inp = case(1, 2, 37, 300, D, seed=420 + D, dtype=dtype)
    for causal in (True, False):
        check(inp, 0.9, causal, dtype=dtype, what=f"prefill simt {dtype} D={D} causal={causal}")


def test_decode_rows_with_v2_value_width():
    # a decode step (one query) with the V2 head's value width goes through
    # the forward kernels as well
    inp = case(2, 4, 1, 3000, 128, seed=430, kv_heads=2, Dv=128)
    check(inp, 0.5, True, shared=True, what="decode V2 value width")


def test_chunk_rows_equal_full_sequence_rows():
    # the last Tq rows of a full causal forward equal a chunk of Tq queries over
    # the same keys (on the GPU: two different launch shapes, one answer)
    w = W.Workload("chunk", B=1, H=4, T=1500, D=64, dtype="bf16", causal=True, seed=440,
                   lambda_init=0.8)
    inp = W.draw(w)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    full = da.differential_attention(*dev, 0.7, causal=True)
    tail = da.differential_attention_decode(dev[0][:, :, -300:], dev[1], dev[2][:, :, -300:],
                                            dev[3], dev[4], 0.7, causal=True)
    torch.cuda.synchronize()
    want = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.7, True,
                                         rows=np.arange(1200, 1500))
    assert_close(to_numpy(tail), want, "bf16", "chunk vs oracle rows")
    assert_close(to_numpy(full[:, :, -300:]), want, "bf16", "full vs oracle rows")


def test_prefill_workload_sampled():
    w = W.PREFILL_WORKLOADS["prefill_b4h16q1024k8192"]
    inp = W.draw_kv(w)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out = da.differential_attention_decode(*dev, w.lambda_value, causal=True)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    sel = [(0, 0), (3, 15), (2, 7)]
    for b, h in sel:
        sub = [x[b:b + 1, h:h + 1] for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
        want = oracle.differential_attention_kv(*sub, w.lambda_value, True)[0, 0]
        assert_close(to_numpy(out[b, h]), want, "bf16", f"{w.name} head ({b},{h})")
