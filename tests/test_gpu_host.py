"""The host-buffer forward (diffattn_fwd_host): inputs and output in host
memory, copies pipelined with the forward over chunks of heads.  Its output is
the device forward's, bit for bit, and the oracle's within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import assert_close, to_device, to_numpy, torch_dtype

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def host(x, dtype):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch_dtype(dtype)).pin_memory()


@pytest.mark.parametrize("B,H,Hk,T,dtype,causal", [(2, 16, 16, 1024, "bf16", True),
                                                   (2, 8, 2, 777, "bf16", False),
                                                   (1, 4, 4, 200, "f32", True),
                                                   (3, 6, 3, 129, "bf16", True)])
def test_host_forward_matches_device_forward(B, H, Hk, T, dtype, causal):
    w = W.Workload("host", B=B, H=H, T=T, D=64 if dtype == "bf16" else 32, dtype=dtype,
                   causal=causal, seed=B * 100 + T)
    inp = W.draw(w, kv_heads=Hk)
    hs = [host(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out = da.differential_attention_host(*hs, 0.7, causal=causal)
    torch.cuda.synchronize()
    assert out.device.type == "cpu"
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    ref_dev = da.differential_attention(*dev, 0.7, causal=causal).cpu()
    assert torch.equal(out, ref_dev)
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.7, causal)
    assert_close(to_numpy(out), ref, dtype, f"host forward B={B} H={H}/{Hk} T={T}")


def test_host_forward_shared_keys_and_reused_buffers():
    w = W.Workload("host", B=2, H=8, T=640, D=64, dtype="bf16", causal=True, seed=7)
    inp = W.draw(w, kv_heads=2)
    k = host(inp.k1, "bf16")
    hs = [host(inp.q1, "bf16"), k, host(inp.q2, "bf16"), k, host(inp.v, "bf16")]
    out1 = da.differential_attention_host(*hs, 0.5, causal=True)
    torch.cuda.synchronize()
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k1, inp.v, 0.5, True)
    assert_close(to_numpy(out1), ref, "bf16", "host forward shared keys")
    # a second call with new inputs into the same device buffers and output
    inp2 = W.draw(w, kv_heads=2, seed=8)
    k2 = host(inp2.k1, "bf16")
    hs2 = [host(inp2.q1, "bf16"), k2, host(inp2.q2, "bf16"), k2, host(inp2.v, "bf16")]
    out2 = da.differential_attention_host(*hs2, 0.5, causal=True, out=out1)
    torch.cuda.synchronize()
    ref2 = oracle.differential_attention(inp2.q1, inp2.k1, inp2.q2, inp2.k1, inp2.v, 0.5, True)
    assert_close(to_numpy(out2), ref2, "bf16", "host forward second call")
