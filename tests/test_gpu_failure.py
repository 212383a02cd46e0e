"""The kernels' failure path on the GPU, without a fault: a bounded mbarrier
wait that runs out (here, a wait on a barrier nothing ever completes) records
the timeout in the device status word, diffattn_get_device_error reports it
once and clears it, and the CUDA context goes on working."""
import time

import pytest
import torch

import oracle
import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import _lib
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import assert_close, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def test_wait_timeout_is_reported_and_the_context_survives():
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.diffattn_get_device_error(stream) == _lib.DIFFATTN_OK
    t0 = time.monotonic()
    assert lib.diffattn_selftest_timeout(stream) == _lib.DIFFATTN_OK
    # the wait gives up at the library's limit (about two seconds)
    assert lib.diffattn_get_device_error(stream) == _lib.DIFFATTN_ERR_TIMEOUT
    assert 1.0 < time.monotonic() - t0 < 60.0
    # reported once, then cleared
    assert lib.diffattn_get_device_error(stream) == _lib.DIFFATTN_OK
    # the context still runs the tensor-core forward correctly
    w = W.Workload("after_timeout", B=1, H=2, T=300, D=64, dtype="bf16", causal=True, seed=11)
    inp = W.draw(w)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    assert da.select_kernel(*dev) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(*dev, 0.6, causal=True)
    ref = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, True)
    assert_close(to_numpy(out), ref, "bf16", "forward after a reported timeout")
    assert lib.diffattn_get_device_error(stream) == _lib.DIFFATTN_OK
