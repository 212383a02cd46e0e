"""The allocation-free decode entry point.

diffattn_decode_noalloc serves callers that cannot allocate device memory when
they run a decode step (for example a runtime that owns all device buffers and
passes only inputs and outputs, or a loop that must not call the allocator):
it keeps the split partial results in a fixed 8 MiB buffer inside the library.
This test calls it through the C ABI twice in a row, on different inputs, and
checks each result against diffattn_decode with a caller workspace, within the
bf16 parity tolerance used by the other tests.  It also checks that a problem
needing more than the buffer holds is refused.  This file is collected last.
"""
import ctypes

import pytest
import torch

import workloads as W
import differential_attention_fwd_gb300 as da
from differential_attention_fwd_gb300 import _lib
from differential_attention_fwd_gb300 import build as build_mod
from tests.helpers import assert_close, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return _lib.load()


def _inputs(seed, Tq, Tk):
    w = W.DecodeWorkload("noalloc", 2, 8, Tq, Tk, 64, "bf16", True, seed)
    inp = W.draw_kv(w)
    return [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]


def _call_noalloc(lib, dev, lam, causal):
    out = torch.empty(dev[0].shape[:3] + (2 * dev[0].shape[3],), dtype=dev[0].dtype, device="cuda")
    d = da.make_kv_desc(*dev, out)
    rc = lib.diffattn_decode_noalloc(ctypes.byref(d), *(ctypes.c_void_p(t.data_ptr()) for t in dev),
                                     ctypes.c_float(lam), None, 1 if causal else 0, None,
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out


def test_noalloc_decode_matches_workspace_decode_twice(lib):
    for seed, Tq, Tk, lam, causal in ((61, 1, 5000, 0.7, True), (62, 4, 3000, -0.2, False)):
        dev = _inputs(seed, Tq, Tk)
        rc, got = _call_noalloc(lib, dev, lam, causal)
        assert rc == _lib.DIFFATTN_OK, _lib.strerror(rc)
        ref = da.differential_attention_decode(*dev, lam, causal=causal)
        torch.cuda.synchronize()
        assert_close(to_numpy(got), to_numpy(ref).astype("float64"), "bf16", "noalloc vs workspace")
    assert da.get_device_error() == 0


def test_noalloc_calls_back_to_back_on_one_stream(lib):
    # Two calls enqueued one after the other on one stream with no host
    # synchronisation between them: the CUDA-core path (one query row) and
    # the tensor-core path (four rows).  Both use the one library buffer; the
    # second call's first pass must not overwrite it while the first call's
    # combine pass still reads it.  Each result is checked against the
    # workspace decode and against the float64 oracle.
    import oracle
    cases = ((71, 1, 6000, 0.6, True), (72, 4, 4000, 0.9, True))
    devs = [_inputs(seed, Tq, Tk) for seed, Tq, Tk, _, _ in cases]
    torch.cuda.synchronize()
    outs = []
    for dev, (_, _, _, lam, causal) in zip(devs, cases):
        rc, out = _call_noalloc(lib, dev, lam, causal)
        assert rc == _lib.DIFFATTN_OK, _lib.strerror(rc)
        outs.append(out)
    torch.cuda.synchronize()
    for dev, out, (_, _, _, lam, causal) in zip(devs, outs, cases):
        ref = da.differential_attention_decode(*dev, lam, causal=causal)
        torch.cuda.synchronize()
        assert_close(to_numpy(out), to_numpy(ref), "bf16", "noalloc back to back vs workspace")
        want = oracle.differential_attention_kv(*(to_numpy(t) for t in dev), lam, causal)
        assert_close(to_numpy(out), want, "bf16", "noalloc back to back vs oracle")
    assert da.get_device_error() == 0


def test_noalloc_refuses_problems_beyond_its_buffer(lib):
    # 8192 heads x 1 split x 2 queries x 260 floats = 17 MB of partial results
    q = torch.zeros(128, 64, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(128, 64, 2, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(128, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(128, 64, 2, 128, dtype=torch.bfloat16, device="cuda")
    d = da.make_kv_desc(q, k, q, k, v, out)
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(d)) > 8 * 1024 * 1024
    rc, _ = _call_noalloc(lib, [q, k, q, k, v], 0.5, True)
    assert rc == _lib.DIFFATTN_ERR_UNSUPPORTED
