"""GPU parity of the DIFF V2 head shape against the float64 oracle.

The aiengineeringfromscratch lesson ("V1 contre V2") keeps the baseline's head
dimension for DIFF V2: Q, K and V are all D = 128 wide (value width Dv = D),
the two branches of a differential head share their key/value head, and 32
query heads run over 8 key/value heads.  bf16 with D = Dv = 128 runs on the
tensor-core kernel; other value widths on the CUDA-core kernel.  A decode step
of that head (bf16, up to 8 queries, one key tensor, dense cache rows) runs on
the tensor-core split-key decode; the rest of its decode shapes on the forward
kernels.
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


def inputs(B, H, T, D, Dv, seed, kv_heads=None, shared=False, dtype="bf16"):
    w = W.Workload("v2", B=B, H=H, T=T, D=D, dtype=dtype, causal=True, seed=seed,
                   kv_heads=kv_heads, shared_keys=shared, value_dim=Dv, lambda_init=0.8)
    return W.draw(w)


def run(inp, lam, causal, dtype="bf16", shared=False, **kw):
    q1, k1, q2, k2, v = (to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v))
    if shared:
        k2 = k1
    kern = da.select_kernel(q1, k1, q2, k2, v)
    out = da.differential_attention(q1, k1, q2, k2, v, lam, causal=causal, **kw)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    return out, kern


def ref(inp, lam, causal, **kw):
    return oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal, **kw)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129, 200, 257, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_d128_dv128_tensor_core_ragged(T, causal):
    inp = inputs(2, 2, T, 128, 128, seed=300 + T)
    out, kern = run(inp, 0.7, causal)
    assert kern == da.DIFFATTN_KERNEL_TCGEN05
    assert_close(to_numpy(out), ref(inp, 0.7, causal), "bf16", f"V2 head T={T} causal={causal}")


@pytest.mark.parametrize("lam", [0.0, 0.5, 1.0, -0.4, 1.6])
def test_d128_grouped_shared_keys(lam):
    # 8 differential heads over 2 key/value heads, one key tensor for both branches
    inp = inputs(2, 8, 700, 128, 128, seed=310, kv_heads=2, shared=True)
    for causal in (True, False):
        out, kern = run(inp, lam, causal, shared=True)
        assert kern == da.DIFFATTN_KERNEL_TCGEN05
        assert_close(to_numpy(out), ref(inp, lam, causal), "bf16",
                     f"V2 grouped shared lam={lam} causal={causal}")


def test_d128_separate_keys_and_identical_branches():
    inp = inputs(1, 4, 513, 128, 128, seed=311, kv_heads=2)
    out, _ = run(inp, 0.3, True)
    assert_close(to_numpy(out), ref(inp, 0.3, True), "bf16", "V2 separate keys")
    # identical branches cancel exactly at lambda = 1
    q1, k1, v = (to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.v))
    o = da.differential_attention(q1, k1, q1, k1, v, 1.0, causal=True)
    torch.cuda.synchronize()
    assert int(torch.count_nonzero(o)) == 0


def test_d128_value_rows_through_ones():
    # V = 1 everywhere: every output is 1 - lambda (each map's rows sum to 1)
    inp = inputs(1, 2, 300, 128, 128, seed=312)
    inp.v = np.ones_like(inp.v)
    out, _ = run(inp, 0.35, True)
    assert float((out.float() - 0.65).abs().max()) <= 2e-2


def test_d128_group_norm_epilogue():
    inp = inputs(1, 4, 384, 128, 128, seed=313)
    g = torch.Generator().manual_seed(3)
    nw = 1 + 0.1 * torch.randn(4, 128, generator=g)
    nb = 0.1 * torch.randn(4, 128, generator=g)
    out, _ = run(inp, 0.6, True, norm="group", norm_eps=1e-5, norm_weight=nw.cuda(),
                 norm_bias=nb.cuda(), out_scale=0.2)
    want = oracle.head_norm(ref(inp, 0.6, True), "group", 1e-5, nw.numpy(), nb.numpy(), 0.2)
    assert_close(to_numpy(out), want, "bf16", "V2 group norm epilogue")


def test_d128_training_outputs():
    inp = inputs(1, 2, 400, 128, 128, seed=314)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    out, out2, lse = da.differential_attention_train(*dev, 0.4, causal=True)
    torch.cuda.synchronize()
    assert_close(to_numpy(out), ref(inp, 0.4, True), "bf16", "V2 train out")
    a2v = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, True)
    assert_close(to_numpy(out2), a2v, "bf16", "V2 train A2 V")
    for b, (q, k) in enumerate(((inp.q1, inp.k1), (inp.q2, inp.k2))):
        want = oracle.branch_logsumexp(q, k, True)
        assert np.max(np.abs(to_numpy(lse[..., b]) - want)) <= 1e-3


def test_headline_size_v2_b2h16kv8t8192_sampled():
    w = W.GQA_WORKLOADS["b2h16kv8t8192_d128_shared_k"]
    inp = W.draw(w)
    lam = float(np.float32(oracle.differential_lambda(inp.lq1, inp.lk1, inp.lq2, inp.lk2,
                                                      W.lambda_init_for(w))))
    q1, k, q2, v = (to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.v))
    assert da.select_kernel(q1, k, q2, k, v) == da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(q1, k, q2, k, v, lam, causal=True)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    for b, h in ((0, 5), (1, 14)):
        want = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, True,
                                             heads=[(b, h)])[0]
        assert_close(to_numpy(out[b, h]), want, "bf16", f"{w.name} head ({b},{h})")
    rows = W.check_rows(w.T, n_random=32, seed=7)[::4]
    want = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, True, rows=rows)
    got = to_numpy(out[:, :, torch.as_tensor(rows, device=out.device)])
    assert_close(got, want, "bf16", f"{w.name} sampled rows")


@pytest.mark.parametrize("dtype,D,Dv", [("f32", 32, 32), ("bf16", 64, 64), ("bf16", 48, 5),
                                        ("f32", 16, 256), ("bf16", 128, 200)])
def test_other_value_widths_on_cuda_cores(dtype, D, Dv):
    inp = inputs(2, 2, 150, D, Dv, seed=320 + Dv, dtype=dtype)
    for causal in (True, False):
        out, kern = run(inp, 0.8, causal, dtype=dtype)
        assert kern == da.DIFFATTN_KERNEL_SIMT
        assert tuple(out.shape) == (2, 2, 150, Dv)
        assert_close(to_numpy(out), ref(inp, 0.8, causal), dtype, f"{dtype} D={D} Dv={Dv}")


def test_backward_rejects_mismatched_dout():
    inp = inputs(1, 2, 64, 128, 128, seed=330)
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    dout = torch.zeros(1, 2, 64, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        da.differential_attention_backward(*dev, 0.5, dout, True)


def _dout(inp, dtype, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    d = rng.standard_normal(inp.q1.shape[:3] + (inp.v.shape[-1],), dtype=np.float32)
    return W.round_to_bf16(d) if dtype == "bf16" else d


@pytest.mark.parametrize("dtype,D,Dv,T", [("bf16", 128, 128, 1), ("bf16", 128, 128, 150),
                                          ("f32", 32, 32, 77), ("bf16", 64, 64, 130),
                                          ("f32", 16, 40, 33)])
def test_backward_other_value_widths(dtype, D, Dv, T):
    # the DIFF V2 head (Dv = D) and other widths: the CUDA-core backward
    from tests.helpers import assert_dlambda_close, assert_grad_close
    inp = inputs(1, 4, T, D, Dv, seed=340 + T + Dv, kv_heads=2, dtype=dtype)
    dout = _dout(inp, dtype, 341 + T)
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    for causal in (True, False):
        got = da.differential_attention_backward(*dev, 0.6, to_device(dout, dtype), causal)
        ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6,
                                                     dout, causal)
        for name, g, r in zip(("dq1", "dk1", "dq2", "dk2", "dv"), got[:5], ref[:5]):
            assert tuple(g.shape) == r.shape
            assert_grad_close(to_numpy(g), r, dtype, f"V2 bwd {dtype} D={D} Dv={Dv} T={T} {name}")
        a2v = oracle.differential_attention(inp.q2, inp.k2, inp.q2, inp.k2, inp.v, 0.0, causal)
        assert_dlambda_close(float(got[5]), ref[5], np.sum(dout * a2v, axis=-1), dtype,
                             f"V2 bwd {dtype} D={D} Dv={Dv} T={T} dlambda")


def test_autograd_v2_head_shared_keys():
    # training through the V2 head: the forward on the tensor cores with its
    # saved results, the backward on the CUDA cores, one key tensor for both
    # branches (its gradient sums both branches' contributions)
    from tests.helpers import SAVED_PATH_SLACK, assert_grad_close
    inp = inputs(1, 4, 200, 128, 128, seed=350, kv_heads=2, shared=True)
    dout = _dout(inp, "bf16", 351)
    q1, k, q2, v = (to_device(x, "bf16").requires_grad_() for x in (inp.q1, inp.k1, inp.q2, inp.v))
    assert da.select_kernel(q1.detach(), k.detach(), q2.detach(), k.detach(), v.detach()) == \
        da.DIFFATTN_KERNEL_TCGEN05
    out = da.differential_attention(q1, k, q2, k, v, 0.5, causal=True)
    out.backward(to_device(dout, "bf16"))
    ref = oracle.differential_attention_backward(inp.q1, inp.k1, inp.q2, inp.k1, inp.v, 0.5, dout, True)
    want_k = ref[1] + ref[3]
    for name, t, r in (("dq1", q1, ref[0]), ("dq2", q2, ref[2]), ("dk", k, want_k), ("dv", v, ref[4])):
        assert_grad_close(to_numpy(t.grad), r, "bf16", f"autograd V2 {name}", slack=SAVED_PATH_SLACK)


def decode_inputs(B, H, Hk, Tq, Tk, seed, shared=True, dtype="bf16"):
    w = W.DecodeWorkload("v2dec", B, H, Tq, Tk, 128, dtype, True, seed=seed, kv_heads=Hk,
                         value_dim=128, shared_keys=shared)
    inp = W.draw_kv(w)
    if shared:
        inp.k2 = inp.k1
    return inp


def decode_run(inp, lam, causal, dtype="bf16", kv=None, **kw):
    q1, k1, q2, k2, v = (to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v))
    if inp.k2 is inp.k1:
        k2 = k1
    if kv is not None:
        k1, k2, v = kv(k1, k2, v)
    out = da.differential_attention_decode(q1, k1, q2, k2, v, lam, causal=causal, **kw)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    return out


def decode_ref(inp, lam, causal):
    return oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, lam, causal)


def split_key_workspace(B, H, Hk, Tq, Tk):
    """Workspace bytes of a V2 decode call: more than the forward kernels'
    nominal 16 when the call is planned for the split-key decode."""
    from differential_attention_fwd_gb300 import _lib
    import ctypes
    d = _lib.DiffattnKvDesc()
    d.B, d.H, d.Tq, d.Tk, d.D, d.Dv = B, H, Tq, Tk, 128, 128
    d.dtype, d.kv_group = _lib.DIFFATTN_BF16, H // Hk
    for f, T, h in (("q1_stride", Tq, H), ("q2_stride", Tq, H), ("k1_stride", Tk, Hk),
                    ("k2_stride", Tk, Hk), ("v_stride", Tk, Hk), ("o_stride", Tq, H)):
        getattr(d, f)[:] = (h * T * 128, T * 128, 128)
    return _lib.load().diffattn_decode_workspace_bytes(ctypes.byref(d))


# rows per key/value head (H / Hk * Tq): 1, 2, 4, 6 (padded to 8), 8, 16 (one
# unit), 48 (three units of 16); caches of one key, a ragged tail, one tile,
# many tiles
@pytest.mark.parametrize("B,H,Hk,Tq,Tk", [(2, 4, 4, 1, 1), (2, 16, 8, 1, 8192), (1, 8, 2, 1, 300),
                                          (2, 8, 1, 1, 1000), (1, 4, 2, 3, 1000), (1, 4, 1, 4, 2000),
                                          (2, 2, 2, 8, 129), (1, 32, 8, 2, 5000), (1, 2, 2, 5, 128),
                                          (2, 4, 2, 8, 1500), (1, 4, 1, 12, 640), (1, 2, 2, 16, 300)])
@pytest.mark.parametrize("causal", [True, False])
def test_v2_decode_split_key_tensor_core(B, H, Hk, Tq, Tk, causal):
    assert split_key_workspace(B, H, Hk, Tq, Tk) > 16
    inp = decode_inputs(B, H, Hk, Tq, Tk, seed=400 + H * Tq + Tk)
    out = decode_run(inp, 0.7, causal)
    assert tuple(out.shape) == (B, H, Tq, 128)
    assert_close(to_numpy(out), decode_ref(inp, 0.7, causal), "bf16",
                 f"V2 decode B={B} H={H} Hk={Hk} Tq={Tq} Tk={Tk} causal={causal}")


@pytest.mark.parametrize("norm", [None, "rms", "group"])
def test_v2_decode_epilogue_device_lambda_repeat(norm):
    inp = decode_inputs(2, 8, 4, 2, 3000, seed=420)
    rng = np.random.default_rng(5)
    wt = (1 + 0.1 * rng.standard_normal((8, 128))).astype(np.float32)
    bs = (0.05 * rng.standard_normal((8, 128))).astype(np.float32)
    lam_t = torch.tensor(-0.3, device="cuda")
    kw = dict(out_scale=0.6)
    if norm:
        kw.update(norm=norm, norm_weight=torch.from_numpy(wt).cuda(), norm_bias=torch.from_numpy(bs).cuda())
    want = oracle.head_norm(decode_ref(inp, -0.3, True), norm or "none", 1e-5, wt if norm else None,
                            bs if norm else None, 0.6)
    for call in range(2):
        out = decode_run(inp, lam_t, True, **kw)
        assert_close(to_numpy(out), want, "bf16", f"V2 decode epilogue {norm} call {call}")


def test_v2_decode_value_rows_through_ones_and_cancellation():
    # V = 1: every output is 1 - lambda; identical branches cancel at lambda = 1
    inp = decode_inputs(1, 8, 2, 1, 777, seed=430)
    inp.v = np.ones_like(inp.v)
    out = decode_run(inp, 0.35, True)
    assert float((out.float() - 0.65).abs().max()) <= 2e-2
    inp.q2 = inp.q1
    out = decode_run(inp, 1.0, True)
    assert int(torch.count_nonzero(out)) == 0


def test_v2_decode_shapes_on_the_forward_kernels():
    """The V2 decode shapes the split-key pass does not take (two key
    tensors, a cache with rows not contiguous along the sequence, fp32, more
    than 16 queries) run on the forward kernels; all match the oracle."""
    inp = decode_inputs(1, 8, 2, 1, 1500, seed=440, shared=False)
    assert_close(to_numpy(decode_run(inp, 0.5, True)), decode_ref(inp, 0.5, True), "bf16",
                 "V2 decode two key tensors")
    inp = decode_inputs(2, 8, 2, 2, 1500, seed=441)

    def token_major(k1, k2, v):
        # [B, Tk, Hk, *] storage seen as [B, Hk, Tk, *], one key tensor
        tm = lambda t: t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3)
        k = tm(k1)
        return k, k, tm(v)

    out = decode_run(inp, 0.5, True, kv=token_major)
    assert_close(to_numpy(out), decode_ref(inp, 0.5, True), "bf16", "V2 decode token-major cache")
    inp = decode_inputs(1, 4, 2, 2, 600, seed=442, dtype="f32")
    assert_close(to_numpy(decode_run(inp, 0.5, True, dtype="f32")), decode_ref(inp, 0.5, True),
                 "f32", "V2 decode fp32")
    assert split_key_workspace(1, 4, 2, 17, 600) == 16
    inp = decode_inputs(1, 4, 2, 17, 600, seed=443)
    assert_close(to_numpy(decode_run(inp, 0.5, True)), decode_ref(inp, 0.5, True), "bf16",
                 "V2 decode Tq=17")


def test_v2_decode_matches_oracle_last_rows_at_full_size():
    # the decode workload's shape (16 heads over 8 key/value heads, 8192
    # cached keys, one new query per head), two of its sequences
    w = W.DECODE_WORKLOADS["decode_b16h16kv8q1k8192_d128_shared_k"]
    inp = W.draw_kv(w, B=2)
    inp.k2 = inp.k1
    out = decode_run(inp, w.lambda_value, w.causal)
    assert_close(to_numpy(out), decode_ref(inp, w.lambda_value, w.causal), "bf16", w.name)
