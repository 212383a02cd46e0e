"""GPU parity of the decode path (Tq queries over a Tk-key cache, split-KV
kernels) against the float64 oracle's differential_attention_kv."""
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


def run(inp, dtype, lam, causal, **kw):
    dev = [to_device(x, dtype) for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    if inp.k2 is inp.k1:
        dev[3] = dev[1]             # one key tensor for both branches
    return da.differential_attention_decode(*dev, lam, causal=causal, **kw), dev


@pytest.mark.parametrize("Tq,Tk", [(1, 1), (1, 100), (1, 256), (1, 257), (2, 1000), (3, 4099),
                                   (4, 8192), (5, 300), (8, 2048), (1, 70000)])
@pytest.mark.parametrize("causal", [True, False])
def test_decode_bf16_d64(Tq, Tk, causal):
    w = W.DecodeWorkload("t", 2, 3, Tq, Tk, 64, "bf16", causal, seed=Tq * 7 + Tk)
    inp = W.draw_kv(w)
    out, _ = run(inp, "bf16", 0.7, causal)
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.7, causal)
    assert_close(to_numpy(out), ref, "bf16", f"decode Tq={Tq} Tk={Tk} causal={causal}")


@pytest.mark.parametrize("dtype,D,Tq", [("f32", 64, 1), ("f32", 32, 8), ("f32", 128, 4),
                                        ("bf16", 32, 3), ("bf16", 128, 2)])
def test_decode_other_shapes(dtype, D, Tq):
    w = W.DecodeWorkload("t", 1, 2, Tq, 1500, D, dtype, True, seed=D + Tq)
    inp = W.draw_kv(w)
    for causal in (True, False):
        out, _ = run(inp, dtype, -0.3, causal)
        ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, -0.3, causal)
        assert_close(to_numpy(out), ref, dtype, f"decode {dtype} D={D} Tq={Tq}")


def test_decode_matches_forward_last_rows():
    inp = W.draw(W.Workload("t", B=1, H=2, T=700, D=64, dtype="bf16", causal=True, seed=9))
    dev = [to_device(x, "bf16") for x in (inp.q1, inp.k1, inp.q2, inp.k2, inp.v)]
    full = da.differential_attention(*dev, 0.5, causal=True)
    dec = da.differential_attention_decode(dev[0][:, :, -3:], dev[1], dev[2][:, :, -3:], dev[3],
                                           dev[4], 0.5, causal=True)
    assert float((full[:, :, -3:].float() - dec.float()).abs().max()) <= 2e-2
    # both against the oracle's rows 697..699 of the full sequence
    want = oracle.differential_attention(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.5, True,
                                         rows=[697, 698, 699])
    assert_close(to_numpy(dec), want, "bf16", "decode last rows vs oracle")
    assert_close(to_numpy(full[:, :, -3:]), want, "bf16", "forward last rows vs oracle")


def test_decode_epilogue_and_device_lambda():
    w = W.DecodeWorkload("t", 2, 4, 2, 3000, 64, "bf16", True, seed=33)
    inp = W.draw_kv(w)
    rng = np.random.default_rng(1)
    wt = (1 + 0.1 * rng.standard_normal((4, 128))).astype(np.float32)
    lam_t = torch.tensor(0.6, device="cuda")
    out, _ = run(inp, "bf16", lam_t, True, norm="rms", norm_weight=torch.from_numpy(wt).cuda(),
                 out_scale=0.4)
    o = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, True)
    assert_close(to_numpy(out), oracle.head_norm(o, "rms", 1e-5, wt, None, 0.4), "bf16", "decode rms")
    assert da.get_device_error() == 0


def test_decode_workloads_sampled():
    for w in W.DECODE_WORKLOADS.values():
        inp = W.draw_kv(w, B=2)      # two of the sequences, full cache length
        if w.shared_keys:
            inp.k2 = inp.k1
        out, _ = run(inp, w.dtype, w.lambda_value, w.causal)
        ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v,
                                               w.lambda_value, w.causal)
        assert_close(to_numpy(out), ref, w.dtype, w.name)


def test_decode_invalid_and_forward_routed_shapes():
    # more queries than keys under the causal mask: no alignment exists
    x = torch.zeros(1, 1, 9, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 5, 64, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(1, 1, 5, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(da.DiffattnError):
        da.differential_attention_decode(x, k, x, k, v, 0.5, causal=True)
    # Tq > 16 and D outside {32, 64, 128} run on the forward kernels, Tq = 9 on
    # the tensor-core decode in a unit of 16 rows: with V = 1 every output is
    # 1 - lambda
    for Tq, D in ((17, 64), (2, 48), (9, 64)):
        x = torch.zeros(1, 1, Tq, D, dtype=torch.bfloat16, device="cuda")
        k = torch.zeros(1, 1, 100, D, dtype=torch.bfloat16, device="cuda")
        v = torch.ones(1, 1, 100, 2 * D, dtype=torch.bfloat16, device="cuda")
        o = da.differential_attention_decode(x, k, x, k, v, 0.25)
        torch.cuda.synchronize()
        assert float((o.float() - 0.75).abs().max()) == 0.0


@pytest.mark.parametrize("H,Hk,Tq,Tk", [(2, 2, 4, 3000), (8, 2, 1, 2500), (3, 3, 8, 700)])
def test_decode_four_plus_rows_both_first_passes(H, Hk, Tq, Tk):
    """Four or more rows per key/value head (bf16, D = 64): a dense cache takes
    the tensor-core first pass, a token-major view of the same cache (rows not
    contiguous along the sequence) the CUDA-core pass; both match the oracle."""
    w = W.DecodeWorkload("t", 2, H, Tq, Tk, 64, "bf16", True, seed=H * 31 + Tq + Tk, kv_heads=Hk)
    inp = W.draw_kv(w)
    q1, q2 = to_device(inp.q1, "bf16"), to_device(inp.q2, "bf16")
    dense = [to_device(x, "bf16") for x in (inp.k1, inp.k2, inp.v)]
    # [B, Tk, Hk, *] storage seen as [B, Hk, Tk, *]
    token_major = [t.permute(0, 2, 1, 3).contiguous().permute(0, 2, 1, 3) for t in dense]
    if Hk > 1:
        assert token_major[0].stride(2) != token_major[0].shape[-1]
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, True)
    for kv, tag in ((dense, "dense"), (token_major, "token-major")):
        out = da.differential_attention_decode(q1, kv[0], q2, kv[1], kv[2], 0.6, causal=True)
        assert_close(to_numpy(out), ref, "bf16", f"decode {tag} H={H} Hk={Hk} Tq={Tq}")


@pytest.mark.parametrize("H,Hk,Tq,Tk,norm", [(4, 4, 4, 200, "rms"), (8, 2, 2, 5000, "group"),
                                             (6, 2, 2, 9000, "group"), (3, 3, 5, 1300, None)])
def test_decode_tensor_core_epilogue(H, Hk, Tq, Tk, norm):
    """Four or more rows per key/value head (the tensor-core first pass) with
    the combine's epilogue: a single split (Tk <= 256) and many, chunks with
    padded rows (3 heads x 2 rows or 5 rows in a chunk of 8), the norm with
    weight, bias and a device lambda, and two calls in a row on the cached
    workspace."""
    w = W.DecodeWorkload("t", 2, H, Tq, Tk, 64, "bf16", True, seed=H * 13 + Tq + Tk, kv_heads=Hk)
    inp = W.draw_kv(w)
    rng = np.random.default_rng(H + Tq)
    wt = (1 + 0.1 * rng.standard_normal((H, 128))).astype(np.float32)
    bs = (0.05 * rng.standard_normal((H, 128))).astype(np.float32)
    lam_t = torch.tensor(0.55, device="cuda")
    kw = dict(out_scale=0.7)
    if norm:
        kw.update(norm=norm, norm_weight=torch.from_numpy(wt).cuda(), norm_bias=torch.from_numpy(bs).cuda())
    o = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.55, True)
    ref = oracle.head_norm(o, norm or "none", 1e-5, wt if norm else None, bs if norm else None, 0.7)
    for call in range(2):
        out, _ = run(inp, "bf16", lam_t, True, **kw)
        assert_close(to_numpy(out), ref, "bf16", f"decode epilogue H={H} Hk={Hk} Tq={Tq} Tk={Tk} call {call}")
    assert da.get_device_error() == 0


def padded_rows(t):
    """The same cache with every row stored in a wider buffer (row stride
    D + 8 elements): not dense along the sequence, still 16-byte aligned."""
    B, H, T, W_ = t.shape
    wide = torch.zeros(B, H, T, W_ + 8, dtype=t.dtype, device=t.device)
    wide[..., :W_] = t
    return wide[..., :W_]


@pytest.mark.parametrize("H,Hk,Tq,Tk,causal", [
    (4, 1, 4, 3000, True),     # 16 rows per key/value head: 4 heads x 4 new queries
    (2, 1, 5, 1000, True),     # 10 rows
    (8, 1, 3, 777, False),     # 24 rows: two units of 12
    (2, 2, 12, 2000, True),    # Tq = 12, one query head per key/value head
    (1, 1, 16, 129, True),     # Tq = 16
    (16, 1, 1, 4096, True),    # 16 query heads per key/value head
    (32, 2, 2, 500, False),    # 32 rows per key/value head: two units of 16
])
def test_decode_sixteen_row_units(H, Hk, Tq, Tk, causal):
    """9 to 16 query rows per unit (bf16, D = 64): the tensor-core pass in units
    of 16 rows over a dense cache; over a cache with padded rows the split-key
    layout of 8-row units on the CUDA cores (Tq <= 8) or the forward kernels
    (Tq > 8).  All against the oracle."""
    w = W.DecodeWorkload("t16", 2, H, Tq, Tk, 64, "bf16", causal, seed=H * 7 + Tq * 3 + Tk, kv_heads=Hk)
    inp = W.draw_kv(w)
    q1, q2 = to_device(inp.q1, "bf16"), to_device(inp.q2, "bf16")
    dense = [to_device(x, "bf16") for x in (inp.k1, inp.k2, inp.v)]
    padded = [padded_rows(t) for t in dense]
    assert padded[0].stride(2) == 72
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, causal)
    for kv, tag in ((dense, "dense"), (padded, "padded rows")):
        out = da.differential_attention_decode(q1, kv[0], q2, kv[1], kv[2], 0.6, causal=causal)
        torch.cuda.synchronize()
        assert da.get_device_error() == 0
        assert_close(to_numpy(out), ref, "bf16", f"decode 16-row units {tag} H={H} Hk={Hk} Tq={Tq} Tk={Tk}")


@pytest.mark.parametrize("norm", ["rms", "group"])
def test_decode_sixteen_row_units_epilogue(norm):
    # 16 rows per unit with the norm epilogue and a device lambda, called twice
    w = W.DecodeWorkload("t16e", 2, 8, 4, 2500, 64, "bf16", True, seed=77, kv_heads=2)
    inp = W.draw_kv(w)
    rng = np.random.default_rng(9)
    wt = (1 + 0.1 * rng.standard_normal((8, 128))).astype(np.float32)
    bs = (0.05 * rng.standard_normal((8, 128))).astype(np.float32)
    lam_t = torch.tensor(0.45, device="cuda")
    o = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.45, True)
    ref = oracle.head_norm(o, norm, 1e-5, wt, bs, 0.5)
    for call in range(2):
        out, _ = run(inp, "bf16", lam_t, True, norm=norm, norm_weight=torch.from_numpy(wt).cuda(),
                     norm_bias=torch.from_numpy(bs).cuda(), out_scale=0.5)
        assert_close(to_numpy(out), ref, "bf16", f"decode 16-row units {norm} call {call}")
    assert da.get_device_error() == 0


def misaligned(x):
    """A bf16 copy of x seen one element into a wider buffer: element-aligned,
    not 16-byte aligned."""
    D = x.shape[-1]
    wide = torch.zeros(*x.shape[:-1], D + 8, dtype=torch.bfloat16, device="cuda")
    wide[..., 1:1 + D] = to_device(x, "bf16")
    return wide[..., 1:1 + D]


@pytest.mark.parametrize("H,Hk,Tq,Tk,D", [(4, 1, 4, 1500, 64), (2, 2, 12, 900, 64), (4, 2, 4, 700, 128)])
def test_decode_sixteen_row_shapes_with_misaligned_queries(H, Hk, Tq, Tk, D):
    """Queries whose rows are not 16-byte aligned: the tensor-core pass cannot
    take them; the split-key layout of 8-row units on the CUDA cores (D = 64,
    Tq <= 8) or the forward kernels run the call.  Against the oracle."""
    shared = D == 128
    w = W.DecodeWorkload("mis", 2, H, Tq, Tk, D, "bf16", True, seed=H + Tq + Tk + D, kv_heads=Hk,
                         value_dim=128, shared_keys=shared)
    inp = W.draw_kv(w)
    if shared:
        inp.k2 = inp.k1
    q1, q2 = misaligned(inp.q1), misaligned(inp.q2)
    assert q1.data_ptr() % 16 != 0
    k1, v = to_device(inp.k1, "bf16"), to_device(inp.v, "bf16")
    k2 = k1 if shared else to_device(inp.k2, "bf16")
    out = da.differential_attention_decode(q1, k1, q2, k2, v, 0.6, causal=True)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, True)
    assert_close(to_numpy(out), ref, "bf16", f"misaligned Q H={H} Hk={Hk} Tq={Tq} D={D}")


@pytest.mark.parametrize("B,H,Hk,Tq,Tk,causal", [(1, 1, 1, 16, 16, True), (2, 16, 1, 1, 1, True),
                                                 (1, 8, 1, 2, 2, True), (2, 4, 2, 8, 8, False)])
def test_decode_sixteen_row_units_edges(B, H, Hk, Tq, Tk, causal):
    # units of 16 rows at their edges: a cache holding exactly the new queries
    # (the first query sees one key), one cached key for 16 query heads
    w = W.DecodeWorkload("e16", B, H, Tq, Tk, 64, "bf16", causal, seed=B + H * 5 + Tq * 7 + Tk, kv_heads=Hk)
    inp = W.draw_kv(w)
    out, _ = run(inp, "bf16", 0.6, causal)
    torch.cuda.synchronize()
    assert da.get_device_error() == 0
    ref = oracle.differential_attention_kv(inp.q1, inp.k1, inp.q2, inp.k2, inp.v, 0.6, causal)
    assert_close(to_numpy(out), ref, "bf16", f"16-row edges B={B} H={H} Hk={Hk} Tq={Tq} Tk={Tk}")
