"""Differential-attention forward for NVIDIA GB300 (sm_103a).

Python binding over the C ABI in include/diffattn.h.  The two functions
mirror the interface of the paperleet "Differential Transformer Attention"
exercise (Functions to implement):

    differential_lambda(q1, k1, q2, k2, lambda_init=0.2) -> 0-d tensor
    differential_attention(q1, k1, q2, k2, value, coefficient, causal=True) -> tensor

This module only marshals arguments (shapes, strides, device pointers, the
current CUDA stream); every step of the computation runs in the library's
CUDA kernels.  There is no CPU path: without the built library, or for
tensors that are not on a CUDA device, the calls raise.
"""
from __future__ import annotations

import ctypes
import numbers
import warnings
from typing import Optional

import torch

from . import _lib
from ._lib import (DIFFATTN_BF16, DIFFATTN_F32, DIFFATTN_KERNEL_SIMT,  # noqa: F401
                   DIFFATTN_KERNEL_TCGEN05, DIFFATTN_NORM_GROUP, DIFFATTN_NORM_NONE,
                   DIFFATTN_NORM_RMS, DiffattnDesc, DiffattnEpilogue, DiffattnError,
                   DiffattnKvDesc)

__all__ = ["differential_lambda", "differential_attention", "differential_attention_host",
           "differential_attention_train",
           "differential_attention_backward",
           "differential_attention_decode",
           "make_desc", "make_kv_desc", "select_kernel", "get_device_error", "version",
           "DiffattnError"]

_DTYPES = {torch.bfloat16: DIFFATTN_BF16, torch.float32: DIFFATTN_F32}


def _stream_handle(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


_WORKSPACES = {}


def workspace_for(device: torch.device, stream) -> torch.Tensor:
    """The scheduler workspace for (device, stream): zero-filled once, left
    zeroed by every call, one per stream so concurrent streams never share."""
    key = (device.index, int(stream.cuda_stream))
    ws = _WORKSPACES.get(key)
    if ws is None:
        nbytes = int(_lib.load().diffattn_workspace_bytes())
        ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=device)
        _WORKSPACES[key] = ws
    return ws


def _require_cuda(t: torch.Tensor, name: str) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device}); there is no CPU path")


def version() -> int:
    return _lib.load().diffattn_version()


def differential_lambda(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor, k2: torch.Tensor,
                        lambda_init: float = 0.2) -> torch.Tensor:
    """lambda = exp(q1 . k1) - exp(q2 . k2) + lambda_init as a 0-d tensor.

    q1, k1, q2, k2 are the four lambda parameter vectors [D_lambda] (equal
    length, non-empty) on one CUDA device.  The result is float32 on that
    device, computed in float64 by the library's kernel.  When grad mode is on
    and a vector requires grad, the result carries an autograd node whose
    backward runs diffattn_lambda_backward.
    """
    if torch.is_grad_enabled() and any(isinstance(t, torch.Tensor) and t.requires_grad
                                       for t in (q1, k1, q2, k2)):
        return _DifferentialLambdaFn.apply(q1, k1, q2, k2, lambda_init)
    return _lambda_forward(q1, k1, q2, k2, lambda_init)


def _lambda_forward(q1, k1, q2, k2, lambda_init):
    vecs = []
    for name, t in (("q1", q1), ("k1", k1), ("q2", q2), ("k2", k2)):
        _require_cuda(t, name)
        if t.dim() != 1:
            raise ValueError(f"{name} must be a 1-D parameter vector")
        vecs.append(t.detach().to(torch.float32).contiguous())
    n = vecs[0].numel()
    if n == 0 or any(v.numel() != n for v in vecs):
        raise ValueError("lambda vectors must be non-empty and of equal length")
    dev = vecs[0].device
    if any(v.device != dev for v in vecs):
        raise ValueError("lambda vectors must be on one device")
    out = torch.empty((), dtype=torch.float32, device=dev)
    lib = _lib.load()
    with torch.cuda.device(dev):
        rc = lib.diffattn_lambda(*(ctypes.c_void_p(v.data_ptr()) for v in vecs), n,
                                 float(lambda_init), ctypes.c_void_p(out.data_ptr()),
                                 _stream_handle(dev))
    _lib.check(rc, "diffattn_lambda")
    return out


def make_desc(q1, k1, q2, k2, v, out) -> DiffattnDesc:
    """Fill a diffattn_desc from tensors (sizes, dtype, B/H/T element strides;
    kv_group = query heads per key/value head)."""
    B, H, T, D = q1.shape
    d = DiffattnDesc()
    d.B, d.H, d.T, d.D = B, H, T, D
    d.Dv = v.shape[-1]
    d.dtype = _DTYPES[q1.dtype]
    d.kv_group = H // k1.shape[1]
    for field, t in (("q1_stride", q1), ("k1_stride", k1), ("q2_stride", q2), ("k2_stride", k2),
                     ("v_stride", v), ("o_stride", out)):
        s = t.stride()
        getattr(d, field)[:] = (s[0], s[1], s[2])
    return d


_WARNED_SLOW = set()


def _warn_if_cuda_cores(lib, d, ptrs, what: str) -> None:
    """Warn once per call site when a bf16 call of a shape the tensor-core
    kernel takes (value width 128 with D = 64 or 128) runs on the CUDA-core
    kernel instead, because a base pointer or a stride is not 16-byte aligned
    (or a stride is 0)."""
    tc_shape = (d.D == 64 and d.Dv in (0, 128)) or (d.D == 128 and d.Dv == 128)
    if d.dtype != DIFFATTN_BF16 or not tc_shape or what in _WARNED_SLOW:
        return
    if lib.diffattn_select_kernel(ctypes.byref(d), *ptrs) == DIFFATTN_KERNEL_SIMT:
        _WARNED_SLOW.add(what)
        warnings.warn(f"{what}: a bf16 call of a tensor-core shape runs on the CUDA-core kernel because a base "
                      "pointer or stride is not 16-byte aligned (or a stride is 0); pass "
                      "16-byte-aligned tensors for the tensor-core kernel", RuntimeWarning,
                      stacklevel=3)


def _prepare(q1, k1, q2, k2, value):
    ts = [q1, k1, q2, k2, value]
    names = ["q1", "k1", "q2", "k2", "value"]
    for n, t in zip(names, ts):
        _require_cuda(t, n)
        if t.dim() != 4:
            raise ValueError(f"{n} must be 4-D [B, H, T, *]")
    if q1.shape != q2.shape or k1.shape != k2.shape:
        raise ValueError("q1, q2 must share one shape [B, H, T, D], and k1, k2 another")
    B, H, T, D = q1.shape
    Hk = k1.shape[1]
    if k1.shape[0] != B or tuple(k1.shape[2:]) != (T, D) or Hk < 1 or H % Hk != 0:
        raise ValueError(f"k1, k2 must be [B, H_kv, T, D] with H_kv dividing H = {H}, "
                         f"got {tuple(k1.shape)}")
    if tuple(value.shape[:3]) != (B, Hk, T) or not 1 <= value.shape[3] <= 256:
        raise ValueError(f"value must be [B, H_kv, T, Dv] = {(B, Hk, T)} + (Dv <= 256,) (Dv = 2D "
                         f"is the operation's own shape), got {tuple(value.shape)}")
    dt = q1.dtype
    if dt not in _DTYPES:
        raise ValueError(f"unsupported dtype {dt}; expected bfloat16 or float32")
    if any(t.dtype != dt for t in ts):
        raise ValueError("all inputs must share one dtype")
    dev = q1.device
    if any(t.device != dev for t in ts):
        raise ValueError("all inputs must be on one device")
    # The ABI wants a contiguous innermost dimension; other strides pass through.
    ts = [t if t.stride(-1) == 1 or t.shape[-1] == 1 else t.contiguous() for t in ts]
    return ts, dev


def select_kernel(q1, k1, q2, k2, value, out=None) -> int:
    """Which kernel differential_attention would launch (DIFFATTN_KERNEL_*)."""
    (q1, k1, q2, k2, value), dev = _prepare(q1, k1, q2, k2, value)
    if out is None:
        out = torch.empty_like(value, memory_format=torch.contiguous_format)
    d = make_desc(q1, k1, q2, k2, value, out)
    rc = _lib.load().diffattn_select_kernel(ctypes.byref(d), *(ctypes.c_void_p(t.data_ptr()) for t in
                                                               (q1, k1, q2, k2, value, out)))
    if rc < 0:
        _lib.check(rc, "diffattn_select_kernel")
    return rc


def differential_attention(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor, k2: torch.Tensor,
                           value: torch.Tensor, coefficient, causal: bool = True,
                           out: Optional[torch.Tensor] = None,
                           dynamic_schedule: bool = True, norm: Optional[str] = None,
                           norm_eps: float = 1e-5, norm_weight: Optional[torch.Tensor] = None,
                           norm_bias: Optional[torch.Tensor] = None,
                           out_scale: float = 1.0) -> torch.Tensor:
    """O = (softmax(Q1 K1^T/sqrt(D) + M) - lambda softmax(Q2 K2^T/sqrt(D) + M)) V.

    q1, q2: [B, H, T, D]; k1, k2: [B, H_kv, T, D]; value: [B, H_kv, T, Dv]
    with Dv = 2D (the operation's own shape) or any width up to 256 (Dv = D
    is the DIFF V2 head; D = 128, Dv = 128 runs on the tensor cores too);
    all bfloat16 or all float32 on one CUDA device, innermost dimension
    contiguous (other strides are passed through).  H_kv must divide H: query
    head h reads key/value head h // (H // H_kv) (grouped key/value heads;
    H_kv = H is the plain layout).  Passing the same tensor as k1 and k2
    shares the keys between the branches.  coefficient: lambda, a Python number or a scalar
    tensor (a CUDA float32 scalar is read by the kernel without a host sync).
    causal: mask key j > query i in both branches.  out: optional preallocated
    [B, H, T, Dv] output of the same dtype.  dynamic_schedule: hand out work
    items at run time through a small per-stream workspace (the result is
    the same either way).

    Optional fused epilogue (the step after the operation in the model):
    norm "rms" or "group" normalises each (b, h, t) row over the head's Dv
    channels (eps norm_eps), then multiplies by norm_weight and adds
    norm_bias ([H, Dv] float32 tensors, optional), and finally scales by
    out_scale (e.g. 1 - lambda_init).

    Returns the [B, H, T, Dv] output; the launch is asynchronous on the
    current CUDA stream.  When grad mode is on and an input or a tensor
    coefficient requires grad, the result carries an autograd node whose
    backward runs diffattn_bwd (no epilogue and no `out` then).
    """
    if torch.is_grad_enabled() and any(
            isinstance(t, torch.Tensor) and t.requires_grad
            for t in (q1, k1, q2, k2, value, coefficient)):
        if out is not None or norm not in (None, "none") or norm_weight is not None or \
                norm_bias is not None or out_scale != 1.0:
            raise ValueError("gradients are available for the bare operation only "
                             "(no out=, norm or out_scale)")
        return _DifferentialAttentionFn.apply(q1, k1, q2, k2, value, coefficient, causal,
                                              dynamic_schedule)
    return _forward(q1, k1, q2, k2, value, coefficient, causal, out, dynamic_schedule, norm,
                    norm_eps, norm_weight, norm_bias, out_scale)


def _forward(q1, k1, q2, k2, value, coefficient, causal, out, dynamic_schedule, norm, norm_eps,
             norm_weight, norm_bias, out_scale, train=False):
    (q1, k1, q2, k2, value), dev = _prepare(q1, k1, q2, k2, value)
    B, H, T, D = q1.shape
    Dv = value.shape[3]
    if out is None:
        out = torch.empty((B, H, T, Dv), dtype=q1.dtype, device=dev)
    else:
        _require_cuda(out, "out")
        if tuple(out.shape) != (B, H, T, Dv) or out.dtype != q1.dtype or out.device != dev:
            raise ValueError("out must be [B, H, T, Dv] with the inputs' dtype and device")
        if out.stride(-1) != 1:
            raise ValueError("out must have a contiguous innermost dimension")
    lam_host, lam_dev = _coefficient(coefficient, dev)
    d = make_desc(q1, k1, q2, k2, value, out)
    epi = _epilogue(norm, norm_eps, norm_weight, norm_bias, out_scale, H, Dv, dev)
    lib = _lib.load()
    lam_ptr = ctypes.c_void_p(lam_dev.data_ptr() if lam_dev is not None else 0)
    ins = [ctypes.c_void_p(t.data_ptr()) for t in (q1, k1, q2, k2, value)]
    _warn_if_cuda_cores(lib, d, ins + [ctypes.c_void_p(out.data_ptr())], "differential_attention")
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        ws = workspace_for(dev, stream) if dynamic_schedule else None
        ws_args = (ctypes.c_void_p(ws.data_ptr() if ws is not None else 0),
                   ctypes.c_size_t(ws.numel() * 4 if ws is not None else 0),
                   ctypes.c_void_p(stream.cuda_stream))
        if train:
            out2 = torch.empty_like(out)
            lse = torch.empty((B, H, T, 2), dtype=torch.float32, device=dev)
            rc = lib.diffattn_fwd_train(ctypes.byref(d), *ins, ctypes.c_float(lam_host), lam_ptr,
                                        1 if causal else 0, ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(out2.data_ptr()),
                                        ctypes.c_void_p(lse.data_ptr()), *ws_args)
            _lib.check(rc, "diffattn_fwd_train")
            return out, out2, lse
        rc = lib.diffattn_fwd_ex(ctypes.byref(d), *ins, ctypes.c_float(lam_host), lam_ptr,
                                 1 if causal else 0, ctypes.byref(epi[0]) if epi else None,
                                 ctypes.c_void_p(out.data_ptr()), *ws_args)
    _lib.check(rc, "diffattn_fwd")
    return out


def differential_attention_host(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor,
                                k2: torch.Tensor, value: torch.Tensor, coefficient,
                                causal: bool = True, out: Optional[torch.Tensor] = None,
                                device=None, buffers=None) -> torch.Tensor:
    """differential_attention for inputs in host memory (CPU tensors,
    preferably pinned): the library copies them to the device, runs the
    forward and copies the output back, overlapping the copies of one chunk of
    heads with the forward of another.  Returns the [B, H, T, Dv] output on
    the host (`out`, a pinned CPU tensor, if given).  `buffers`: optional
    device tensors (q1, k1, q2, k2, value, out) to reuse between calls.  The
    result is ready when the current stream of `device` has completed."""
    ts = [q1, k1, q2, k2, value]
    if any(t.device.type != "cpu" for t in ts):
        raise ValueError("differential_attention_host takes CPU tensors")
    ts = [t.contiguous() for t in ts]
    q1, k1, q2, k2, value = ts
    B, H, T, D = q1.shape
    Dv = value.shape[3]
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if out is None:
        out = torch.empty((B, H, T, Dv), dtype=q1.dtype).pin_memory()
    if buffers is None:
        dk1 = torch.empty(k1.shape, dtype=k1.dtype, device=dev)
        buffers = [torch.empty(q1.shape, dtype=q1.dtype, device=dev), dk1,
                   torch.empty(q2.shape, dtype=q2.dtype, device=dev),
                   dk1 if k2 is k1 else torch.empty(k2.shape, dtype=k2.dtype, device=dev),
                   torch.empty(value.shape, dtype=value.dtype, device=dev),
                   torch.empty((B, H, T, Dv), dtype=q1.dtype, device=dev)]
    lam_host, lam_dev = _coefficient(coefficient, dev)
    d = make_desc(*buffers[:5], buffers[5])
    lib = _lib.load()
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        ws = workspace_for(dev, stream)
        rc = lib.diffattn_fwd_host(ctypes.byref(d), *(ctypes.c_void_p(t.data_ptr()) for t in ts),
                                   ctypes.c_float(lam_host),
                                   ctypes.c_void_p(lam_dev.data_ptr() if lam_dev is not None else 0),
                                   1 if causal else 0, ctypes.c_void_p(out.data_ptr()),
                                   *(ctypes.c_void_p(t.data_ptr()) for t in buffers),
                                   ctypes.c_void_p(ws.data_ptr()), ctypes.c_size_t(ws.numel() * 4),
                                   ctypes.c_void_p(stream.cuda_stream))
    _lib.check(rc, "diffattn_fwd_host")
    return out


def differential_attention_train(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor,
                                 k2: torch.Tensor, value: torch.Tensor, coefficient,
                                 causal: bool = True, dynamic_schedule: bool = True):
    """The forward of a training step: returns (out, out2, lse) where out is
    differential_attention's output, out2 = A_2 V (same shape and dtype) and
    lse the natural-log log-sum-exp of each branch's scaled scores, float32
    [B, H, T, 2].  Pass them to differential_attention_backward(saved=...)."""
    return _forward(q1, k1, q2, k2, value, coefficient, causal, None, dynamic_schedule, None,
                    1e-5, None, None, 1.0, train=True)


def differential_attention_backward(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor,
                                    k2: torch.Tensor, value: torch.Tensor, coefficient,
                                    dout: torch.Tensor, causal: bool = True, saved=None):
    """Gradients of differential_attention given dout = dL/dO.

    Inputs as differential_attention (the forward's inputs and coefficient);
    dout: [B, H, T, Dv] of the inputs' dtype (Dv the width of value; the
    tensor cores take bf16 with D = 64 and Dv = 2D, other shapes run on the
    CUDA cores).  saved: optional (out, out2,
    lse) from differential_attention_train with the same inputs; with it the
    forward is not recomputed.  Returns (dq1, dk1, dq2, dk2, dvalue,
    dcoefficient): contiguous tensors of the inputs' shapes and dtype, and a
    float32 scalar tensor on the device.  The gradients of the four lambda
    vectors follow from dcoefficient (see differential_lambda)."""
    (q1, k1, q2, k2, value), dev = _prepare(q1, k1, q2, k2, value)
    B, H, T, D = q1.shape
    Dv = value.shape[3]
    _require_cuda(dout, "dout")
    if tuple(dout.shape) != (B, H, T, Dv) or dout.dtype != q1.dtype or dout.device != dev:
        raise ValueError("dout must be [B, H, T, Dv] with the inputs' dtype and device")
    if dout.stride(-1) != 1:
        dout = dout.contiguous()
    if saved is not None:
        out, out2, lse = saved
        # out, out2 and dout share one layout in the ABI
        if dout.stride() != out.stride():
            dout = dout.contiguous()
            out, out2 = out.contiguous(), out2.contiguous()
        if out2.stride() != out.stride():
            out2 = out2.contiguous()
        if tuple(lse.shape) != (B, H, T, 2) or lse.dtype != torch.float32 or not lse.is_contiguous():
            raise ValueError("lse must be a contiguous float32 [B, H, T, 2] tensor")
        if out.dtype != q1.dtype or out2.dtype != q1.dtype or out.shape != dout.shape or \
                out2.shape != dout.shape:
            raise ValueError("out and out2 must match dout's shape and dtype")
    lam_host, lam_dev = _coefficient(coefficient, dev)
    d = make_desc(q1, k1, q2, k2, value, dout)
    grads = [torch.empty(t.shape, dtype=t.dtype, device=dev) for t in (q1, k1, q2, k2, value)]
    dlam = torch.empty((), dtype=torch.float32, device=dev)
    lib = _lib.load()
    need = int(lib.diffattn_bwd_workspace_bytes(ctypes.byref(d)))
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        ws = torch.empty(need // 4 + 4, dtype=torch.float32, device=dev)
        head = [ctypes.byref(d), *(ctypes.c_void_p(t.data_ptr()) for t in (q1, k1, q2, k2, value)),
                ctypes.c_float(lam_host),
                ctypes.c_void_p(lam_dev.data_ptr() if lam_dev is not None else 0),
                1 if causal else 0]
        tail = [ctypes.c_void_p(dout.data_ptr()), *(ctypes.c_void_p(g.data_ptr()) for g in grads),
                ctypes.c_void_p(dlam.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                ctypes.c_size_t(ws.numel() * 4), ctypes.c_void_p(stream.cuda_stream)]
        if saved is not None:
            rc = lib.diffattn_bwd_saved(*head, ctypes.c_void_p(out.data_ptr()),
                                        ctypes.c_void_p(out2.data_ptr()),
                                        ctypes.c_void_p(lse.data_ptr()), *tail)
        else:
            rc = lib.diffattn_bwd(*head, *tail)
    _lib.check(rc, "diffattn_bwd")
    return (*grads, dlam)


class _DifferentialAttentionFn(torch.autograd.Function):
    """Autograd node: forward through diffattn_fwd, backward through diffattn_bwd."""

    @staticmethod
    def forward(ctx, q1, k1, q2, k2, value, coefficient, causal, dynamic_schedule):
        out, out2, lse = _forward(q1, k1, q2, k2, value, coefficient, causal, None,
                                  dynamic_schedule, None, 1e-5, None, None, 1.0, train=True)
        coef_t = coefficient if isinstance(coefficient, torch.Tensor) else None
        ctx.save_for_backward(q1, k1, q2, k2, value, coef_t, out, out2, lse)
        ctx.coefficient = None if coef_t is not None else coefficient
        ctx.causal = causal
        return out

    @staticmethod
    def backward(ctx, dout):
        q1, k1, q2, k2, value, coef_t, out, out2, lse = ctx.saved_tensors
        coefficient = coef_t if coef_t is not None else ctx.coefficient
        dq1, dk1, dq2, dk2, dv, dlam = differential_attention_backward(
            q1, k1, q2, k2, value, coefficient, dout.to(q1.dtype), ctx.causal,
            saved=(out, out2, lse))
        dcoef = None
        if coef_t is not None and ctx.needs_input_grad[5]:
            dcoef = dlam.to(device=coef_t.device, dtype=coef_t.dtype).reshape(coef_t.shape)
        return dq1, dk1, dq2, dk2, dv, dcoef, None, None


class _DifferentialLambdaFn(torch.autograd.Function):
    """Autograd node: forward through diffattn_lambda, backward through
    diffattn_lambda_backward."""

    @staticmethod
    def forward(ctx, q1, k1, q2, k2, lambda_init):
        out = _lambda_forward(q1, k1, q2, k2, lambda_init)
        ctx.save_for_backward(q1, k1, q2, k2)
        return out

    @staticmethod
    def backward(ctx, dlam):
        vecs = [t.detach().to(torch.float32).contiguous() for t in ctx.saved_tensors]
        grads = [torch.empty_like(v) for v in vecs]
        g = dlam.detach().to(device=vecs[0].device, dtype=torch.float32).reshape(()).contiguous()
        dev = vecs[0].device
        with torch.cuda.device(dev):
            rc = _lib.load().diffattn_lambda_backward(
                *(ctypes.c_void_p(v.data_ptr()) for v in vecs), vecs[0].numel(),
                ctypes.c_void_p(g.data_ptr()), *(ctypes.c_void_p(x.data_ptr()) for x in grads),
                _stream_handle(dev))
        _lib.check(rc, "diffattn_lambda_backward")
        return (*(x.to(t.dtype) for x, t in zip(grads, ctx.saved_tensors)), None)


def _coefficient(coefficient, dev):
    """(host lambda, device lambda tensor or None) from a number or scalar tensor."""
    if isinstance(coefficient, torch.Tensor):
        if coefficient.numel() != 1:
            raise ValueError("coefficient must be a scalar")
        if coefficient.device.type == "cuda":
            if coefficient.device != dev:
                raise ValueError("coefficient tensor must be on the inputs' device")
            return 0.0, coefficient.detach().reshape(()).to(torch.float32)
        return float(coefficient.item()), None
    if isinstance(coefficient, numbers.Real):
        return float(coefficient), None
    raise TypeError("coefficient must be a real number or a scalar tensor")


def make_kv_desc(q1, k1, q2, k2, v, out) -> DiffattnKvDesc:
    """Fill a diffattn_kv_desc from tensors."""
    B, H, Tq, D = q1.shape
    d = DiffattnKvDesc()
    d.B, d.H, d.Tq, d.Tk, d.D = B, H, Tq, k1.shape[2], D
    d.Dv = v.shape[-1]
    d.dtype = _DTYPES[q1.dtype]
    d.kv_group = H // k1.shape[1]
    for field, t in (("q1_stride", q1), ("k1_stride", k1), ("q2_stride", q2), ("k2_stride", k2),
                     ("v_stride", v), ("o_stride", out)):
        s = t.stride()
        getattr(d, field)[:] = (s[0], s[1], s[2])
    return d


_DECODE_WS = {}


def decode_workspace_for(device: torch.device, stream, nbytes: int) -> torch.Tensor:
    """A per-(device, stream) decode workspace of at least nbytes (grown on
    demand; its contents need no initialisation)."""
    key = (device.index, int(stream.cuda_stream))
    ws = _DECODE_WS.get(key)
    if ws is None or ws.numel() * 4 < nbytes:
        ws = torch.empty((nbytes + 15) // 4 + 4, dtype=torch.float32, device=device)
        _DECODE_WS[key] = ws
    return ws


def differential_attention_decode(q1: torch.Tensor, k1: torch.Tensor, q2: torch.Tensor,
                                  k2: torch.Tensor, value: torch.Tensor, coefficient,
                                  causal: bool = True, out: Optional[torch.Tensor] = None,
                                  norm: Optional[str] = None, norm_eps: float = 1e-5,
                                  norm_weight: Optional[torch.Tensor] = None,
                                  norm_bias: Optional[torch.Tensor] = None,
                                  out_scale: float = 1.0) -> torch.Tensor:
    """Queries over a key/value cache: Tq new queries q1, q2 [B, H, Tq, D]
    over cached keys k1, k2 [B, H_kv, Tk, D] and values [B, H_kv, Tk, Dv]
    (H_kv dividing H; query head h reads key/value head h // (H // H_kv);
    Dv = 2D is the operation's own shape).  With causal=True query i sits at
    position Tk - Tq + i.  A few queries (a decode step) run on the split-key
    decode kernels; more (a chunk of a prefill) on the forward kernels.
    Epilogue arguments as differential_attention.  Returns [B, H, Tq, Dv].
    (Forward only.)"""
    ts = [q1, k1, q2, k2, value]
    for n, t in zip(("q1", "k1", "q2", "k2", "value"), ts):
        _require_cuda(t, n)
        if t.dim() != 4:
            raise ValueError(f"{n} must be 4-D")
    B, H, Tq, D = q1.shape
    Hk, Tk = k1.shape[1], k1.shape[2]
    if q2.shape != q1.shape or k1.shape != k2.shape or tuple(k1.shape) != (B, Hk, Tk, D) or \
            H % Hk != 0 or tuple(value.shape[:3]) != (B, Hk, Tk) or not 1 <= value.shape[3] <= 256:
        raise ValueError("expected q1, q2 [B, H, Tq, D], k1, k2 [B, H_kv, Tk, D], "
                         "value [B, H_kv, Tk, Dv] with H_kv dividing H and Dv <= 256")
    Dv = value.shape[3]
    dt, dev = q1.dtype, q1.device
    if dt not in _DTYPES or any(t.dtype != dt or t.device != dev for t in ts):
        raise ValueError("inputs must share one dtype (bfloat16 or float32) and device")
    ts = [t if t.stride(-1) == 1 else t.contiguous() for t in ts]
    q1, k1, q2, k2, value = ts
    if out is None:
        out = torch.empty((B, H, Tq, Dv), dtype=dt, device=dev)
    lam_host, lam_dev = 0.0, None
    if isinstance(coefficient, torch.Tensor):
        if coefficient.device.type == "cuda":
            lam_dev = coefficient.detach().reshape(()).to(torch.float32)
        else:
            lam_host = float(coefficient.item())
    else:
        lam_host = float(coefficient)
    d = make_kv_desc(q1, k1, q2, k2, value, out)
    epi = _epilogue(norm, norm_eps, norm_weight, norm_bias, out_scale, H, Dv, dev)
    lib = _lib.load()
    need = int(lib.diffattn_decode_workspace_bytes(ctypes.byref(d)))
    if need == 0:
        raise DiffattnError(_lib.DIFFATTN_ERR_UNSUPPORTED, "diffattn_decode_workspace_bytes")
    with torch.cuda.device(dev):
        stream = torch.cuda.current_stream(dev)
        ws = decode_workspace_for(dev, stream, need)
        rc = lib.diffattn_decode(ctypes.byref(d), *(ctypes.c_void_p(t.data_ptr()) for t in ts),
                                 ctypes.c_float(lam_host),
                                 ctypes.c_void_p(lam_dev.data_ptr() if lam_dev is not None else 0),
                                 1 if causal else 0, ctypes.byref(epi[0]) if epi else None,
                                 ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(ws.data_ptr()),
                                 ctypes.c_size_t(ws.numel() * 4), ctypes.c_void_p(stream.cuda_stream))
    _lib.check(rc, "diffattn_decode")
    return out


_NORMS = {None: DIFFATTN_NORM_NONE, "none": DIFFATTN_NORM_NONE, "rms": DIFFATTN_NORM_RMS,
          "group": DIFFATTN_NORM_GROUP}


def _epilogue(norm, eps, weight, bias, out_scale, H, Dv, dev):
    """diffattn_epilogue for the call (None when there is nothing to apply);
    returns (struct, tensors kept alive for the launch)."""
    if norm not in _NORMS:
        raise ValueError(f"norm must be one of {sorted(k for k in _NORMS if k)}, got {norm!r}")
    code = _NORMS[norm]
    if code == DIFFATTN_NORM_NONE and weight is None and bias is None and out_scale == 1.0:
        return None
    keep = []
    ptrs = []
    for name, t in (("norm_weight", weight), ("norm_bias", bias)):
        if t is None:
            ptrs.append(0)
            continue
        _require_cuda(t, name)
        if t.device != dev or tuple(t.shape) not in ((H, Dv), (H * Dv,)):
            raise ValueError(f"{name} must be [H, Dv] = {(H, Dv)} on the inputs' device")
        t = t.detach().to(torch.float32).contiguous()
        keep.append(t)
        ptrs.append(t.data_ptr())
    e = DiffattnEpilogue()
    e.norm, e.eps, e.out_scale, e.reserved = code, float(eps), float(out_scale), 0
    e.weight, e.bias = ptrs
    return e, keep


def get_device_error(device=None) -> int:
    """Synchronise the current stream and return the library's device status
    (0, or DIFFATTN_ERR_TIMEOUT if a kernel's bounded wait ran out)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return _lib.load().diffattn_get_device_error(_stream_handle(dev))
