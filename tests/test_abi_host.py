"""Host-side checks of the C ABI: the library builds, loads and exports every
symbol include/diffattn.h declares; argument checks reject bad calls before
any CUDA call (so these run without a GPU); kernel selection is host logic."""
import ctypes
import os
import re

import pytest

from differential_attention_fwd_gb300 import _lib
from differential_attention_fwd_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "diffattn.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(diffattn_\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), f"missing export {n}"


def test_desc_layout_matches_header():
    # 4 x int64, 2 x int32, 6 x int64[3], then Dv (int64) last
    assert ctypes.sizeof(_lib.DiffattnDesc) == 4 * 8 + 2 * 4 + 6 * 3 * 8 + 8
    assert _lib.DiffattnDesc.Dv.offset == 4 * 8 + 2 * 4 + 6 * 3 * 8
    assert ctypes.sizeof(_lib.DiffattnKvDesc) == 5 * 8 + 2 * 4 + 6 * 3 * 8 + 8


def test_version_and_strerror(lib):
    assert lib.diffattn_version() == 200
    for code in (0, -1, -2, -3, -4, 7):
        assert isinstance(lib.diffattn_strerror(code), bytes)
    assert lib.diffattn_strerror(-4) != lib.diffattn_strerror(0)


FAKE = 0x10000  # 64 KiB-aligned stand-in addresses; never dereferenced on the host path


def desc(B=1, H=2, T=128, D=64, dtype=_lib.DIFFATTN_BF16, contiguous=True, kv_group=0, Dv=0):
    d = _lib.DiffattnDesc()
    d.B, d.H, d.T, d.D, d.dtype, d.kv_group = B, H, T, D, dtype, kv_group
    d.Dv = Dv
    Hk = H // max(kv_group, 1)
    wv = Dv or 2 * D
    for f, w, h in (("q1_stride", D, H), ("k1_stride", D, Hk), ("q2_stride", D, H),
                    ("k2_stride", D, Hk), ("v_stride", wv, Hk), ("o_stride", wv, H)):
        getattr(d, f)[:] = (h * T * w, T * w, w)
    return d


def ptrs(n=6, base=FAKE):
    return [ctypes.c_void_p(base * (i + 1)) for i in range(n)]


def select(lib, d, p=None):
    p = p or ptrs()
    return lib.diffattn_select_kernel(ctypes.byref(d), *p)


def test_select_tcgen05_for_aligned_bf16_d64(lib):
    assert select(lib, desc()) == _lib.DIFFATTN_KERNEL_TCGEN05


@pytest.mark.parametrize("kw", [dict(D=32), dict(D=128), dict(D=48), dict(dtype=_lib.DIFFATTN_F32),
                                dict(D=64, Dv=64), dict(D=128, Dv=64), dict(D=96, Dv=128),
                                dict(D=128, Dv=128, dtype=_lib.DIFFATTN_F32)])
def test_select_simt_otherwise(lib, kw):
    assert select(lib, desc(**kw)) == _lib.DIFFATTN_KERNEL_SIMT


@pytest.mark.parametrize("kw", [dict(D=64, Dv=128), dict(D=128, Dv=128), dict(D=64)])
def test_select_tcgen05_for_value_width_128(lib, kw):
    # the tensor-core kernel's value width is 128: V = 2D at D = 64 (Dv 0 or
    # 128), and the DIFF V2 head D = Dv = 128
    assert select(lib, desc(**kw)) == _lib.DIFFATTN_KERNEL_TCGEN05


def test_value_width_rejected_out_of_range(lib):
    for dv in (-1, 257):
        assert select(lib, desc(Dv=dv)) == _lib.DIFFATTN_ERR_INVALID


def test_select_simt_for_unaligned(lib):
    p = ptrs()
    p[2] = ctypes.c_void_p(FAKE * 3 + 2)   # q2 not 16-byte aligned
    assert select(lib, desc(), p) == _lib.DIFFATTN_KERNEL_SIMT
    d = desc()
    d.v_stride[2] = 132                     # row stride not a multiple of 8 elements
    assert select(lib, d) == _lib.DIFFATTN_KERNEL_SIMT


def test_size_one_dims_ignore_strides(lib):
    d = desc(B=1, H=1, T=1)
    for f in ("q1_stride", "k1_stride", "q2_stride", "k2_stride", "v_stride", "o_stride"):
        getattr(d, f)[:] = (0, 0, 3)
    assert select(lib, d) == _lib.DIFFATTN_KERNEL_TCGEN05


@pytest.mark.parametrize("mutate", [
    lambda d: setattr(d, "B", 0),
    lambda d: setattr(d, "H", 0),
    lambda d: setattr(d, "T", 0),
    lambda d: setattr(d, "D", 0),
    lambda d: setattr(d, "D", 129),
    lambda d: setattr(d, "dtype", 2),
    lambda d: setattr(d, "kv_group", -1),
    lambda d: setattr(d, "kv_group", 3),      # does not divide H = 2
    lambda d: d.k2_stride.__setitem__(1, -1),
])
def test_invalid_desc_rejected_without_gpu(lib, mutate):
    d = desc()
    mutate(d)
    assert select(lib, d) == _lib.DIFFATTN_ERR_INVALID
    rc = lib.diffattn_fwd(ctypes.byref(d), *ptrs(5), ctypes.c_float(0.5), None, 1,
                          ctypes.c_void_p(FAKE * 9), None, 0, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID


def test_null_pointers_rejected(lib):
    d = desc()
    for i in range(6):
        p = ptrs()
        p[i] = None
        assert lib.diffattn_select_kernel(ctypes.byref(d), *p) == _lib.DIFFATTN_ERR_INVALID
    assert lib.diffattn_fwd(None, *ptrs(5), ctypes.c_float(0.5), None, 1, ctypes.c_void_p(FAKE),
                            None, 0, None) == _lib.DIFFATTN_ERR_INVALID


@pytest.mark.parametrize("lam", [float("nan"), float("inf"), -float("inf")])
def test_non_finite_lambda_rejected(lib, lam):
    rc = lib.diffattn_fwd(ctypes.byref(desc()), *ptrs(5), ctypes.c_float(lam), None, 1,
                          ctypes.c_void_p(FAKE * 9), None, 0, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID


def test_bad_workspace_rejected(lib):
    need = lib.diffattn_workspace_bytes()
    assert 8 <= need <= 4096
    ws = ctypes.c_void_p(FAKE * 11)
    rc = lib.diffattn_fwd(ctypes.byref(desc()), *ptrs(5), ctypes.c_float(0.5), None, 1,
                          ctypes.c_void_p(FAKE * 9), ws, need - 4, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID
    rc = lib.diffattn_fwd(ctypes.byref(desc()), *ptrs(5), ctypes.c_float(0.5), None, 1,
                          ctypes.c_void_p(FAKE * 9), ctypes.c_void_p(FAKE * 11 + 2), need, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID


def test_oversized_rejected(lib):
    d = desc(B=1 << 20, H=1 << 20, T=1 << 20)
    assert select(lib, d) == _lib.DIFFATTN_ERR_UNSUPPORTED


def test_lambda_args_rejected(lib):
    p = ptrs(5)
    assert lib.diffattn_lambda(p[0], p[1], p[2], p[3], 0, 0.2, p[4], None) == _lib.DIFFATTN_ERR_INVALID
    assert lib.diffattn_lambda(None, p[1], p[2], p[3], 4, 0.2, p[4], None) == _lib.DIFFATTN_ERR_INVALID
    assert lib.diffattn_lambda(p[0], p[1], p[2], p[3], 4, float("nan"), p[4], None) == _lib.DIFFATTN_ERR_INVALID
    assert lib.diffattn_lambda(p[0], p[1], p[2], p[3], 4, 0.2, None, None) == _lib.DIFFATTN_ERR_INVALID


def test_binding_rejects_cpu_tensors():
    import torch
    import differential_attention_fwd_gb300 as da
    x = torch.zeros(1, 1, 4, 8)
    v = torch.zeros(1, 1, 4, 16)
    with pytest.raises(ValueError, match="CUDA"):
        da.differential_attention(x, x, x, x, v, 0.5)
    with pytest.raises(ValueError, match="CUDA"):
        da.differential_lambda(torch.zeros(4), torch.zeros(4), torch.zeros(4), torch.zeros(4))


@pytest.mark.parametrize("field,value", [("norm", 3), ("norm", -1), ("eps", 0.0), ("eps", float("nan")),
                                         ("out_scale", float("inf")), ("reserved", 2)])
def test_bad_epilogue_rejected(lib, field, value):
    e = _lib.DiffattnEpilogue()
    e.norm, e.eps, e.out_scale, e.reserved = _lib.DIFFATTN_NORM_RMS, 1e-5, 1.0, 0
    setattr(e, field, value)
    rc = lib.diffattn_fwd_ex(ctypes.byref(desc()), *ptrs(5), ctypes.c_float(0.5), None, 1,
                             ctypes.byref(e), ctypes.c_void_p(FAKE * 9), None, 0, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID


def kv_desc(B=2, H=3, Tq=1, Tk=1000, D=64, dtype=_lib.DIFFATTN_BF16, kv_group=0, Dv=0):
    d = _lib.DiffattnKvDesc()
    d.B, d.H, d.Tq, d.Tk, d.D, d.dtype, d.kv_group = B, H, Tq, Tk, D, dtype, kv_group
    d.Dv = Dv
    Hk = H // max(kv_group, 1)
    wv = Dv or 2 * D
    for f, T, w, h in (("q1_stride", Tq, D, H), ("q2_stride", Tq, D, H), ("k1_stride", Tk, D, Hk),
                       ("k2_stride", Tk, D, Hk), ("v_stride", Tk, wv, Hk),
                       ("o_stride", Tq, wv, H)):
        getattr(d, f)[:] = (h * T * w, T * w, w)
    return d


def test_decode_workspace_query(lib):
    d = kv_desc()
    n = lib.diffattn_decode_workspace_bytes(ctypes.byref(d))
    assert n > 0 and n % 4 == 0
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tk=100000))) >= n
    # shapes the split-key decode does not take run on the forward kernels,
    # which use no workspace (a nominal 16 bytes)
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=48))) == 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tq=17))) == 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tq=9, dtype=_lib.DIFFATTN_F32))) == 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tq=1024, Tk=8192))) == 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=64, Dv=128))) == n
    # the DIFF V2 head (bf16, D = Dv = 128) up to 16 queries: the tensor-core
    # split-key decode's partial results; more queries or fp32: the forward
    v2 = lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=128, Dv=128)))
    assert v2 > 16 and v2 % 4 == 0
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=128, Dv=128, Tq=8))) > 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=128, Dv=128, Tq=16))) > 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=128, Dv=128, Tq=17))) == 16
    assert lib.diffattn_decode_workspace_bytes(
        ctypes.byref(kv_desc(D=128, Dv=128, dtype=_lib.DIFFATTN_F32))) == 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=128, Dv=64))) == 16
    # the V2 decode workload (16 sequences of 8192 keys, 16 heads over 8)
    # fits the 8 MiB buffer of diffattn_decode_noalloc
    w = lib.diffattn_decode_workspace_bytes(
        ctypes.byref(kv_desc(B=16, H=16, kv_group=2, Tk=8192, D=128, Dv=128)))
    assert 16 < w <= 8 * 1024 * 1024
    # invalid descriptors
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(D=200))) == 0
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Dv=300))) == 0
    assert lib.diffattn_decode_workspace_bytes(None) == 0


def test_decode_workspace_four_row_shapes_fit_noalloc_buffer(lib):
    # 32 query heads over 8 key/value heads (four rows per key/value head,
    # the tensor-core pass's shape), 16 sequences of 8192 cached keys: the
    # partial results fit the 8 MiB buffer of diffattn_decode_noalloc, both
    # the tensor-core pass's slots and the CUDA-core layout it falls back to
    n = lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(B=16, H=32, kv_group=4, Tk=8192)))
    assert 0 < n <= 8 * 1024 * 1024
    n4 = lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(B=16, H=16, Tq=4, Tk=8192)))
    assert 0 < n4 <= 8 * 1024 * 1024


@pytest.mark.parametrize("kw,code", [(dict(Tq=0), _lib.DIFFATTN_ERR_INVALID),
                                     (dict(D=200), _lib.DIFFATTN_ERR_INVALID),
                                     (dict(Dv=-2), _lib.DIFFATTN_ERR_INVALID),
                                     (dict(Dv=257), _lib.DIFFATTN_ERR_INVALID),
                                     (dict(Tk=2 ** 31), _lib.DIFFATTN_ERR_UNSUPPORTED),
                                     (dict(Tq=4, Tk=3), _lib.DIFFATTN_ERR_INVALID)])
def test_decode_rejects(lib, kw, code):
    d = kv_desc(**kw)
    ws = ctypes.c_void_p(FAKE * 20)
    rc = lib.diffattn_decode(ctypes.byref(d), *ptrs(5), ctypes.c_float(0.5), None, 1, None,
                             ctypes.c_void_p(FAKE * 9), ws, 1 << 30, None)
    assert rc == code


def test_decode_requires_workspace(lib):
    d = kv_desc()
    rc = lib.diffattn_decode(ctypes.byref(d), *ptrs(5), ctypes.c_float(0.5), None, 1, None,
                             ctypes.c_void_p(FAKE * 9), None, 0, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID


def test_decode_noalloc_reports_argument_errors_before_its_size_limit(lib):
    # a problem too big for the 8 MiB buffer, with a NULL output: the argument
    # error of diffattn_decode comes first, the buffer limit only after it
    big = kv_desc(B=128, H=64, Tq=2, Tk=2)
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(big)) > 8 * 1024 * 1024
    rc = lib.diffattn_decode_noalloc(ctypes.byref(big), *ptrs(5), ctypes.c_float(0.5), None, 1,
                                     None, None, None)
    assert rc == _lib.DIFFATTN_ERR_INVALID
    rc = lib.diffattn_decode_noalloc(ctypes.byref(big), *ptrs(5), ctypes.c_float(float("nan")), None, 1,
                                     None, ctypes.c_void_p(FAKE * 9), None)
    assert rc == _lib.DIFFATTN_ERR_INVALID
    # unsupported sizes report as diffattn_decode does
    rc = lib.diffattn_decode_noalloc(ctypes.byref(kv_desc(Tk=2 ** 31)), *ptrs(5),
                                     ctypes.c_float(0.5), None, 1, None, ctypes.c_void_p(FAKE * 9),
                                     None)
    assert rc == _lib.DIFFATTN_ERR_UNSUPPORTED


def test_grouped_heads_select_and_reject(lib):
    # H = 8 query heads over 2 key/value heads: still the tensor-core kernel
    assert select(lib, desc(H=8, kv_group=4)) == _lib.DIFFATTN_KERNEL_TCGEN05
    assert select(lib, desc(H=8, kv_group=1)) == _lib.DIFFATTN_KERNEL_TCGEN05
    assert select(lib, desc(H=8, kv_group=8)) == _lib.DIFFATTN_KERNEL_TCGEN05
    assert select(lib, desc(H=6, kv_group=4)) == _lib.DIFFATTN_ERR_INVALID


def test_decode_grouped_heads_share_ctas(lib):
    # 8 query heads over 2 key/value heads, one query each: the 4 heads of a
    # group go in one CTA (4 rows), so the partial results take as many
    # floats as 2 heads of 4 queries -- not 8 heads of 1 query.
    size = lambda **kw: lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(**kw)))
    assert size(H=8, kv_group=4, Tq=1) == size(H=2, Tq=4)
    # 16 rows per key/value head (g = 8, Tq = 2): two CTAs of 8 rows
    assert size(H=8, kv_group=8, Tq=2) == size(H=2, Tq=8)
    assert size(H=8, kv_group=3) == 0
    assert size(H=8, kv_group=-2) == 0


def test_bwd_workspace_size(lib):
    d = desc(B=2, H=4, T=100)
    assert lib.diffattn_bwd_workspace_bytes(ctypes.byref(d)) == 2 * 4 * 100 * 16 + 512
    assert lib.diffattn_bwd_workspace_bytes(None) == 0
    assert lib.diffattn_bwd_workspace_bytes(ctypes.byref(desc(T=0))) == 0


def bwd(lib, d, grads=None, ws=FAKE * 30, ws_bytes=1 << 30, lam=0.5):
    grads = grads if grads is not None else ptrs(5, base=FAKE * 40)
    return lib.diffattn_bwd(ctypes.byref(d), *ptrs(5), ctypes.c_float(lam), None, 1,
                            ctypes.c_void_p(FAKE * 9), *grads, ctypes.c_void_p(FAKE * 50),
                            ctypes.c_void_p(ws), ctypes.c_size_t(ws_bytes), None)


def test_bwd_rejects_without_gpu(lib):
    assert bwd(lib, desc(D=0)) == _lib.DIFFATTN_ERR_INVALID
    assert bwd(lib, desc(H=6, kv_group=4)) == _lib.DIFFATTN_ERR_INVALID
    assert bwd(lib, desc(), lam=float("nan")) == _lib.DIFFATTN_ERR_INVALID
    g = ptrs(5, base=FAKE * 40)
    g[3] = None
    assert bwd(lib, desc(), grads=g) == _lib.DIFFATTN_ERR_INVALID
    assert bwd(lib, desc(), ws_bytes=16) == _lib.DIFFATTN_ERR_INVALID
    assert bwd(lib, desc(), ws=FAKE * 30 + 4) == _lib.DIFFATTN_ERR_INVALID
    assert bwd(lib, desc(), ws=0) == _lib.DIFFATTN_ERR_INVALID


def test_lambda_backward_rejects_without_gpu(lib):
    p = ptrs(9)
    assert lib.diffattn_lambda_backward(*p[:4], 0, *p[4:], None) == _lib.DIFFATTN_ERR_INVALID
    q = list(p)
    q[5] = None
    assert lib.diffattn_lambda_backward(*q[:4], 8, *q[4:], None) == _lib.DIFFATTN_ERR_INVALID


def test_fwd_host_rejects_without_gpu(lib):
    def call(d, hp=None):
        hp = hp if hp is not None else ptrs(6, base=FAKE * 60)
        return lib.diffattn_fwd_host(ctypes.byref(d), *hp[:5], ctypes.c_float(0.5), None, 1, hp[5],
                                     *ptrs(6), None, 0, None)
    hp = ptrs(6, base=FAKE * 60)
    hp[2] = None
    assert call(desc(), hp) == _lib.DIFFATTN_ERR_INVALID
    d = desc(B=2)
    d.v_stride[2] = 2 * 64 + 8           # not dense
    assert call(d) == _lib.DIFFATTN_ERR_INVALID
    d = desc(B=2)
    d.q1_stride[1] = 0                   # broadcast heads are not dense
    assert call(d) == _lib.DIFFATTN_ERR_INVALID


def _max_segments(units, tpu, grid):
    """Brute force: the most CTA ranges [c*total//grid, (c+1)*total//grid)
    that meet one unit's tiles [u*tpu, (u+1)*tpu)."""
    total = units * tpu
    bounds = [c * total // grid for c in range(grid + 1)]
    best = 0
    for u in range(units):
        t0, t1 = u * tpu, (u + 1) * tpu
        meets = sum(1 for c in range(grid) if bounds[c] < t1 and bounds[c + 1] > t0)
        best = max(best, meets)
    return best


@pytest.mark.parametrize("B,H,kv_group,Tq,Tk", [(2, 3, 0, 4, 1000), (2, 3, 0, 8, 200), (1, 4, 4, 1, 129),
                                                 (3, 8, 4, 2, 4099), (16, 32, 4, 1, 8192), (5, 6, 3, 2, 700),
                                                 (40, 4, 4, 1, 256), (1, 1, 0, 5, 70000)])
def test_decode_workspace_holds_every_tensor_core_segment(lib, B, H, kv_group, Tq, Tk):
    # Four or eight rows per key/value head (bf16, D = 64): the tensor-core
    # first pass gives every CTA one contiguous range of the units' 128-key
    # tiles and writes one partial slot per (unit, CTA meeting it).  The
    # workspace must hold that many slots per unit for any GPU of up to 1024
    # SMs (4 + 4 D floats per row and slot).
    g = max(kv_group, 1)
    rows = g * Tq
    chunks = -(-rows // 8)
    per = -(-rows // chunks)
    tqb = 1
    while tqb < per:
        tqb *= 2
    assert tqb >= 4
    units = B * (H // g) * chunks
    tpu = -(-Tk // 128)
    need = lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(B=B, H=H, Tq=Tq, Tk=Tk, kv_group=kv_group)))
    for sms in (1, 7, 148, 152, 160, 1024):
        grid = min(units * tpu, sms)
        assert need >= units * _max_segments(units, tpu, grid) * tqb * (4 + 4 * 64) * 4, sms


def test_decode_workspace_sixteen_row_units(lib):
    # bf16 D = 64 with 9 to 16 query rows per key/value head (here 4 query
    # heads per key/value head and 4 new queries): units of 16 rows on the
    # tensor cores, with room for the split-key layout of 8-row units that a
    # call runs on the CUDA cores when its cache rows are not dense
    d16 = kv_desc(B=16, H=32, kv_group=4, Tq=4, Tk=8192)
    n16 = lib.diffattn_decode_workspace_bytes(ctypes.byref(d16))
    assert n16 > 16 and n16 % 4 == 0
    d8 = kv_desc(B=16, H=32, kv_group=4, Tq=2, Tk=8192)      # 8 rows: one 8-row unit
    assert n16 > lib.diffattn_decode_workspace_bytes(ctypes.byref(d8))
    # Tq up to 16 with one query head per key/value head: the tensor cores
    # alone (no split-key layout of 8-row units exists beyond 8 queries)
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tq=16))) > 16
    assert lib.diffattn_decode_workspace_bytes(ctypes.byref(kv_desc(Tq=12, H=4, kv_group=2))) > 16
