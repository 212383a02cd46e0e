"""Shared test utilities: device placement and the parity tolerances.

Tolerances (stated for this operation): bf16 inputs with fp32 accumulation,
max-abs error <= 2e-2 and mean-abs error <= 2e-3 against the float64 oracle;
float32 path, max-abs error <= 1e-4.

bf16 output rounding: an output of magnitude >= 8 cannot be represented in
bf16 to within 2e-2 (half an ulp there is 2^-5 = 0.031).  For those elements
the max-abs bound applies to the error in excess of half an ulp of the oracle
value, i.e. to what the kernel adds beyond rounding its fp32 result to bf16.
The mean-abs bound applies to the raw mean error whenever the rounding floor
(the mean error of the exact result correctly rounded to bf16) is below
1e-3.  Only where that floor is material (>= 1e-3: outputs of magnitude ~2-8
on average, as on the value-offset workload at lambda = 0, where the floor
alone is ~2e-3) does the bound apply to the mean error in excess of the
floor.  Both raw figures are reported as well (DIFFATTN_PARITY_LOG).
"""
from __future__ import annotations

import json
import os

import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_ABS = 1e-4
# Rounding floor from which the mean-abs bound is read as an excess over it.
MATERIAL_FLOOR = 1e-3


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half a unit in the last place of bf16 (8 significant bits) at |x|."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bfloat16 (ties to even) of float64 values, via float32."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return r.view(np.float32).astype(np.float64)


def compare(got: np.ndarray, ref: np.ndarray, dtype: str) -> dict:
    """Error statistics of `got` against the float64 oracle `ref`."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite output"
    err = np.abs(got - ref)
    stats = {"max_abs": float(err.max()) if err.size else 0.0,
             "mean_abs": float(err.mean()) if err.size else 0.0, "n": int(err.size)}
    if dtype == "bf16":
        big = np.abs(ref) >= 8.0
        small_err = err[~big]
        stats["max_abs_below_8"] = float(small_err.max()) if small_err.size else 0.0
        excess = err[big] - bf16_half_ulp(ref[big])
        stats["n_ge_8"] = int(big.sum())
        stats["max_excess_ge_8"] = float(excess.max()) if excess.size else 0.0
        floor = float(np.abs(round_bf16(ref) - ref).mean()) if err.size else 0.0
        stats["rounding_floor_mean"] = floor
        stats["mean_abs_excess"] = stats["mean_abs"] - floor
    return stats


def assert_close(got, ref, dtype: str, what: str = "") -> dict:
    s = compare(got, ref, dtype)
    log = os.environ.get("DIFFATTN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "dtype": dtype, **s}) + "\n")
    if dtype == "f32":
        assert s["max_abs"] <= F32_MAX_ABS, f"{what} fp32 max-abs {s}"
    else:
        assert s["max_abs_below_8"] <= BF16_MAX_ABS, f"{what} bf16 max-abs {s}"
        assert s["max_excess_ge_8"] <= BF16_MAX_ABS, f"{what} bf16 excess over rounding {s}"
        if s["rounding_floor_mean"] < MATERIAL_FLOOR:
            assert s["mean_abs"] <= BF16_MEAN_ABS, f"{what} bf16 mean-abs (raw) {s}"
        else:
            assert s["mean_abs_excess"] <= BF16_MEAN_ABS, f"{what} bf16 mean-abs {s}"
    return s


# dlambda = -sum over rows of t_r = dO_r . (A_2 V)_r is a sum of many terms of
# either sign; its natural scale is the L2 norm of the row terms,
# sqrt(sum_r t_r^2), the typical size of such a sum (an L1 scale, sum |t_r|,
# would grow with the square root of the number of rows faster).  The output
# bounds apply in units of that scale: |err| <= 2e-2 * max(1, scale) for bf16,
# 1e-4 * max(1, scale) for float32.
def assert_dlambda_close(got: float, ref: float, row_terms, dtype: str, what: str = "") -> dict:
    t = np.asarray(row_terms, dtype=np.float64)
    scale = max(1.0, float(np.sqrt(np.sum(t * t))))
    err = abs(float(got) - float(ref))
    stats = {"dlambda": float(got), "ref": float(ref), "abs_err": err, "l2_scale": scale,
             "rel_to_scale": err / scale, "rel_to_ref": err / max(abs(float(ref)), 1e-30)}
    log = os.environ.get("DIFFATTN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "dtype": dtype, "dlambda": True, **stats}) + "\n")
    bound = (F32_MAX_ABS if dtype == "f32" else BF16_MAX_ABS) * scale
    assert err <= bound, f"{what} dlambda {stats}"
    return stats


def torch_dtype(dtype: str):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[dtype]


def to_device(x: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    """float32 array holding dtype-representable values -> device tensor."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(device=device, dtype=torch_dtype(dtype))


def to_numpy(t: torch.Tensor) -> np.ndarray:
    return t.detach().to(device="cpu", dtype=torch.float64).numpy()


# Gradients.  Their magnitudes grow with the number of terms each one sums
# (queries per key, keys per query), so the output tolerances above are
# applied to the error measured in units of the gradient tensor's own scale,
# s = max(1, rms(reference)): max |err| / s <= 2e-2 and mean |err| / s <= 2e-3
# for bf16, max |err| / s <= 1e-4 for float32.  A bf16 gradient is rounded to
# bf16 on output, which alone costs up to half an ulp of the element (2^-9
# relative: 0.0156 at |g| = 4, more above); as for the forward's large
# outputs, the bf16 bounds apply to the error in excess of that rounding:
# max(0, |err| - half_ulp(ref)) for the max, and the mean error in excess of
# the mean error of the exact gradient rounded to bf16 for the mean.
def grad_scale(ref: np.ndarray) -> float:
    ref = np.asarray(ref, dtype=np.float64)
    return max(1.0, float(np.sqrt(np.mean(ref * ref)))) if ref.size else 1.0


# Backward from saved forward results: the row statistics Dd_b are formed from
# the bf16-rounded saved outputs (Dd_2 = dO . O2, Dd_1 = dO . (O + lambda O2),
# two roundings of half an ulp each per element of O and O2).  That error is
# the same for every key of a row, so it adds coherently along each row of dS:
# dQ_b and dK_b take it once more on top of the recomputing path's error.  The
# bf16 bounds for that path are therefore twice the above (slack = 2).
SAVED_PATH_SLACK = 2.0


def assert_grad_close(got, ref, dtype: str, what: str = "", slack: float = 1.0) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    s = grad_scale(ref)
    err = np.abs(got - ref)
    stats = {"scale": s, "max_rel": float(err.max() / s) if err.size else 0.0,
             "mean_rel": float(err.mean() / s) if err.size else 0.0, "n": int(err.size)}
    if dtype == "bf16" and err.size:
        excess = np.maximum(0.0, err - bf16_half_ulp(ref))
        floor = float(np.abs(round_bf16(ref) - ref).mean())
        stats["max_excess_rel"] = float(excess.max() / s)
        stats["mean_excess_rel"] = max(0.0, float(err.mean()) - floor) / s
    log = os.environ.get("DIFFATTN_PARITY_LOG")
    if log:
        with open(log, "a") as f:
            f.write(json.dumps({"case": what, "dtype": dtype, "grad": True, "slack": slack,
                                **stats}) + "\n")
    if dtype == "f32":
        assert stats["max_rel"] <= F32_MAX_ABS, f"{what} fp32 gradient {stats}"
    else:
        assert stats["max_excess_rel"] <= slack * BF16_MAX_ABS, f"{what} bf16 gradient max {stats}"
        assert stats["mean_excess_rel"] <= slack * BF16_MEAN_ABS, f"{what} bf16 gradient mean {stats}"
    return stats
