"""Helpers shared by the GPU parity tests: host->device copies of generated inputs and
the comparison rules.

Tolerance.  The build's bar for attention outputs is max |err| <= 2e-3 for fp16/bf16
outputs against the fp64 oracle, with fp32 intermediates good to 1e-5 relative.  The
tests apply two rules to every output element o (exact = oracle fp64 value):

  1. |gpu - exact| <= 2e-3, wherever half a unit in the last place of the output
     format is below 2e-3 (|exact| < 1 for bf16, < 8 for fp16); above that, the output
     rounding alone can exceed 2e-3, so rule 2 governs.
  2. |gpu - exact| <= half_ulp_T(exact) + 1e-4 * cond + 1e-6, where cond = sum_t w_t |V_t|
     (the oracle's attention over |V|): the output rounding plus an fp32 accumulation
     allowance proportional to the row's condition scale.  This is much tighter than rule
     1 for typical outputs (|o| ~ 0.05), so e.g. one dropped or extra token in a context
     of a few thousand fails it.

A rule of the form "within one ulp of the rounded oracle" is not used: for outputs near
zero (cancellation) the fp32 noise, though tiny next to cond, spans many ulps.
"""
import numpy as np
import torch

import oracle

ATOL = 2e-3


def to_dev(bits: np.ndarray, dtype_code: int, device="cuda"):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    t = t.view(torch.bfloat16 if dtype_code == 1 else torch.float16)
    return t.to(device)


def to_dev_i(a: np.ndarray, dtype, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).to(device)


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def abs_bits(bits: np.ndarray) -> np.ndarray:
    """|x| of fp16/bf16 bit patterns (clears the sign bit; NaN stays NaN)."""
    return bits & np.uint16(0x7FFF)


def ulp_distance(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def half_ulp(x: np.ndarray, dtype_code: int) -> np.ndarray:
    mant = 7 if dtype_code == 1 else 10
    e = np.floor(np.log2(np.maximum(np.abs(x), 1e-30)))
    e = np.maximum(e, -126 if dtype_code == 1 else -14)
    return 0.5 * 2.0 ** (e - mant)


def check_attention(gpu_bits: np.ndarray, exact: np.ndarray, dtype_code: int, what: str = "", cond=None,
                    rel: float = 1e-4):
    """Assert rules 1 and 2 above (rule 2 only when cond is given; `rel` replaces the 1e-4
    factor where a path adds a known rounding of its own); returns max |err|."""
    assert np.isfinite(exact).all(), f"{what}: oracle produced non-finite values"
    got = oracle.to_double(gpu_bits, dtype_code).reshape(exact.shape)
    assert np.isfinite(got).all(), f"{what}: GPU output has NaN/inf (a canary was read?)"
    err = np.abs(got - exact)
    hu = half_ulp(exact, dtype_code)
    r1 = (hu < ATOL) & (err > ATOL)
    if cond is not None:
        allow2 = hu + rel * cond + 1e-6
        r2 = err > allow2
    else:
        allow2 = np.maximum(ATOL, hu)
        r2 = err > allow2
    bad = r1 | r2
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(bad, err / allow2, 0)), err.shape)
        c = "" if cond is None else f", cond {cond[i]:.4e}"
        raise AssertionError(f"{what}: {int(bad.sum())} of {err.size} elements out of tolerance; worst at {i}: "
                             f"gpu {got[i]:.6e} exact {exact[i]:.6e} err {err[i]:.3e}{c}")
    return float(err.max())
