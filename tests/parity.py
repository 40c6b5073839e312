"""Shared helpers for the GPU parity tests: numpy <-> torch marshalling and
the tolerance of the method's floating-point outputs.

Tolerance: max |y - y_ref| <= 2e-2 * RMS(y_ref) over the compared elements
(the bar the target states for every GEMM output; the GPU computes in bf16
with fp32 accumulation, the oracle in double).

Every output of the library is stored in bf16, whose rounding alone exceeds
that bound on the tails: a bf16 value x carries up to half an ulp,
<= 2^-8 |x|, of rounding, and the largest outputs reach 5-20 x RMS (silu(a)*b
is heavy-tailed), i.e. 2e-2 to 8e-2 RMS from the format alone.  The bound is
therefore applied to the error left after the output format's own quantum:

    max_i ( |y_i - ref_i| - 2^-8 |ref_i| ) <= 2e-2 * RMS(ref)

with ref the oracle's exact (double) value.  The allowance covers correct
rounding and a one-ulp flip when the fp32 accumulation lands next to a
rounding midpoint; everything else (accumulation order, the bf16
intermediate H of the FFN, a wrong tile or row) must fit in 2e-2 RMS.
"""
import numpy as np
import torch

from group_masked_gemm_gb300 import synthetic as syn

TOL = 2e-2


def to_dev(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> CUDA bf16 tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def mask_dev(mask: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(mask, np.uint8)).cuda()


def to_f64(t: torch.Tensor) -> np.ndarray:
    """CUDA bf16 tensor -> float64 numpy (exact)."""
    bits = t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return syn.bf16_to_f32(bits).astype(np.float64)


def rel_err(y: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.square(ref)))) if ref.size else 0.0
    err = float(np.max(np.abs(y - ref))) if ref.size else 0.0
    if rms == 0.0:
        return 0.0 if err == 0.0 else float("inf")
    return err / rms


BF16_HALF_ULP = 2.0 ** -8


def excess_err(y: np.ndarray, ref: np.ndarray) -> float:
    """max(|y - ref| - 2^-8 |ref|) / RMS(ref)."""
    if ref.size == 0:
        return 0.0
    rms = float(np.sqrt(np.mean(np.square(ref))))
    ex = float(np.max(np.abs(y - ref) - BF16_HALF_ULP * np.abs(ref)))
    if rms == 0.0:
        return 0.0 if ex <= 0.0 else float("inf")
    return max(ex, 0.0) / rms


def assert_close(y: np.ndarray, ref: np.ndarray, what: str = ""):
    """y: the library's bf16 output (as float64); ref: the oracle's exact value."""
    e = excess_err(y, ref)
    raw = rel_err(y, ref)
    assert e <= TOL, (f"{what}: max(|y-ref| - 2^-8|ref|) / RMS(ref) = {e:.3e} > {TOL} "
                      f"(plain max|y-ref|/RMS = {raw:.3e})")
    return e


def inactive_columns(mask: np.ndarray, G: int) -> np.ndarray:
    return ~np.repeat(mask.astype(bool), G, axis=1)
