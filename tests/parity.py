"""Comparison rules between the CUDA path and the oracle (the tolerances the
method's statement fixes):

  * fp32 scales: relative 1e-6 (exact zero where the oracle has zero);
  * E4M3FN codes: within 1 code step (the two sides take the rounding
    decision on fp32 vs fp64 normalized values, so a value within a few fp32
    ULPs of a rounding midpoint may land on either neighbour), and at least
    99.9% identical;
  * bf16 words: within 1 bf16 ULP;
  * GEMM output: relative Frobenius error <= 5e-3 against the fp64
    dequantized product.
"""

from __future__ import annotations

import numpy as np
import torch

SCALE_RTOL = 1e-6
CODE_EXACT_MIN = 0.999
GEMM_REL_FRO = 5e-3


def code_ordinal(c: np.ndarray) -> np.ndarray:
    """Signed position of an E4M3FN code on the number line (+0 and -0 equal)."""
    c = np.asarray(c, dtype=np.uint8).astype(np.int64)
    mag = c & 0x7F
    return np.where(c & 0x80, -mag, mag)


def bf16_ordinal(w: np.ndarray) -> np.ndarray:
    w = np.asarray(w, dtype=np.uint16).astype(np.int64)
    mag = w & 0x7FFF
    return np.where(w & 0x8000, -mag, mag)


def assert_codes_close(got, want, what="codes"):
    got, want = np.asarray(got, np.uint8), np.asarray(want, np.uint8)
    assert got.shape == want.shape, (got.shape, want.shape)
    d = np.abs(code_ordinal(got) - code_ordinal(want))
    assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} codes more than 1 step apart"
    exact = (code_ordinal(got) == code_ordinal(want)).mean() if got.size else 1.0
    assert exact >= CODE_EXACT_MIN, f"{what}: only {exact:.6f} exact"
    return exact


def assert_scales_close(got, want, what="scales"):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape
    zero = want == 0
    assert np.all(got[zero] == 0), f"{what}: nonzero where the oracle has 0"
    rel = np.abs(got[~zero] - want[~zero]) / np.abs(want[~zero])
    assert rel.max(initial=0) <= SCALE_RTOL, f"{what}: max rel err {rel.max():.3e}"


def assert_bf16_close(got, want, what="bf16"):
    got, want = np.asarray(got, np.uint16), np.asarray(want, np.uint16)
    assert got.shape == want.shape
    d = np.abs(bf16_ordinal(got) - bf16_ordinal(want))
    assert d.max(initial=0) <= 1, f"{what}: {int((d > 1).sum())} words more than 1 ULP apart"


def rel_fro(got: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.uint8).cpu().numpy()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_value(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)
