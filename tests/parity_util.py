"""Element-wise parity bounds shared by the GEMM and linear-layer tests.

The GPU sums the exact products of dequantized NVFP4 operands (and of the BF16
branch factors) in FP32 tensor-core accumulators; the oracle sums them in FP64.
With at most K + r rounding events of relative size 2^-24 on partial sums
bounded by S = sum_k |a_k||b_k| (+ the branch's sum of |p_j||q_j|), the FP32
accumulation error is at most (K + r) 2^-24 S.  The output is then rounded
once: to BF16 (the GPU rounds its FP32 value, the oracle its exact value, so
the two can land one BF16 step apart) or, in FP32 mode, by half an FP32 step.
A fault confined to a few tiles (a dropped K stage, a wrong scale atom, a
misplaced 32-column chunk) moves elements by a sizeable fraction of |C|, far
beyond this bound, while leaving the relative Frobenius error of the whole
matrix small.
"""
import numpy as np


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """One BF16 step (8 significand bits) at the magnitude of v (normal range)."""
    a = np.maximum(np.abs(v), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7.0)


def elementwise_bound(abs_sum: np.ndarray, terms: int, ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    acc = terms * 2.0 ** -24 * abs_sum
    out = ulp_bf16(ref) if bf16_out else 2.0 ** -24 * np.abs(ref)
    return acc + out


def assert_elementwise(got: np.ndarray, ref: np.ndarray, abs_sum: np.ndarray, terms: int, bf16_out: bool,
                       what: str = "") -> None:
    bound = elementwise_bound(abs_sum, terms, ref, bf16_out)
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the bound; worst at {tuple(int(x) for x in i)}:"
                             f" got {got[i]!r}, want {ref[i]!r}, bound {bound[i]!r}")
