"""Parity bounds shared by the GEMM and linear-layer tests, beside the whole-matrix
relative Frobenius check.

1. Element-wise.  The GPU sums the exact products of dequantized NVFP4 operands (and of
   the BF16 branch factors) in FP32 tensor-core accumulators; the oracle sums them in
   FP64.  With at most K + r rounding events of relative size 2^-24 on partial sums
   bounded by S = sum_k |a_k||b_k| (+ the branch's sum of |p_j||q_j|), the FP32
   accumulation error is at most (K + r) 2^-24 S.  The output is then rounded once: to
   BF16 (the GPU rounds its FP32 value, the oracle its exact value, so the two can land
   one BF16 step apart) or, in FP32 mode, by half an FP32 step.  Where the branch factor
   P itself comes from the GPU (the linear calls form P = bf16(X L^T) with an FP32
   accumulation, which can round to the other BF16 neighbour of the oracle's FP64 value),
   each p_j may differ by one BF16 step, 2^-7 |p_j| at most: the caller passes that
   term, 2^-7 beta sum_j |p_j||q_j|, as `extra`.
2. Per chunk.  The element-wise bound grows with K, so for long contractions it would
   not see a dropped K stage.  Each output row is also cut into the 32-column chunks the
   epilogue drains, and each chunk's relative Frobenius error against the (rounded)
   reference must stay below 8e-3: a rounding that lands on the other BF16 neighbour
   moves one element by at most 2^-8 of itself, i.e. a chunk by about 7e-4 per flip
   (2e-3 for an element three times the chunk's RMS), while a fault confined to one
   tile or chunk (a dropped K stage or a wrong scale atom at K = 16384, a misplaced
   chunk) moves it by 5e-2 or more.
"""
import numpy as np

CHUNK_COLS = 32
CHUNK_TOL = 8e-3


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    """One BF16 step (8 significand bits) at the magnitude of v (normal range)."""
    a = np.maximum(np.abs(v), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7.0)


def elementwise_bound(abs_sum: np.ndarray, terms: int, ref: np.ndarray, bf16_out: bool) -> np.ndarray:
    acc = terms * 2.0 ** -24 * abs_sum
    out = ulp_bf16(ref) if bf16_out else 2.0 ** -24 * np.abs(ref)
    return acc + out


def assert_chunks(got: np.ndarray, ref: np.ndarray, what: str = "") -> None:
    R, C = got.shape
    n = C // CHUNK_COLS
    g = got[:, : n * CHUNK_COLS].reshape(R, n, CHUNK_COLS)
    w = ref[:, : n * CHUNK_COLS].reshape(R, n, CHUNK_COLS)
    num = np.sqrt(((g - w) ** 2).sum(axis=2))
    den = np.maximum(np.sqrt((w ** 2).sum(axis=2)), 1e-300)
    e = num / den
    if (e >= CHUNK_TOL).any():
        i = np.unravel_index(np.argmax(e), e.shape)
        raise AssertionError(f"{what}: {int((e >= CHUNK_TOL).sum())} of {e.size} 32-column chunks beyond "
                             f"{CHUNK_TOL}; worst row {int(i[0])} chunk {int(i[1])}: {float(e[i]):.3e}")


def assert_elementwise(got: np.ndarray, exact: np.ndarray, abs_sum: np.ndarray, terms: int, bf16_out: bool,
                       what: str = "", rounded: np.ndarray | None = None, extra=0.0) -> None:
    """`exact`: the oracle's FP64 result; `rounded`: the same rounded to the output type
    (for BF16 outputs), against which the chunks are compared; `extra`: an added
    absolute bound (the branch-factor rounding term)."""
    bound = elementwise_bound(abs_sum, terms, exact, bf16_out) + extra
    err = np.abs(got - exact)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err / bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} elements beyond the bound; worst at {tuple(int(x) for x in i)}:"
                             f" got {got[i]!r}, want {exact[i]!r}, bound {bound[i]!r}")
    assert_chunks(got, exact if rounded is None else rounded, what)
