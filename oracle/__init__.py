"""NVFP4 oracle: plain, slow, obviously-correct CPU reference for the NVFP4
linear-projection hot path of "Full-Stack FP4: Stable LLM Pretraining with
Quantized Projections, Optimizers, and Attention".

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  It
shares no code with the CUDA library and never imports it.

The quantizer is plain C (``nvfp4_oracle.c``, FP32 steps with FMA contraction
off, brute-force rounding); the products are NumPy FP64 matmuls of the exactly
dequantized operands.  Functions and the passages they follow:

- ``quantize``: NVFP4 block quantization, "standard NVFP4" (section 3, Key
  contributions) with SR for gradients (SR is named in section 2.2, Q-AdamW).
  The format itself (E2M1 codes, E4M3 scale per 16 elements, FP32 tensor
  scale) is not defined on the pages; see the C file for every reading.
- ``lora_svd_split``: W = W_res + beta * L2 @ L1 (section 2.1, LoRA-SVD linear
  projections, the "Mechanism" paragraph), initialised by an exact truncated
  SVD (READING: the pages realign with a randomized SVD; for a one-off split
  the exact SVD is the plainest choice, and Sigma goes into L2).
- ``branch_factor``: P = bf16(X @ L^T), the BF16 low-rank branch (section 2.1:
  the subspace L2 L1 is kept in BF16).  READING: the intermediate P is rounded
  to BF16 once.
- ``lora_factor_grads``: the gradients of the branch factors, dL2 = beta dY^T P
  and dL1 = beta P'^T X with P = bf16(X L1^T) and P' = bf16(dY L2) (section 2.1:
  the backward pass is restricted to the subspace).  READING: straight through
  the BF16 factors (the same rounded P and P' the forward and dX products use),
  FP64 products, FP32 results; the Cholesky-QR constraint on the subspace is not
  specified on the pages and is not applied here.
- ``lora_realign``: the periodic realignment of the LoRA-SVD subspace by a
  randomized SVD (section 2.1, Realignment).  READING: the randomized subspace
  iteration and direct SVD of Halko, Martinsson and Tropp (SIAM Review 2011,
  Algorithms 4.4 and 5.1) on W = W_res + beta L2 L1 with a caller-supplied
  Gaussian test matrix Omega (K x s, s >= r) and q power iterations, each
  product re-orthonormalised; then L2 = U_r Sigma_r / beta, L1 = V_r^T (each
  row's largest-magnitude entry made positive), W_res = W - beta L2 L1 with the
  BF16 factors; FP64, each output rounded to BF16 once.
- ``cholesky_lower`` / ``lora_cholqr``: the Cholesky-QR step of the LoRA-SVD
  backward (section 2.1: the backward pass is restricted to the subspace under a
  Cholesky-QR constraint).  READING (no formula on the pages): the rows of L1
  are re-orthonormalised through the Cholesky factor of their Gram matrix,
  L1 L1^T = L L^T, L1 <- L^-1 L1, and L2 <- L2 L keeps beta L2 L1 unchanged;
  FP64, each factor rounded to BF16 once.
- ``p99_clip`` / ``ns_normalize`` / ``ns_step`` / ``newton_schulz``: Q-Root,
  Newton-Schulz iterations with every matrix product in NVFP4 (section 2.3, NVFP4
  Root optimizer: direct NVFP4 execution; shape-dependent coefficients a, b, c and
  p99 outlier clipping).  READINGS (the pages print neither the coefficients nor
  the clipping rule): the quintic step X <- a X + (b A + c A^2) X with A = X X^T,
  caller-chosen (a, b, c) (default: the cubic 1.5, -0.5, 0 for 12 steps; the
  widely used quintic 3.4445, -4.7750, 2.0315 diverges with NVFP4 products here),
  X_0 = G / ||G||_F, m <= n; the iterate X is clipped at the start of
  each step to +-v, v the ceil(0.99 N)-th smallest |x| of its BF16 values (the
  Gram matrices are not: their largest entries are the diagonal); RTN;
  BF16 products; the two linear combinations in FP32 without contraction; with
  c = 0 the A^2 product is skipped.
- ``fwht16`` / ``vt_encode`` / ``vt_decode``: the Q-AdamW second-moment codec
  (section 2.2, Quantized-state AdamW: square root, tile mean kept in BF16,
  Hadamard transform of the residual, NVFP4; rebuilt by inverting the transform
  and the mean, then squaring).  READINGS (the pages give no sizes): the tile and
  the Hadamard both span one 16-element NVFP4 block along a row; the mean is the
  FP32 pairwise-tree sum of the 16 square roots times 1/16, rounded to BF16; the
  transform is the Walsh-Hadamard butterfly in natural order, FP32, scaled by
  1/4 (orthonormal, its own inverse); RTN with one tensor scale from the
  transformed residual's amax; the decode takes each dequantized value to FP32
  once, then inverts in FP32; every step in FP32 without contraction.
- ``gemm`` / ``linear_fwd`` / ``linear_bwd``: the three products of a linear
  layer, Y = X W^T, dX = dY W, dW = dY^T X, with the residual in NVFP4 and the
  branch in BF16 (section 2.1).  READING: gradients (dY) use SR in both dX and
  dW; X and W use RTN; beta = 1 unless given; the branch factor is stored as
  P~ = bf16(P * beta / alpha) next to the residual's accumulator
  (``fold_branch``).

Parity pins: see ``tests/test_oracle_pins.py``.  The scale layout and the SR
bit mapping are this library's chosen conventions (parity unpinned by the
pages; pinned by invariants and brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

RTN = 0
SR = 1


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i64, u64, u32, f32, f64 = (ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                       ctypes.c_float, ctypes.c_double)
            L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_f32.restype = f32
            L.oracle_f64_to_bf16_rn.argtypes = [f64]
            L.oracle_f64_to_bf16_rn.restype = ctypes.c_uint16
            L.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_value.restype = f64
            L.oracle_e4m3_encode_rn_sat.argtypes = [f32]
            L.oracle_e4m3_encode_rn_sat.restype = ctypes.c_uint8
            L.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            L.oracle_e2m1_value.restype = f64
            L.oracle_e2m1_rtn.argtypes = [f32]
            L.oracle_e2m1_rtn.restype = ctypes.c_uint8
            L.oracle_e2m1_sr.argtypes = [f32, u32]
            L.oracle_e2m1_sr.restype = ctypes.c_uint8
            L.oracle_philox4x32_10.argtypes = [P, P, P]
            L.oracle_philox4x32_10.restype = None
            L.oracle_sr_bits.argtypes = [u64, u32, u64]
            L.oracle_sr_bits.restype = u32
            L.oracle_amax_bf16.argtypes = [P, i64, i64, i64]
            L.oracle_amax_bf16.restype = f32
            L.oracle_tensor_scale.argtypes = [f32]
            L.oracle_tensor_scale.restype = f32
            for name in ("oracle_quantize_rows", "oracle_quantize_cols"):
                fn = getattr(L, name)
                fn.argtypes = [P, i64, i64, i64, ctypes.c_int, u64, u32, f32, P, P]
                fn.restype = None
            L.oracle_quantize_rows_f32.argtypes = [P, i64, i64, f32, P, P]
            L.oracle_quantize_rows_f32.restype = None
            L.oracle_dequantize.argtypes = [P, P, f32, i64, i64, P]
            L.oracle_dequantize.restype = None
            L.oracle_mma_scale_offset.argtypes = [i64, i64, i64]
            L.oracle_mma_scale_offset.restype = i64
            L.oracle_mma_scale_bytes.argtypes = [i64, i64]
            L.oracle_mma_scale_bytes.restype = i64
            L.oracle_scales_to_mma.argtypes = [P, i64, i64, P]
            L.oracle_scales_to_mma.restype = None
            L.oracle_f64_to_bf16_rn_array.argtypes = [P, i64, P]
            L.oracle_f64_to_bf16_rn_array.restype = None
            L.oracle_e4m3_encode_array.argtypes = [P, i64, P]
            L.oracle_e4m3_encode_array.restype = None
            L.oracle_e2m1_rtn_array.argtypes = [P, i64, P]
            L.oracle_e2m1_rtn_array.restype = None
            L.oracle_e2m1_sr_array.argtypes = [P, P, i64, P]
            L.oracle_e2m1_sr_array.restype = None
            L.oracle_sr_bits_array.argtypes = [u64, u32, u64, i64, P]
            L.oracle_sr_bits_array.restype = None
            L.oracle_max_threads.argtypes = []
            L.oracle_max_threads.restype = ctypes.c_int
            L.oracle_set_threads.argtypes = [ctypes.c_int]
            L.oracle_set_threads.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------------------
# scalar / elementwise definitions
# ---------------------------------------------------------------------------

def bf16_to_f32(u16: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(u16, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_rn(x: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16 (nearest, ties to even); returns bit patterns."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    lib().oracle_f64_to_bf16_rn_array(_ptr(v), v.size, _ptr(out))
    return out


def e4m3_value(b: int) -> float:
    return lib().oracle_e4m3_value(int(b))


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(v), v.size, _ptr(out))
    return out


def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(int(code))


def e2m1_rtn(y: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32)
    out = np.empty(y.shape, dtype=np.uint8)
    lib().oracle_e2m1_rtn_array(_ptr(y), y.size, _ptr(out))
    return out


def e2m1_sr(y: np.ndarray, rnd16: np.ndarray) -> np.ndarray:
    y = np.ascontiguousarray(y, dtype=np.float32)
    r = np.ascontiguousarray(rnd16, dtype=np.uint32)
    assert r.shape == y.shape
    out = np.empty(y.shape, dtype=np.uint8)
    lib().oracle_e2m1_sr_array(_ptr(y), _ptr(r), y.size, _ptr(out))
    return out


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
    out = np.empty(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed: int, stream: int, e0: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint32)
    lib().oracle_sr_bits_array(seed, stream, e0, n, _ptr(out))
    return out


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


# ---------------------------------------------------------------------------
# quantizer
# ---------------------------------------------------------------------------

def amax(x_bf16: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    return float(lib().oracle_amax_bf16(_ptr(x), R, C, C))


def tensor_scale(amax_value: float) -> float:
    return float(lib().oracle_tensor_scale(float(amax_value)))


class QTensor:
    """Quantized tensor in the oracle's own (row-major) layout.

    codes: uint8 [rows, cols/2], element 2i in the low nibble.
    scales: uint8 [rows, cols/16] row-major E4M3 bytes.
    S_t: float32 tensor (decode) scale; amax: the tensor amax it came from.
    rows/cols describe the quantized (possibly transposed) tensor.
    """

    def __init__(self, codes, scales, S_t, amax_value, rows, cols):
        self.codes, self.scales = codes, scales
        self.S_t, self.amax = float(S_t), float(amax_value)
        self.rows, self.cols = rows, cols

    def mma_scales(self) -> np.ndarray:
        return scales_to_mma(self.scales)

    def dequantize(self, rows=None) -> np.ndarray:
        if rows is None:
            return dequantize(self.codes, self.scales, self.S_t)
        rows = np.asarray(rows)
        return dequantize(np.ascontiguousarray(self.codes[rows]),
                          np.ascontiguousarray(self.scales[rows]), self.S_t)


def quantize(x_bf16: np.ndarray, mode: int = RTN, seed: int = 0, stream: int = 0,
             transposed: bool = False, amax_value: float | None = None) -> QTensor:
    """Quantize a BF16 [R, C] tensor (uint16 bit patterns).

    transposed=False: blocks of 16 along C, result is R x C.
    transposed=True: blocks of 16 along R, result is the C x R tensor.
    """
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    R, C = x.shape
    a = amax(x) if amax_value is None else float(np.float32(amax_value))
    S = tensor_scale(a)
    if not transposed:
        assert C % 16 == 0
        codes = np.zeros((R, C // 2), dtype=np.uint8)
        scales = np.zeros((R, C // 16), dtype=np.uint8)
        lib().oracle_quantize_rows(_ptr(x), R, C, C, mode, seed, stream, S, _ptr(codes), _ptr(scales))
        return QTensor(codes, scales, S, a, R, C)
    assert R % 16 == 0
    codes = np.zeros((C, R // 2), dtype=np.uint8)
    scales = np.zeros((C, R // 16), dtype=np.uint8)
    lib().oracle_quantize_cols(_ptr(x), R, C, C, mode, seed, stream, S, _ptr(codes), _ptr(scales))
    return QTensor(codes, scales, S, a, C, R)


def dequantize(codes: np.ndarray, scales: np.ndarray, S_t: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    R = codes.shape[0]
    C = codes.shape[1] * 2
    out = np.empty((R, C), dtype=np.float64)
    lib().oracle_dequantize(_ptr(codes), _ptr(scales), float(S_t), R, C, _ptr(out))
    return out


def mma_scale_offset(r: int, k: int, kb: int) -> int:
    return int(lib().oracle_mma_scale_offset(r, k, kb))


def mma_scale_bytes(rows: int, kb: int) -> int:
    return int(lib().oracle_mma_scale_bytes(rows, kb))


def scales_to_mma(scales_rowmajor: np.ndarray) -> np.ndarray:
    s = np.ascontiguousarray(scales_rowmajor, dtype=np.uint8)
    R, KB = s.shape
    out = np.empty(mma_scale_bytes(R, KB), dtype=np.uint8)
    lib().oracle_scales_to_mma(_ptr(s), R, KB, _ptr(out))
    return out


# ---------------------------------------------------------------------------
# products (FP64 of exactly dequantized operands)
# ---------------------------------------------------------------------------

def fold_branch(P_bf16: np.ndarray, beta: float, S_tA: float, S_tB: float):
    """The branch operand as stored next to the residual's accumulator.

    READING (section 2.1 keeps the L2 L1 subspace in BF16 and adds it to the
    same output): with alpha = fl32(S_tA * S_tB) (1 when that is 0) and
    g = fl32(beta / alpha), the BF16 factor is P~ = bf16(fl32(P * g)), so that
    alpha * (A B^T + P~ Q^T) = A_deq B_deq^T + beta P Q^T up to the one extra
    BF16 rounding of P~.  Returns (alpha, P~ bits)."""
    alpha = np.float32(np.float32(S_tA) * np.float32(S_tB))
    if alpha == 0:
        alpha = np.float32(1.0)
    g = np.float32(np.float32(beta) / alpha)
    prod = bf16_to_f32(P_bf16) * g  # float32 x float32 -> float32, IEEE round to nearest
    return float(alpha), bf16_rn(prod.astype(np.float64))


def gemm(deqA: np.ndarray, deqB: np.ndarray, P_bf16=None, Q_bf16=None, beta: float = 1.0,
         S_tA: float | None = None, S_tB: float | None = None) -> np.ndarray:
    """out = A @ B^T (+ alpha * P~ @ Q^T, see fold_branch), FP64.
    A: M x K and B: N x K dequantized (tensor scales included); P: M x r, Q: N x r
    BF16; S_tA, S_tB: the operands' tensor scales (required with a branch)."""
    out = deqA.astype(np.float64) @ deqB.astype(np.float64).T
    if P_bf16 is not None and P_bf16.shape[1] > 0:
        if S_tA is None or S_tB is None:
            raise ValueError("a branch needs the operands' tensor scales")
        alpha, Pt = fold_branch(P_bf16, beta, S_tA, S_tB)
        P = bf16_to_f32(Pt).astype(np.float64)
        Q = bf16_to_f32(Q_bf16).astype(np.float64)
        out += alpha * (P @ Q.T)
    return out


def branch_factor(x_bf16: np.ndarray, L_bf16_t: np.ndarray) -> np.ndarray:
    """P = bf16(X @ L^T) with the product in FP64.  X: M x K, L: r x K."""
    X = bf16_to_f32(x_bf16).astype(np.float64)
    L = bf16_to_f32(L_bf16_t).astype(np.float64)
    return bf16_rn(X @ L.T)


def lora_svd_split(W_bf16: np.ndarray, r: int):
    """Exact truncated SVD split of W (N x K): returns (W_res, L1, L2) as BF16
    bit patterns with L2 = bf16(U_r Sigma_r) (N x r), L1 = bf16(V_r^T) (r x K),
    W_res = bf16(W - L2 @ L1) (beta = 1)."""
    W = bf16_to_f32(W_bf16).astype(np.float64)
    if r == 0:
        N, K = W.shape
        return np.ascontiguousarray(W_bf16), np.zeros((0, K), np.uint16), np.zeros((N, 0), np.uint16)
    U, S, Vt = np.linalg.svd(W, full_matrices=False)
    L2 = bf16_rn(U[:, :r] * S[:r])
    L1 = bf16_rn(Vt[:r, :])
    low = bf16_to_f32(L2).astype(np.float64) @ bf16_to_f32(L1).astype(np.float64)
    W_res = bf16_rn(W - low)
    return W_res, L1, L2


def linear_fwd(X, W_res, L1, L2, beta: float = 1.0, out_rows=None):
    """Y = bf16( deq(Xq) deq(Wq)^T + beta * bf16(X L1^T) L2^T ), returned as FP64
    before the final rounding (callers round with bf16_rn or compare directly).

    Also returns the quantized operands.  out_rows restricts the product to a
    subset of output rows (the quantization is always of the full tensors)."""
    Xq = quantize(X, RTN)
    Wq = quantize(W_res, RTN)
    rows = slice(None) if out_rows is None else np.asarray(out_rows)
    A = Xq.dequantize(None if out_rows is None else rows)
    B = Wq.dequantize()
    if L1.shape[0] > 0:
        P = branch_factor(np.ascontiguousarray(X[rows]), L1)
        Y = gemm(A, B, P, L2, beta, Xq.S_t, Wq.S_t)
    else:
        Y = gemm(A, B)
    return Y, Xq, Wq


def linear_bwd(dY, X, W_res, L1, L2, seed: int, beta: float = 1.0, dx_rows=None, dw_rows=None):
    """dX = deq(SR_row(dY)) deq(RTN_col(W_res))^T + beta * bf16(dY L2) L1  (M x K)
    dW = deq(SR_col(dY)) deq(RTN_col(X))^T                                 (N x K)
    SR streams: 0 for the row (dX) operand, 1 for the column (dW) operand."""
    dYq = quantize(dY, SR, seed=seed, stream=0)
    WqT = quantize(W_res, RTN, transposed=True)        # K x N
    dYqT = quantize(dY, SR, seed=seed, stream=1, transposed=True)  # N x M
    XqT = quantize(X, RTN, transposed=True)             # K x M
    xr = slice(None) if dx_rows is None else np.asarray(dx_rows)
    A = dYq.dequantize(None if dx_rows is None else xr)
    B = WqT.dequantize()
    if L1.shape[0] > 0:
        P2 = branch_factor(np.ascontiguousarray(dY[xr]), np.ascontiguousarray(L2.T))
        dX = gemm(A, B, P2, np.ascontiguousarray(L1.T), beta, dYq.S_t, WqT.S_t)
    else:
        dX = gemm(A, B)
    wr = slice(None) if dw_rows is None else np.asarray(dw_rows)
    dW = gemm(dYqT.dequantize(None if dw_rows is None else wr), XqT.dequantize())
    return dX, dW, dict(dYq=dYq, WqT=WqT, dYqT=dYqT, XqT=XqT)


def lora_factor_grads(dY64: np.ndarray, X64: np.ndarray, P64: np.ndarray, P2_64: np.ndarray, beta: float = 1.0):
    """Gradients of the branch factors of Y = X W_res^T + beta * P L2^T, P = X L1^T:
        dL2 = beta * dY^T P    (N x r)      dL1 = beta * P'^T X    (r x K),  P' = dY L2.
    All arguments FP64 (the caller decodes the BF16 tensors; P and P' are the rounded
    factors of the BF16 branch).  FP64 products; the results are returned in FP64."""
    dL2 = beta * (dY64.T @ P64)
    dL1 = beta * (P2_64.T @ X64)
    return dL1, dL2


def lora_factor_grads_bf16(dY_bf16, X_bf16, L1_bf16, L2_bf16, beta: float = 1.0):
    """lora_factor_grads on BF16 tensors, with P and P' formed as the branch does it."""
    P = branch_factor(X_bf16, L1_bf16)                                  # T x r, BF16
    P2 = branch_factor(dY_bf16, np.ascontiguousarray(L2_bf16.T))        # T x r, BF16
    f64 = lambda u: bf16_to_f32(u).astype(np.float64)
    dL1, dL2 = lora_factor_grads(f64(dY_bf16), f64(X_bf16), f64(P), f64(P2), beta)
    return dL1, dL2, P, P2


# ---------------------------------------------------------------------------
# Randomized-SVD realignment of the LoRA-SVD subspace (section 2.1)
# ---------------------------------------------------------------------------

def _orth(Y: np.ndarray) -> np.ndarray:
    """An orthonormal basis of the columns of Y (Householder QR)."""
    return np.linalg.qr(Y)[0]


def lora_realign_f64(W_res_bf16, L1_bf16, L2_bf16, beta: float, Omega_bf16, q: int):
    """FP64 (L2', L1', sigma_r, W) before rounding: the randomized range finder with q
    power iterations on W = W_res + beta L2 L1 and the SVD of the small projection."""
    f = lambda u: bf16_to_f32(u).astype(np.float64)
    r = L1_bf16.shape[0]
    W = f(W_res_bf16) + beta * (f(L2_bf16) @ f(L1_bf16))
    Y = W @ f(Omega_bf16)                       # N x s sketch of the range
    for _ in range(q):                          # subspace iteration, orthonormalising each product
        Y = W @ _orth(W.T @ _orth(Y))
    Q = _orth(Y)
    B = Q.T @ W                                 # s x K
    Ub, sig, Vt = np.linalg.svd(B, full_matrices=False)
    U = Q @ Ub[:, :r]
    V = Vt[:r]
    flip = np.sign(V[np.arange(r), np.argmax(np.abs(V), axis=1)])
    flip[flip == 0] = 1.0
    return (U * (sig[:r] * flip)) / beta, V * flip[:, None], sig[:r], W


def lora_realign(W_res_bf16, L1_bf16, L2_bf16, beta: float, Omega_bf16, q: int = 2):
    """BF16 (W_res', L1', L2') with W_res' = bf16(W - beta bf16(L2') bf16(L1'))."""
    L2n, L1n, _, W = lora_realign_f64(W_res_bf16, L1_bf16, L2_bf16, beta, Omega_bf16, q)
    L2b, L1b = bf16_rn(L2n), bf16_rn(L1n)
    f = lambda u: bf16_to_f32(u).astype(np.float64)
    return bf16_rn(W - beta * (f(L2b) @ f(L1b))), L1b, L2b


# ---------------------------------------------------------------------------
# Cholesky-QR of the LoRA-SVD factors (section 2.1)
# ---------------------------------------------------------------------------

def cholesky_lower(G: np.ndarray):
    """Cholesky-Banachiewicz, row by row, FP64: G = L L^T with L lower triangular and a
    positive diagonal.  Returns (L, info): info = 0, or j >= 1 when the leading minor of
    order j is not positive definite (L is then only filled up to row j - 1)."""
    G = np.asarray(G, dtype=np.float64)
    r = G.shape[0]
    L = np.zeros_like(G)
    for i in range(r):
        for j in range(i + 1):
            s = G[i, j] - float(np.dot(L[i, :j], L[j, :j]))
            if i == j:
                if not s > 0.0:
                    return L, i + 1
                L[i, i] = np.sqrt(s)
            else:
                L[i, j] = s / L[j, j]
    return L, 0


def lora_cholqr_f64(L1_bf16: np.ndarray, L2_bf16: np.ndarray):
    """(L1', L2', info) in FP64: L1 L1^T = L L^T, L1' = L^-1 L1, L2' = L2 L."""
    l1 = bf16_to_f32(L1_bf16).astype(np.float64)
    l2 = bf16_to_f32(L2_bf16).astype(np.float64)
    L, info = cholesky_lower(l1 @ l1.T)
    if info:
        return None, None, info
    return np.linalg.solve(L, l1), l2 @ L, 0


def lora_cholqr(L1_bf16: np.ndarray, L2_bf16: np.ndarray):
    """BF16 (L1', L2', info); L1: r x K, L2: N x r (bit patterns)."""
    a, b, info = lora_cholqr_f64(L1_bf16, L2_bf16)
    if info:
        return None, None, info
    return bf16_rn(a), bf16_rn(b), 0


# ---------------------------------------------------------------------------
# Q-AdamW second-moment codec (section 2.2)
# ---------------------------------------------------------------------------

def fwht16(x) -> np.ndarray:
    """Walsh-Hadamard transform (unnormalised, natural order) of each trailing
    16-vector, FP32: four butterfly stages, stage h pairing i and i + h within
    groups of 2h, (a, b) -> (a + b, a - b)."""
    y = np.array(x, dtype=np.float32, copy=True)
    for h in (1, 2, 4, 8):
        v = y.reshape(y.shape[:-1] + (16 // (2 * h), 2, h))
        a = v[..., 0, :].copy()
        b = v[..., 1, :].copy()
        v[..., 0, :] = a + b
        v[..., 1, :] = a - b
    return y


def _tree_sum16(u):
    """FP32 pairwise sum of each trailing 16-vector: adjacent pairs, then pairs of those."""
    t = np.asarray(u, dtype=np.float32)
    while t.shape[-1] > 1:
        t = t[..., 0::2] + t[..., 1::2]
    return t[..., 0]


def vt_transform(v_f32: np.ndarray):
    """The encoder's steps before quantization: returns (h, mean_bf16) with
    u = sqrt(v), mean = bf16(tree_sum(u) / 16) per 16-block, r = u - mean,
    h = fwht16(r) / 4, all FP32."""
    v = np.ascontiguousarray(v_f32, dtype=np.float32)
    R, C = v.shape
    assert C % 16 == 0
    u = np.sqrt(v).reshape(R, C // 16, 16)
    mean = bf16_rn(_tree_sum16(u).astype(np.float64) / 16.0)
    r = u - bf16_to_f32(mean)[..., None]
    h = fwht16(r) * np.float32(0.25)
    return h.reshape(R, C), mean


def quantize_f32(x_f32: np.ndarray) -> QTensor:
    """RTN row quantization of an FP32 [R, C] tensor (blocks of 16 along C)."""
    x = np.ascontiguousarray(x_f32, dtype=np.float32)
    R, C = x.shape
    a = float(np.max(np.abs(x))) if x.size else 0.0
    S = tensor_scale(a)
    codes = np.zeros((R, C // 2), dtype=np.uint8)
    scales = np.zeros((R, C // 16), dtype=np.uint8)
    lib().oracle_quantize_rows_f32(_ptr(x), R, C, S, _ptr(codes), _ptr(scales))
    return QTensor(codes, scales, S, np.float32(a), R, C)


def vt_encode(v_f32: np.ndarray):
    """Encode a non-negative FP32 second moment: (QTensor of the transformed
    residual, BF16 tile means [R, C/16])."""
    h, mean = vt_transform(v_f32)
    return quantize_f32(h), mean


def vt_inverse(h_f32: np.ndarray, mean_bf16: np.ndarray) -> np.ndarray:
    """The decoder's steps after dequantization: u = fwht16(h) / 4 + mean, v = u * u (FP32)."""
    h = np.asarray(h_f32, dtype=np.float32)
    R, C = h.shape
    r = fwht16(h.reshape(R, C // 16, 16)) * np.float32(0.25)
    u = r + bf16_to_f32(mean_bf16)[..., None]
    return (u * u).reshape(R, C)


def vt_decode(q: QTensor, mean_bf16: np.ndarray) -> np.ndarray:
    return vt_inverse(q.dequantize().astype(np.float32), mean_bf16)


# The cubic Newton-Schulz polynomial (1.5 s - 0.5 s^3, converging to 1 with zero slope there)
# is the default: with NVFP4 products the widely used quintic (3.4445, -4.7750, 2.0315) pushes
# singular values past its stable range and diverges in this reading (see the pins).
NS_COEFFS = (1.5, -0.5, 0.0)
NS_STEPS = 12
MUON_QUINTIC = (3.4445, -4.7750, 2.0315)


def p99_clip(x_bf16: np.ndarray, q_num: int = 99, q_den: int = 100) -> np.ndarray:
    """Clip a BF16 tensor to +-v, v = the k-th smallest |x| with k = ceil(N q_num / q_den).
    v is one of the tensor's own values, so the result is exactly BF16."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    mag = (x & 0x7FFF).astype(np.uint16)             # |x| patterns, ordered like |x|
    n = mag.size
    k = (n * q_num + q_den - 1) // q_den
    v = np.sort(mag, axis=None)[k - 1]
    return np.where(mag > v, (x & 0x8000) | v, x).astype(np.uint16)


def _fl32(v):
    return np.asarray(v, dtype=np.float32)


def ns_lincomb(p: float, x_bf16, q: float, y_bf16) -> np.ndarray:
    """bf16(fl32(fl32(p x) + fl32(q y))): the step's linear combinations, no FMA contraction."""
    x = bf16_to_f32(x_bf16)
    y = bf16_to_f32(y_bf16)
    return bf16_rn((_fl32(np.float32(p) * x) + _fl32(np.float32(q) * y)).astype(np.float32).astype(np.float64))


def ns_normalize(G_bf16: np.ndarray) -> np.ndarray:
    """X_0 = bf16(G / max(||G||_F, 1e-7)), the norm and the quotient in FP64."""
    g = bf16_to_f32(G_bf16).astype(np.float64)
    return bf16_rn(g / max(float(np.sqrt(np.sum(g * g))), 1e-7))


def ns_step(X_bf16: np.ndarray, a: float, b: float, c: float, clip: bool = True) -> np.ndarray:
    """One Newton-Schulz step with NVFP4 products (section 2.3):
    A = X X^T, B = b A + c A A, X' = a X + B X; X is m x n, m <= n.  With c = 0 (the
    cubic) the A A product is not formed and B = bf16(fl32(b A))."""
    X = p99_clip(X_bf16) if clip else X_bf16          # the iterate's outliers (not the Gram
    Xq = quantize(X)                                   # matrices, whose largest entries are
    XqT = quantize(X, transposed=True)                 # their diagonal); blocks along n / m
    A = bf16_rn(gemm(Xq.dequantize(), Xq.dequantize()))
    if c != 0.0:
        Aq = quantize(A)
        A2 = bf16_rn(gemm(Aq.dequantize(), Aq.dequantize()))   # A is symmetric: A A = A A^T
        B = ns_lincomb(b, A, c, A2)
    else:                                              # the cubic: B = bf16(fl32(b A))
        B = bf16_rn(_fl32(np.float32(b) * bf16_to_f32(A)).astype(np.float64))
    Bq = quantize(B)                                   # blocks along the contraction dim m
    BX = bf16_rn(gemm(Bq.dequantize(), XqT.dequantize()))
    return ns_lincomb(a, X, 1.0, BX)


def newton_schulz(G_bf16: np.ndarray, steps: int = NS_STEPS, coeffs=NS_COEFFS, clip: bool = True) -> np.ndarray:
    X = ns_normalize(G_bf16)
    for _ in range(steps):
        X = ns_step(X, *coeffs, clip=clip)
    return X


def newton_schulz_fp64(G: np.ndarray, steps: int = NS_STEPS, coeffs=NS_COEFFS) -> np.ndarray:
    """The same iteration in FP64 without quantization or clipping (the exact reference)."""
    a, b, c = coeffs
    X = G / max(float(np.linalg.norm(G)), 1e-7)
    for _ in range(steps):
        A = X @ X.T
        X = a * X + (b * A + c * (A @ A)) @ X
    return X

