"""Python binding of the GB300 NVFP4 linear-projection library.

Argument marshalling only: every computation runs in the CUDA kernels of
``libnvfp4_gb300.so`` (built in-tree by ``build.py``); PyTorch provides device
memory and streams.  Names and semantics follow ``include/nvfp4_gb300.h``.
There is no CPU fallback: if the library is missing or cannot be loaded,
importing a call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnvfp4_gb300.so")

FP4_OK = 0
FP4_ERR_INVALID_ARG = 1
FP4_ERR_MISALIGNED = 2
FP4_ERR_UNSUPPORTED_SHAPE = 3
FP4_ERR_CUDA = 4
FP4_ERR_TIMEOUT = 5
FP4_ERR_WORKSPACE = 6
STATUS_NAMES = {0: "FP4_OK", 1: "FP4_ERR_INVALID_ARG", 2: "FP4_ERR_MISALIGNED", 3: "FP4_ERR_UNSUPPORTED_SHAPE",
                4: "FP4_ERR_CUDA", 5: "FP4_ERR_TIMEOUT", 6: "FP4_ERR_WORKSPACE"}
RTN = 0
SR = 1
OUT_BF16 = 0
OUT_F32 = 1

EXPORTS = ["fp4_scale_bytes", "fp4_amax", "fp4_quantize", "fp4_quantize_transposed", "fp4_quantize_dual",
           "fp4_gemm_blockscaled", "fp4_gemm_split_workspace", "fp4_gemm_blockscaled_workspace",
           "fp4_gemm_blockscaled_ws", "fp4_branch_factor", "fp4_linear_fwd_workspace", "fp4_linear_bwd_workspace",
           "fp4_linear_fwd", "fp4_linear_fwd_noalloc", "fp4_linear_bwd", "fp4_lora_factor_grad_workspace",
           "fp4_lora_factor_grad", "fp4_lora_cholqr_workspace", "fp4_lora_cholqr", "fp4_lora_realign_workspace",
           "fp4_lora_realign", "fp4_newton_schulz_workspace", "fp4_newton_schulz", "fp4_qadamw_v_encode",
           "fp4_qadamw_v_decode", "fp4_check_status", "fp4_last_error", "fp4_launch_count",
           "fp4_debug_convert", "fp4_debug_sr_round", "fp4_debug_force_counter64", "fp4_mma_peak_probe"]


class FP4Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class CTensor(ctypes.Structure):
    """Mirror of ``fp4_tensor``."""
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library {LIB_PATH} is missing: run nvfp4_quantized_pretraining_gb300.build.build()")
    L = ctypes.CDLL(LIB_PATH)
    P, i64, u64, u32, i32, f32 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32,
                                  ctypes.c_int, ctypes.c_float)
    T = ctypes.POINTER(CTensor)
    sig = {
        "fp4_scale_bytes": (i64, [i64, i64]),
        "fp4_amax": (i32, [P, i64, i64, i64, P, P]),
        "fp4_quantize": (i32, [P, i64, i64, i64, i32, u64, u32, P, T, P]),
        "fp4_quantize_transposed": (i32, [P, i64, i64, i64, i32, u64, u32, P, T, P]),
        "fp4_quantize_dual": (i32, [P, i64, i64, i64, i32, u64, u32, u32, P, T, T, P]),
        "fp4_gemm_blockscaled": (i32, [T, T, P, P, i32, f32, P, i32, i64, P]),
        "fp4_gemm_split_workspace": (ctypes.c_size_t, []),
        "fp4_gemm_blockscaled_workspace": (ctypes.c_size_t, [i64, i32]),
        "fp4_gemm_blockscaled_ws": (i32, [T, T, P, P, i32, f32, P, i32, i64, P, ctypes.c_size_t, P]),
        "fp4_branch_factor": (i32, [P, i64, i64, i64, P, i32, P, P, P]),
        "fp4_linear_fwd_workspace": (ctypes.c_size_t, [i64, i64, i64, i32]),
        "fp4_linear_bwd_workspace": (ctypes.c_size_t, [i64, i64, i64, i32]),
        "fp4_linear_fwd": (i32, [P, i64, i64, i64, T, P, P, i32, f32, P, i64, T, P, ctypes.c_size_t, P]),
        "fp4_linear_fwd_noalloc": (i32, [P, i64, i64, i64, T, P, P, i32, f32, P, i64, T, P]),
        "fp4_linear_bwd": (i32, [P, i64, i64, i64, T, T, P, P, i32, f32, u64, P, i64, P, i32, i64, P,
                                 ctypes.c_size_t, P]),
        "fp4_lora_factor_grad_workspace": (ctypes.c_size_t, [i64, i64, i32]),
        "fp4_lora_factor_grad": (i32, [P, i64, i64, i64, P, i32, f32, P, i64, i32, P, ctypes.c_size_t, P]),
        "fp4_lora_cholqr_workspace": (ctypes.c_size_t, [i64, i32]),
        "fp4_lora_realign_workspace": (ctypes.c_size_t, [i64, i64, i32, i32]),
        "fp4_lora_realign": (i32, [P, i64, i64, i64, P, P, i32, f32, P, i32, i32, P, P, P, P, P, ctypes.c_size_t,
                                   P]),
        "fp4_lora_cholqr": (i32, [P, i64, i64, P, i64, i32, P, P, P, P, ctypes.c_size_t, P]),
        "fp4_newton_schulz_workspace": (ctypes.c_size_t, [i64, i64, f32]),
        "fp4_newton_schulz": (i32, [P, i64, i64, i64, i32, i32, f32, f32, f32, i32, P, i64, P, ctypes.c_size_t,
                                    P]),
        "fp4_qadamw_v_encode": (i32, [P, i64, i64, i64, T, P, P]),
        "fp4_qadamw_v_decode": (i32, [T, P, P, i64, P]),
        "fp4_check_status": (i32, [P]),
        "fp4_last_error": (ctypes.c_char_p, []),
        "fp4_launch_count": (u64, []),
        "fp4_debug_convert": (i32, [P, i64, P, P, P]),
        "fp4_debug_sr_round": (i32, [P, P, i64, P, P]),
        "fp4_debug_force_counter64": (None, [i32]),
        "fp4_mma_peak_probe": (i32, [i32, i32, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int) -> None:
    if status != FP4_OK:
        raise FP4Error(status, lib().fp4_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _bf16_2d(x: torch.Tensor, name: str):
    if x.dtype != torch.bfloat16 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D CUDA bfloat16 tensor with unit column stride")
    return x.shape[0], x.shape[1], x.stride(0)


def _check_out(t: torch.Tensor, shape, dtypes, device, name: str) -> None:
    """A caller-owned output: exact shape and dtype, on ``device``, unit column stride."""
    if not isinstance(dtypes, tuple):
        dtypes = (dtypes,)
    if (t.dim() != 2 or tuple(t.shape) != tuple(shape) or t.dtype not in dtypes or t.device != device
            or t.stride(1) != 1 or t.stride(0) < shape[1]):
        raise ValueError(f"{name} must be a {shape[0]} x {shape[1]} {'/'.join(str(d) for d in dtypes)} tensor on "
                         f"{device} with unit column stride (got {tuple(t.shape)} {t.dtype} on {t.device}, "
                         f"strides {t.stride()})")


def _check_factor(t, shape, device, name: str) -> None:
    """A LoRA factor read by the kernels with a pitch equal to its width: contiguous BF16."""
    if (t.dtype != torch.bfloat16 or t.device != device or not t.is_contiguous()
            or tuple(t.shape) != tuple(shape)):
        raise ValueError(f"{name} must be a contiguous {shape[0]} x {shape[1]} bfloat16 tensor on {device} "
                         f"(got {tuple(t.shape)} {t.dtype} on {t.device})")


def _check_qtensor(q, rows: int, cols: int, name: str) -> None:
    if (q.rows, q.cols) != (rows, cols):
        raise ValueError(f"{name} is {q.rows} x {q.cols}, expected {rows} x {cols}")


def _branch_factors(L1, L2, N: int, K: int, device):
    """Rank of the branch (0 without one) after checking L1 (r x K) and L2 (N x r)."""
    if L1 is None and L2 is None:
        return 0
    if L1 is None or L2 is None:
        raise ValueError("L1 and L2 must both be given or both be None")
    r = L1.shape[0]
    _check_factor(L1, (r, K), device, "L1")
    _check_factor(L2, (N, r), device, "L2")
    return r


def scale_bytes(rows: int, cols: int) -> int:
    return int(lib().fp4_scale_bytes(rows, cols))


@dataclass
class NVFP4Tensor:
    """Device buffers of one NVFP4 tensor (rows x cols, blocks of 16 along cols).

    codes: uint8 [rows, cols/2]; scales: uint8 [fp4_scale_bytes] in the MMA
    layout; scale: float32 [2] = (S_t, amax)."""
    codes: torch.Tensor
    scales: torch.Tensor
    scale: torch.Tensor
    rows: int
    cols: int

    @staticmethod
    def empty(rows: int, cols: int, device="cuda") -> "NVFP4Tensor":
        codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
        scales = torch.empty(scale_bytes(rows, cols), dtype=torch.uint8, device=device)
        scale = torch.zeros(2, dtype=torch.float32, device=device)
        return NVFP4Tensor(codes, scales, scale, rows, cols)

    def c(self) -> CTensor:
        return CTensor(self.codes.data_ptr(), self.scales.data_ptr(), self.scale.data_ptr(), self.rows, self.cols)

    @property
    def tensor_scale(self) -> float:
        return float(self.scale[0])


def fp4_amax(x: torch.Tensor, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    R, C, ld = _bf16_2d(x, "x")
    out = torch.empty(1, dtype=torch.float32, device=x.device) if out is None else out
    _check(lib().fp4_amax(x.data_ptr(), R, C, ld, out.data_ptr(), _stream(stream)))
    return out


def fp4_quantize(x, round_mode=RTN, seed=0, sr_stream=0, amax=None, out=None, stream=None) -> NVFP4Tensor:
    R, C, ld = _bf16_2d(x, "x")
    out = NVFP4Tensor.empty(R, C, x.device) if out is None else out
    ct = out.c()
    _check(lib().fp4_quantize(x.data_ptr(), R, C, ld, round_mode, seed, sr_stream, _ptr(amax),
                              ctypes.byref(ct), _stream(stream)))
    return out


def fp4_quantize_transposed(x, round_mode=RTN, seed=0, sr_stream=1, amax=None, out=None, stream=None) -> NVFP4Tensor:
    R, C, ld = _bf16_2d(x, "x")
    out = NVFP4Tensor.empty(C, R, x.device) if out is None else out
    ct = out.c()
    _check(lib().fp4_quantize_transposed(x.data_ptr(), R, C, ld, round_mode, seed, sr_stream, _ptr(amax),
                                         ctypes.byref(ct), _stream(stream)))
    return out


def fp4_quantize_dual(x, round_mode=RTN, seed=0, sr_stream_row=0, sr_stream_col=1, amax=None,
                      out_row=None, out_col=None, stream=None):
    R, C, ld = _bf16_2d(x, "x")
    out_row = NVFP4Tensor.empty(R, C, x.device) if out_row is None else out_row
    out_col = NVFP4Tensor.empty(C, R, x.device) if out_col is None else out_col
    cr, cc = out_row.c(), out_col.c()
    _check(lib().fp4_quantize_dual(x.data_ptr(), R, C, ld, round_mode, seed, sr_stream_row, sr_stream_col,
                                   _ptr(amax), ctypes.byref(cr), ctypes.byref(cc), _stream(stream)))
    return out_row, out_col


def _gemm_args(A, B, P, Q, out, out_dtype):
    r = 0 if P is None else P.shape[1]
    if out is None:
        out = torch.empty((A.rows, B.rows), dtype=out_dtype, device=A.codes.device)
    _check_out(out, (A.rows, B.rows), (torch.bfloat16, torch.float32), A.codes.device, "out")
    if r:
        _check_factor(P, (A.rows, r), A.codes.device, "P")
        _check_factor(Q, (B.rows, r), A.codes.device, "Q")
    return r, out, OUT_F32 if out.dtype == torch.float32 else OUT_BF16


def fp4_gemm_blockscaled(A: NVFP4Tensor, B: NVFP4Tensor, P=None, Q=None, beta=1.0, out=None,
                         out_dtype=torch.bfloat16, stream=None) -> torch.Tensor:
    r, out, c_dtype = _gemm_args(A, B, P, Q, out, out_dtype)
    ca, cb = A.c(), B.c()
    _check(lib().fp4_gemm_blockscaled(ctypes.byref(ca), ctypes.byref(cb), _ptr(P), _ptr(Q), r, float(beta),
                                      out.data_ptr(), c_dtype, out.stride(0), _stream(stream)))
    return out


def gemm_split_workspace() -> int:
    return int(lib().fp4_gemm_split_workspace())


def gemm_blockscaled_workspace(M, r) -> int:
    return int(lib().fp4_gemm_blockscaled_workspace(M, r))


def fp4_gemm_blockscaled_ws(A: NVFP4Tensor, B: NVFP4Tensor, P=None, Q=None, beta=1.0, out=None,
                            out_dtype=torch.bfloat16, workspace=None, stream=None) -> torch.Tensor:
    """fp4_gemm_blockscaled with a workspace (allocated here when not given): the branch fold by a
    launch of its own, and the split tail."""
    r, out, c_dtype = _gemm_args(A, B, P, Q, out, out_dtype)
    if workspace is None:
        workspace = torch.empty(gemm_blockscaled_workspace(A.rows, r), dtype=torch.uint8, device=A.codes.device)
    ca, cb = A.c(), B.c()
    _check(lib().fp4_gemm_blockscaled_ws(ctypes.byref(ca), ctypes.byref(cb), _ptr(P), _ptr(Q), r, float(beta),
                                         out.data_ptr(), c_dtype, out.stride(0), workspace.data_ptr(),
                                         workspace.numel(), _stream(stream)))
    return out


def fp4_branch_factor(X: torch.Tensor, L: torch.Tensor, out=None, amax=None, stream=None) -> torch.Tensor:
    """P = bf16(X L^T); with ``amax`` (a 1-element float32 device tensor) also max |X|."""
    M, K, ldx = _bf16_2d(X, "X")
    r = L.shape[0]
    _check_factor(L, (r, K), X.device, "L")
    out = torch.empty((M, r), dtype=torch.bfloat16, device=X.device) if out is None else out
    _check_factor(out, (M, r), X.device, "out")
    _check(lib().fp4_branch_factor(X.data_ptr(), M, K, ldx, L.data_ptr(), r, out.data_ptr(), _ptr(amax),
                                   _stream(stream)))
    return out


def linear_fwd_workspace(M, N, K, r) -> int:
    return int(lib().fp4_linear_fwd_workspace(M, N, K, r))


def linear_bwd_workspace(M, N, K, r) -> int:
    return int(lib().fp4_linear_bwd_workspace(M, N, K, r))


def fp4_linear_fwd(X, Wq: NVFP4Tensor, L1=None, L2=None, beta=1.0, Y=None, xqT_saved=None, workspace=None,
                   stream=None):
    """Y = X W^T with W = W_res + beta L2 L1 (Wq = NVFP4 of W_res).  Returns (Y, xqT_saved)."""
    M, K, ldx = _bf16_2d(X, "X")
    N = Wq.rows
    _check_qtensor(Wq, N, K, "Wq")
    r = _branch_factors(L1, L2, N, K, X.device)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=X.device) if Y is None else Y
    _check_out(Y, (M, N), torch.bfloat16, X.device, "Y")
    xqT_saved = NVFP4Tensor.empty(K, M, X.device) if xqT_saved is None else xqT_saved
    _check_qtensor(xqT_saved, K, M, "xqT_saved")
    if workspace is None:  # with the room for the GEMM's split tail
        workspace = torch.empty(linear_fwd_workspace(M, N, K, r) + gemm_split_workspace(), dtype=torch.uint8,
                                device=X.device)
    cw, cx = Wq.c(), xqT_saved.c()
    _check(lib().fp4_linear_fwd(X.data_ptr(), M, K, ldx, ctypes.byref(cw), _ptr(L1), _ptr(L2), r, float(beta),
                                Y.data_ptr(), Y.stride(0), ctypes.byref(cx), workspace.data_ptr(),
                                workspace.numel(), _stream(stream)))
    return Y, xqT_saved


def fp4_linear_fwd_noalloc(X, Wq: NVFP4Tensor, L1, L2, beta, Y, xqT_saved, stream=None):
    """fp4_linear_fwd with the library's static scratch instead of a workspace.
    Y (M x N BF16) and xqT_saved (K x M) are caller-owned; nothing is allocated."""
    M, K, ldx = _bf16_2d(X, "X")
    N = Wq.rows
    _check_qtensor(Wq, N, K, "Wq")
    r = _branch_factors(L1, L2, N, K, X.device)
    _check_out(Y, (M, N), torch.bfloat16, X.device, "Y")
    _check_qtensor(xqT_saved, K, M, "xqT_saved")
    cw, cx = Wq.c(), xqT_saved.c()
    _check(lib().fp4_linear_fwd_noalloc(X.data_ptr(), M, K, ldx, ctypes.byref(cw), _ptr(L1), _ptr(L2), r,
                                        float(beta), Y.data_ptr(), Y.stride(0), ctypes.byref(cx), _stream(stream)))
    return Y, xqT_saved


def fp4_linear_bwd(dY, WqT: NVFP4Tensor, xqT_saved: NVFP4Tensor, L1=None, L2=None, beta=1.0, seed=0,
                   dX=None, dW=None, dw_dtype=torch.bfloat16, workspace=None, stream=None):
    """dX = dY W, dW_res = dY^T X.  Returns (dX, dW)."""
    M, N, lddy = _bf16_2d(dY, "dY")
    K = WqT.rows
    _check_qtensor(WqT, K, N, "WqT")
    _check_qtensor(xqT_saved, K, M, "xqT_saved")
    r = _branch_factors(L1, L2, N, K, dY.device)
    dX = torch.empty((M, K), dtype=torch.bfloat16, device=dY.device) if dX is None else dX
    dW = torch.empty((N, K), dtype=dw_dtype, device=dY.device) if dW is None else dW
    _check_out(dX, (M, K), torch.bfloat16, dY.device, "dX")
    _check_out(dW, (N, K), (torch.bfloat16, torch.float32), dY.device, "dW")
    if workspace is None:  # with the room for the GEMMs' split tail
        workspace = torch.empty(linear_bwd_workspace(M, N, K, r) + gemm_split_workspace(), dtype=torch.uint8,
                                device=dY.device)
    cw, cx = WqT.c(), xqT_saved.c()
    _check(lib().fp4_linear_bwd(dY.data_ptr(), M, N, lddy, ctypes.byref(cw), ctypes.byref(cx), _ptr(L1), _ptr(L2),
                                r, float(beta), seed, dX.data_ptr(), dX.stride(0), dW.data_ptr(),
                                OUT_F32 if dW.dtype == torch.float32 else OUT_BF16, dW.stride(0),
                                workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return dX, dW


def fp4_lora_factor_grad(A: torch.Tensor, B: torch.Tensor, beta: float = 1.0, transpose: bool = False, out=None,
                         workspace=None, stream=None) -> torch.Tensor:
    """C = beta * A^T B (FP32) for A: T x M and B: T x r BF16; r x M when ``transpose``.
    dL2 = fp4_lora_factor_grad(dY, P, beta); dL1 = fp4_lora_factor_grad(X, P2, beta, transpose=True)."""
    T, M, lda = _bf16_2d(A, "A")
    assert B.dtype == torch.bfloat16 and B.is_contiguous() and B.shape[0] == T
    r = B.shape[1]
    if out is None:
        out = torch.empty((r, M) if transpose else (M, r), dtype=torch.float32, device=A.device)
    need = lib().fp4_lora_factor_grad_workspace(T, M, r)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=A.device) if workspace is None else workspace
    _check(lib().fp4_lora_factor_grad(A.data_ptr(), T, M, lda, B.data_ptr(), r, float(beta), out.data_ptr(),
                                      out.stride(0), 1 if transpose else 0, workspace.data_ptr(), workspace.numel(),
                                      _stream(stream)))
    return out


def lora_factor_grads(X, dY, P, P2, beta: float = 1.0, stream=None):
    """(dL1, dL2) of the LoRA-SVD branch: dL1 = beta P2^T X (r x K), dL2 = beta dY^T P (N x r), FP32."""
    dL2 = fp4_lora_factor_grad(dY, P, beta, stream=stream)
    dL1 = fp4_lora_factor_grad(X, P2, beta, transpose=True, stream=stream)
    return dL1, dL2


def fp4_lora_cholqr(L1: torch.Tensor, L2: torch.Tensor, L1_out=None, L2_out=None, info=None, workspace=None,
                    stream=None):
    """Cholesky-QR of the LoRA-SVD factors: L1 (r x K) <- L^-1 L1, L2 (N x r) <- L2 L with
    L1 L1^T = L L^T (beta L2 L1 unchanged).  Pass L1_out=L1, L2_out=L2 to update in place.
    Returns (L1_out, L2_out, info); info (device int32) is 0 or the order of the first
    non-positive-definite leading minor, in which case the outputs are not written."""
    r, K, ld1 = _bf16_2d(L1, "L1")
    N = L2.shape[0]
    assert L2.dtype == torch.bfloat16 and L2.is_contiguous() and L2.shape[1] == r
    if L1_out is None:  # the C ABI writes L1_out with L1's row pitch
        L1_out = torch.empty((r, ld1), dtype=torch.bfloat16, device=L1.device)[:, :K]
    L2_out = torch.empty_like(L2) if L2_out is None else L2_out
    assert L1_out.stride(0) == ld1
    info = torch.zeros(1, dtype=torch.int32, device=L1.device) if info is None else info
    need = lib().fp4_lora_cholqr_workspace(K, r)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=L1.device) if workspace is None else workspace
    _check(lib().fp4_lora_cholqr(L1.data_ptr(), K, ld1, L2.data_ptr(), N, r, L1_out.data_ptr(), L2_out.data_ptr(),
                                 info.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return L1_out, L2_out, info


def fp4_lora_realign(W_res: torch.Tensor, L1: torch.Tensor, L2: torch.Tensor, Omega: torch.Tensor,
                     beta: float = 1.0, q: int = 2, out=None, info=None, workspace=None, stream=None):
    """Randomized-SVD realignment of W = W_res + beta L2 L1 with the test matrix Omega (K x s, BF16)
    and q power iterations.  Returns (W_res', L1', L2', info); pass out=(W_res, L1, L2) to update in
    place.  info (device int32) is nonzero when a Cholesky factorisation failed (nothing written)."""
    N, K, ldw = _bf16_2d(W_res, "W_res")
    r = L1.shape[0]
    s = Omega.shape[1]
    for t, shape in ((L1, (r, K)), (L2, (N, r)), (Omega, (K, s))):
        assert t.dtype == torch.bfloat16 and t.is_contiguous() and tuple(t.shape) == shape
    if out is None:
        out = (torch.empty((N, ldw), dtype=torch.bfloat16, device=W_res.device)[:, :K], torch.empty_like(L1),
               torch.empty_like(L2))
    Wo, L1o, L2o = out
    assert Wo.stride(0) == ldw
    info = torch.zeros(1, dtype=torch.int32, device=W_res.device) if info is None else info
    need = lib().fp4_lora_realign_workspace(N, K, r, s)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=W_res.device) if workspace is None else workspace
    _check(lib().fp4_lora_realign(W_res.data_ptr(), N, K, ldw, L1.data_ptr(), L2.data_ptr(), r, float(beta),
                                  Omega.data_ptr(), s, int(q), Wo.data_ptr(), L1o.data_ptr(), L2o.data_ptr(),
                                  info.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream(stream)))
    return Wo, L1o, L2o, info


NS_COEFFS = (1.5, -0.5, 0.0)  # the cubic Newton-Schulz polynomial
NS_STEPS = 12


def newton_schulz_workspace(m: int, n: int, c: float = 0.0) -> int:
    return int(lib().fp4_newton_schulz_workspace(m, n, float(c)))


def fp4_newton_schulz(G: torch.Tensor, steps: int = NS_STEPS, coeffs=NS_COEFFS, clip: bool = True,
                      normalize: bool = True, out=None, workspace=None, stream=None) -> torch.Tensor:
    """Q-Root orthogonalisation of an m x n BF16 matrix (m <= n the efficient orientation):
    X_0 = G / ||G||_F (``normalize``), then ``steps`` Newton-Schulz steps
    X <- a X + (b A + c A^2) X, A = X X^T, every product in NVFP4, the iterate p99-clipped
    (``clip``) at the start of each step.  Returns the BF16 result (``out`` if given)."""
    m, n, ldg = _bf16_2d(G, "G")
    a, b, c = (float(v) for v in coeffs)
    if out is None:
        out = torch.empty((m, n), dtype=torch.bfloat16, device=G.device)
    mo, no, ldx = _bf16_2d(out, "out")
    if (mo, no) != (m, n):
        raise ValueError(f"out is {mo} x {no}, expected {m} x {n}")
    need = newton_schulz_workspace(m, n, c)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=G.device) if workspace is None else workspace
    _check(lib().fp4_newton_schulz(G.data_ptr(), m, n, ldg, 1 if normalize else 0, int(steps), a, b, c,
                                   1 if clip else 0, out.data_ptr(), ldx, workspace.data_ptr(), workspace.numel(),
                                   _stream(stream)))
    return out


def _f32_2d(x: torch.Tensor, name: str):
    if x.dtype != torch.float32 or x.dim() != 2 or not x.is_cuda or x.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D CUDA float32 tensor with unit column stride")
    return x.shape[0], x.shape[1], x.stride(0)


def _check_means(mean: torch.Tensor, R: int, C: int) -> None:
    if (mean.dtype != torch.bfloat16 or not mean.is_cuda or not mean.is_contiguous()
            or tuple(mean.shape) != (R, C // 16)):
        raise ValueError(f"mean must be a contiguous CUDA bfloat16 tensor of shape ({R}, {C // 16})")


def fp4_qadamw_v_encode(v: torch.Tensor, out: NVFP4Tensor | None = None, mean: torch.Tensor | None = None,
                        stream=None):
    """Encode AdamW's second moment v (FP32, >= 0): sqrt, BF16 mean per 16-element block,
    16-point Hadamard of the residual, NVFP4.  Returns (NVFP4Tensor, BF16 means [R, C/16])."""
    R, C, ldv = _f32_2d(v, "v")
    out = NVFP4Tensor.empty(R, C, v.device) if out is None else out
    if mean is None:
        mean = torch.empty((R, C // 16), dtype=torch.bfloat16, device=v.device)
    _check_means(mean, R, C)
    if (out.rows, out.cols) != (R, C):
        raise ValueError(f"out is {out.rows} x {out.cols}, expected {R} x {C}")
    ct = out.c()
    _check(lib().fp4_qadamw_v_encode(v.data_ptr(), R, C, ldv, ctypes.byref(ct), mean.data_ptr(), _stream(stream)))
    return out, mean


def fp4_qadamw_v_decode(q: NVFP4Tensor, mean: torch.Tensor, out: torch.Tensor | None = None,
                        stream=None) -> torch.Tensor:
    """Rebuild v (FP32) from fp4_qadamw_v_encode's output."""
    _check_means(mean, q.rows, q.cols)
    if out is None:
        out = torch.empty((q.rows, q.cols), dtype=torch.float32, device=mean.device)
    R, C, ldo = _f32_2d(out, "out")
    if (R, C) != (q.rows, q.cols):
        raise ValueError(f"out is {R} x {C}, expected {q.rows} x {q.cols}")
    ct = q.c()
    _check(lib().fp4_qadamw_v_decode(ctypes.byref(ct), mean.data_ptr(), out.data_ptr(), ldo, _stream(stream)))
    return out


def fp4_check_status(stream=None) -> None:
    _check(lib().fp4_check_status(_stream(stream)))


def fp4_last_error() -> str:
    return lib().fp4_last_error().decode()


def fp4_launch_count() -> int:
    return int(lib().fp4_launch_count())


def fp4_debug_convert(x: torch.Tensor, stream=None):
    n = x.numel()
    e2m1 = torch.empty(n, dtype=torch.uint8, device=x.device)
    e4m3 = torch.empty(n, dtype=torch.uint8, device=x.device)
    _check(lib().fp4_debug_convert(x.data_ptr(), n, e2m1.data_ptr(), e4m3.data_ptr(), _stream(stream)))
    return e2m1, e4m3


def fp4_debug_sr_round(y: torch.Tensor, rnd16: torch.Tensor, stream=None) -> torch.Tensor:
    """Stochastic rounding of float32 ``y`` with the given 16-bit random values
    (int32 or uint16 tensor on the same device); E2M1 codes, one per byte."""
    assert y.dtype == torch.float32 and y.is_contiguous() and y.numel() > 0
    r = rnd16.to(torch.int32).to(torch.int16).contiguous()  # same bits as uint16
    assert r.numel() == y.numel() and r.device == y.device
    out = torch.empty(y.numel(), dtype=torch.uint8, device=y.device)
    _check(lib().fp4_debug_sr_round(y.data_ptr(), r.data_ptr(), y.numel(), out.data_ptr(), _stream(stream)))
    return out


def fp4_mma_peak_probe(n: int = 256, iters: int = 20000, stream=None) -> dict:
    """Times the dense NVFP4 MMA probe with CUDA events; returns TFLOP/s."""
    st = torch.cuda.current_stream() if stream is None else stream
    sms = ctypes.c_int(0)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _check(lib().fp4_mma_peak_probe(n, max(1, iters // 10), ctypes.byref(sms), st.cuda_stream))  # warm-up
    e0.record(st)
    _check(lib().fp4_mma_peak_probe(n, iters, ctypes.byref(sms), st.cuda_stream))
    e1.record(st)
    e1.synchronize()
    fp4_check_status(st)
    ms = e0.elapsed_time(e1)
    flops = sms.value * 4 * iters * 2 * 128 * n * 64
    return {"n": n, "iters": iters, "sms": sms.value, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12}
