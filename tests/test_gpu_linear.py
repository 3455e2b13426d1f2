"""GPU parity of the composed NVFP4 linear projection (forward: Y; backward:
dX and dW_res) with the LoRA-SVD BF16 branch, through the C ABI, against the
oracle on the same seeded inputs: relative Frobenius error below 1e-3, and every
compared element and 32-column chunk within the bounds of parity_util."""
import numpy as np
import pytest
import torch

from nvfp4_quantized_pretraining_gb300 import synthetic as S
from parity_util import assert_elementwise

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 1e-3


@pytest.fixture(scope="module")
def F():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_pretraining_gb300 as F
    return F


def dev(u16):
    return S.bits_to_torch(u16, DEV)


def rel(got, want):
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def run_layer(F, oracle_mod, M, K, N, r, seed, x_kind="normal", dx_rows=None, dw_rows=None, beta=1.0,
              w_kind="outlier_cols", dw_dtype=torch.float32):
    X = S.normal((M, K), 1.0, seed) if x_kind == "normal" else S.student_t((M, K), 3.0, seed)
    W = (S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, seed + 1) if w_kind == "outlier_cols"
         else S.normal((N, K), 0.02, seed + 1))
    dY = S.normal((M, N), 1e-3, seed + 2)
    Wres, L1, L2 = oracle_mod.lora_svd_split(W, r)
    Wq, WqT = F.fp4_quantize_dual(dev(Wres))
    l1 = dev(L1) if r else None
    l2 = dev(L2) if r else None
    Y, xqT = F.fp4_linear_fwd(dev(X), Wq, l1, l2, beta=beta)
    dX, dW = F.fp4_linear_bwd(dev(dY), WqT, xqT, l1, l2, beta=beta, seed=seed, dw_dtype=dw_dtype)
    torch.cuda.synchronize()
    F.fp4_check_status()
    # the saved column form of X equals the oracle's RTN column quantization
    oq = oracle_mod.quantize(X, 0, transposed=True)
    assert np.array_equal(xqT.codes.cpu().numpy(), oq.codes)
    Y_ref, Xq, Wq_o = oracle_mod.linear_fwd(X, Wres, L1, L2, beta=beta, out_rows=dx_rows)
    dX_ref, dW_ref, q = oracle_mod.linear_bwd(dY, X, Wres, L1, L2, seed=seed, beta=beta, dx_rows=dx_rows,
                                              dw_rows=dw_rows)
    sel_x = slice(None) if dx_rows is None else dx_rows
    sel_w = slice(None) if dw_rows is None else dw_rows
    bf = lambda a: oracle_mod.bf16_to_f32(oracle_mod.bf16_rn(a)).astype(np.float64)
    got = dict(Y=f64(Y)[sel_x], dX=f64(dX)[sel_x], dW=f64(dW)[sel_w])
    dw_bf16 = dw_dtype == torch.bfloat16
    errs = dict(Y=rel(got["Y"], bf(Y_ref)), dX=rel(got["dX"], bf(dX_ref)),
                dW=rel(got["dW"], bf(dW_ref) if dw_bf16 else dW_ref))
    assert all(v < TOL for v in errs.values()), errs
    # element-wise: sum |a||b| over the quantized operands (+ the branch's |P||Q|)
    a64 = lambda u: np.abs(oracle_mod.bf16_to_f32(u).astype(np.float64))
    rows = None if dx_rows is None else dx_rows
    sY = np.abs(Xq.dequantize(rows)) @ np.abs(Wq_o.dequantize()).T
    sX = np.abs(q["dYq"].dequantize(rows)) @ np.abs(q["WqT"].dequantize()).T
    bY = bX = 0.0
    if r:
        # the branch: |P||L2|^T and |P'||L1|; P and P' come from the GPU's branch factor, each
        # element within one BF16 step of the oracle's (2^-7 of itself at most)
        bY = abs(beta) * (a64(oracle_mod.branch_factor(np.ascontiguousarray(X[sel_x]), L1)) @ a64(L2).T)
        bX = abs(beta) * (a64(oracle_mod.branch_factor(np.ascontiguousarray(dY[sel_x]), np.ascontiguousarray(L2.T)))
                          @ a64(L1))
        sY += bY
        sX += bX
    sW = np.abs(q["dYqT"].dequantize(None if dw_rows is None else dw_rows)) @ np.abs(q["XqT"].dequantize()).T
    assert_elementwise(got["Y"], Y_ref, sY, K + r, True, "Y", rounded=bf(Y_ref), extra=2.0 ** -7 * bY)
    assert_elementwise(got["dX"], dX_ref, sX, N + r, True, "dX", rounded=bf(dX_ref), extra=2.0 ** -7 * bX)
    assert_elementwise(got["dW"], dW_ref, sW, M, dw_bf16, "dW", rounded=bf(dW_ref) if dw_bf16 else None)
    return errs


def test_single_forward_shape(F, oracle_mod):
    run_layer(F, oracle_mod, 256, 512, 512, 16, seed=0)


@pytest.mark.parametrize("r", [0, 16, 32, 48, 64])
def test_ranks(F, oracle_mod, r):
    run_layer(F, oracle_mod, 384, 256, 256, r, seed=10 + r, beta=0.5 if r else 1.0)


def test_mlp_up_1b_sampled(F, oracle_mod):
    rng = np.random.default_rng(1)
    run_layer(F, oracle_mod, 8192, 2048, 5632, 32, seed=1, dx_rows=np.sort(rng.choice(8192, 64, replace=False)),
              dw_rows=np.sort(rng.choice(5632, 64, replace=False)))


def sample_rows(n_rows, n, rng):
    # n rows, four of them in the last 256: the GEMMs with M > N split their last partial wave
    # of 256 x 256 tiles along K, and those tiles lie in the last tile row
    tail = np.array([n_rows - 256, n_rows - 150, n_rows - 77, n_rows - 1])
    return np.sort(np.concatenate([rng.choice(n_rows - 256, n - tail.size, replace=False), tail]))


# The four projections of the 3B-class block (T = 16384 tokens, rank 64, Student-t activations),
# each through fp4_linear_fwd / fp4_linear_bwd at full size (workspaces with the split-tail room,
# as the benchmark runs them); 32 sampled rows of Y, dX and dW.
@pytest.mark.parametrize("name,N,K", S.BLOCK_3B_PROJECTIONS)
def test_block3b_projection_sampled(F, oracle_mod, name, N, K):
    seed = {"qkv": 5, "o": 3, "gate_up": 7, "down": 9}[name]
    rng = np.random.default_rng(seed)
    run_layer(F, oracle_mod, 16384, K, N, 64, seed=seed, x_kind="student", dx_rows=sample_rows(16384, 32, rng),
              dw_rows=sample_rows(N, 32, rng), w_kind="normal", dw_dtype=torch.bfloat16)


def test_lora_branch_lowers_error_vs_exact(F, oracle_mod):
    # quality proxy on the single-forward shape: with the rank-16 BF16 subspace the
    # output is closer to the exact BF16 product than plain NVFP4 of W
    M, K, N = 256, 512, 512
    X = S.normal((M, K), 1.0, 0)
    W = S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, 1)
    exact = oracle_mod.bf16_to_f32(X).astype(np.float64) @ oracle_mod.bf16_to_f32(W).astype(np.float64).T
    Wq0, _ = F.fp4_quantize_dual(dev(W))
    Y0, _ = F.fp4_linear_fwd(dev(X), Wq0)
    Wres, L1, L2 = oracle_mod.lora_svd_split(W, 16)
    Wq1, _ = F.fp4_quantize_dual(dev(Wres))
    Y1, _ = F.fp4_linear_fwd(dev(X), Wq1, dev(L1), dev(L2))
    torch.cuda.synchronize()
    assert rel(f64(Y1), exact) < rel(f64(Y0), exact)


def test_smoke_entry(F):
    import __graft_entry__
    __graft_entry__.smoke()
