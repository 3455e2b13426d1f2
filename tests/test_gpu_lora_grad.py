"""Gradients of the LoRA-SVD branch factors through the C ABI against the oracle:
C = beta * A^T B over the token dimension (dL2 = beta dY^T P, dL1 = beta P'^T X),
FP32 results within a relative Frobenius error of 1e-4 of the FP64 products of the
same BF16 operands, and bit-for-bit reproducible.  The bound: the BF16 products are
exact in FP32, and an FP32 running sum over T terms has a relative error of at most
about T * 2^-24 (1e-3 at T = 16384) and typically sqrt(T) * 2^-24; one CTA summing
16384 tokens measured 1.9e-5."""
TOL = 1e-4
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_quantized_pretraining_gb300 import synthetic as S

DEV = "cuda"


@pytest.fixture(scope="module")
def F():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_pretraining_gb300 as F
    return F


def rel(got, want):
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def test_lora_factor_grad_rejects_bad_shapes(F):
    # host-side checks only; nothing is launched
    fake = 1 << 20
    L = F.lib()
    assert L.fp4_lora_factor_grad(fake, 64, 100, 128, fake, 16, 1.0, fake, 16, 0, fake, 1 << 30, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE  # M % 128
    assert L.fp4_lora_factor_grad(fake, 64, 128, 128, fake, 8, 1.0, fake, 16, 0, fake, 1 << 30, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE  # r
    assert L.fp4_lora_factor_grad(fake, 64, 128, 128, fake, 16, 1.0, fake, 16, 0, fake, 64, None) == \
        F.FP4_ERR_WORKSPACE
    assert L.fp4_lora_factor_grad(fake, 64, 128, 128, fake, 16, 1.0, fake, 100, 1, fake, 1 << 30, None) == \
        F.FP4_ERR_INVALID_ARG  # ldc < M for the transposed output


@pytest.mark.gpu
@pytest.mark.parametrize("T,M,r,transpose", [
    (64, 128, 16, False), (200, 384, 32, True),     # ragged token count (zero-filled tail)
    (1024, 256, 48, False), (4096, 3072, 64, True),  # many token splits
    (16384, 1024, 64, False), (16384, 16384, 64, False),  # few splits; the gate_up dL2 shape
])
def test_lora_factor_grad_matches_fp64(F, oracle_mod, T, M, r, transpose):
    rng_seed = T + M + r
    A_bits = S.normal((T, M), 1.0, rng_seed)
    B_bits = S.normal((T, r), 0.5, rng_seed + 1)
    A, B = S.bits_to_torch(A_bits, DEV), S.bits_to_torch(B_bits, DEV)
    beta = 0.75
    C = F.fp4_lora_factor_grad(A, B, beta, transpose=transpose)
    C2 = F.fp4_lora_factor_grad(A, B, beta, transpose=transpose)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert torch.equal(C, C2)  # deterministic
    a = oracle_mod.bf16_to_f32(A_bits).astype(np.float64)
    b = oracle_mod.bf16_to_f32(B_bits).astype(np.float64)
    want = beta * (a.T @ b)
    got = C.cpu().numpy().astype(np.float64)
    if transpose:
        got = got.T
    assert got.shape == want.shape
    assert rel(got, want) < TOL


@pytest.mark.gpu
def test_lora_factor_grads_of_a_layer(F, oracle_mod):
    # dL1, dL2 of one layer with the oracle's own P and P' (BF16), against the oracle
    T, K, N, r, beta = 512, 256, 384, 16, 1.25
    X = S.normal((T, K), 1.0, 3)
    dY = S.normal((T, N), 1e-3, 4)
    W = S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, 5)
    _, L1, L2 = oracle_mod.lora_svd_split(W, r)
    dL1_ref, dL2_ref, P, P2 = oracle_mod.lora_factor_grads_bf16(dY, X, L1, L2, beta)
    dev = lambda u: S.bits_to_torch(u, DEV)
    dL1, dL2 = F.lora_factor_grads(dev(X), dev(dY), dev(P), dev(P2), beta)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert dL1.shape == (r, K) and dL2.shape == (N, r)
    assert rel(dL1.cpu().numpy().astype(np.float64), dL1_ref) < TOL
    assert rel(dL2.cpu().numpy().astype(np.float64), dL2_ref) < TOL
