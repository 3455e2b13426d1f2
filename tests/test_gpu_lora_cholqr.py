"""Cholesky-QR of the LoRA-SVD factors through the C ABI against the oracle
(FP64 Gram, Cholesky and triangular solve; each factor rounded to BF16 once).

The GPU works in FP32: the Gram entries are sums of exact BF16 products, the
factorisation and the forward substitution of an r x r system (r <= 64) add
normwise relative errors of order r * 2^-24 * cond(L1 L1^T) (~4e-6 for rows near
orthonormal, ~4e-4 at cond = 100), and each output is one FP32 dot product.
Normwise that stays below TOL = 2e-3 relative Frobenius after the BF16 rounding.
Elementwise, an output formed by cancellation can have a large relative error,
so the bound of one BF16 step per element is checked only for near-orthonormal
factors (cond ~ 1), where the FP32 error of every element stays far below half a
BF16 step."""
TOL = 2e-3
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


def test_lora_cholqr_rejects_bad_arguments(F):
    L = F.lib()
    fake, info = 1 << 20, 1 << 21
    assert L.fp4_lora_cholqr(fake, 256, 256, fake, 64, 8, fake, fake, info, fake, 1 << 30, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_lora_cholqr(fake, 256, 250, fake, 64, 16, fake, fake, info, fake, 1 << 30, None) == \
        F.FP4_ERR_INVALID_ARG  # ld1 < K
    assert L.fp4_lora_cholqr(fake, 256, 256, fake, 64, 16, fake, fake, None, fake, 1 << 30, None) == \
        F.FP4_ERR_INVALID_ARG
    assert L.fp4_lora_cholqr(fake, 256, 256, fake, 64, 16, fake, fake, info, fake, 64, None) == \
        F.FP4_ERR_WORKSPACE


def ulp_distance(a_bits, b_bits):
    """Distance in BF16 steps between finite patterns of the same sign."""
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    sa = np.where(a & 0x8000, -(a & 0x7FFF), a & 0x7FFF)
    sb = np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)
    return np.abs(sa - sb)


def factors(oracle_mod, r, K, N, kind, seed):
    if kind == "svd":
        W = S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, seed)
        _, L1, L2 = oracle_mod.lora_svd_split(W, r)
        return L1, L2
    if kind == "near":  # rows near orthonormal, as after a few small updates of an SVD split
        return S.spectrum_matrix(r, K, 0.95, 1.05, seed), S.normal((N, r), 0.05, seed + 1)
    # a factor part-way off orthonormal: U diag(s) V^T rows with s in [1, 10] (cond(G) <= 100)
    return S.spectrum_matrix(r, K, 1.0, 10.0, seed), S.normal((N, r), 0.05, seed + 1)


@pytest.mark.gpu
@pytest.mark.parametrize("r,K,N,pad,kind", [
    (16, 256, 128, 0, "svd"), (32, 1001, 384, 7, "spread"),   # ragged K (pitch 1008)
    (48, 2048, 640, 0, "spread"), (64, 3072, 16384, 0, "near"),  # the 3B gate_up factors
    (64, 8192, 3072, 8, "spread"),
])
def test_lora_cholqr_matches_oracle(F, oracle_mod, r, K, N, pad, kind):
    L1, L2 = factors(oracle_mod, r, K, N, kind, r + K)
    full = torch.zeros((r, K + pad), dtype=torch.bfloat16, device=DEV)
    full[:, :K] = S.bits_to_torch(L1, DEV)
    L1d = full[:, :K]
    L2d = S.bits_to_torch(L2, DEV)
    a, b, info = F.fp4_lora_cholqr(L1d, L2d)
    torch.cuda.synchronize()
    assert int(info.item()) == 0
    wa, wb, winfo = oracle_mod.lora_cholqr(L1, L2)
    assert winfo == 0
    ga, gb = S.torch_to_bits(a), S.torch_to_bits(b)
    if kind in ("svd", "near"):
        assert ulp_distance(ga, wa).max() <= 1 and ulp_distance(gb, wb).max() <= 1
    f = lambda u: oracle_mod.bf16_to_f32(u).astype(np.float64)
    rel = lambda g, w: np.linalg.norm(f(g) - f(w)) / np.linalg.norm(f(w))
    assert rel(ga, wa) < TOL and rel(gb, wb) < TOL
    # properties of the result itself: orthonormal rows, the product kept (BF16 rounding only)
    assert np.abs(f(ga) @ f(ga).T - np.eye(r)).max() < 2e-2
    assert np.linalg.norm(f(gb) @ f(ga) - f(L2) @ f(L1)) / np.linalg.norm(f(L2) @ f(L1)) < 1e-2
    # in place gives the same bits
    L1i = torch.empty_like(full)[:, :K]  # same row pitch as L1d
    L1i.copy_(L1d)
    L2i = L2d.clone()
    F.fp4_lora_cholqr(L1i, L2i, L1_out=L1i, L2_out=L2i)
    torch.cuda.synchronize()
    assert torch.equal(L1i, a) and torch.equal(L2i, b)


@pytest.mark.gpu
def test_lora_cholqr_reports_a_singular_gram_and_writes_nothing(F, oracle_mod):
    r, K, N = 32, 512, 256
    L1 = S.normal((r, K), 0.1, 40)
    L1[5] = 0  # a zero row: the 6th pivot is exactly 0
    L2 = S.normal((N, r), 0.1, 41)
    out1 = torch.full((r, K), 7.0, dtype=torch.bfloat16, device=DEV)
    out2 = torch.full((N, r), 7.0, dtype=torch.bfloat16, device=DEV)
    _, _, info = F.fp4_lora_cholqr(S.bits_to_torch(L1, DEV), S.bits_to_torch(L2, DEV), L1_out=out1, L2_out=out2)
    torch.cuda.synchronize()
    assert int(info.item()) == 6 == oracle_mod.lora_cholqr(L1, L2)[2]
    assert bool((out1 == 7.0).all()) and bool((out2 == 7.0).all())


@pytest.mark.gpu
def test_lora_cholqr_waits_for_a_copy_queued_after_the_previous_call(F, oracle_mod):
    # Calls queued back to back with a copy between them: the second call's first kernel must be
    # ordered after the copy (which is not a kernel), not only after the first call's kernels.
    r, K, N = 16, 256, 128
    L1, L2 = factors(oracle_mod, r, K, N, "svd", r + K)
    L1d, L2d = S.bits_to_torch(L1, DEV), S.bits_to_torch(L2, DEV)
    a, b, _ = F.fp4_lora_cholqr(L1d, L2d)
    torch.cuda.synchronize()
    for _ in range(4):
        F.fp4_lora_cholqr(L1d, L2d)
        F.fp4_lora_cholqr(L1d, L2d)
        L1i, L2i = L1d.clone(), L2d.clone()
        _, _, info = F.fp4_lora_cholqr(L1i, L2i, L1_out=L1i, L2_out=L2i)
        torch.cuda.synchronize()
        assert int(info.item()) == 0
        assert torch.equal(L1i, a) and torch.equal(L2i, b)
