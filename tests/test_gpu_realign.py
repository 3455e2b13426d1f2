"""Randomized-SVD realignment of the LoRA-SVD subspace through the C ABI against
the FP64 oracle (the same algorithm with the same Gaussian test matrix Omega).

The GPU computes in FP32.  Where the spectrum has a gap after r (the rank-r
subspace is well conditioned), FP32 perturbs the subspace by ~1e-6 / gap, so the
GPU's rank-r product beta L2' L1' differs from the oracle's unrounded FP64
product by the BF16 rounding of its two factors: each element of each factor is
off by at most 2^-8 of itself, uniformly spread, so normwise about
2 * 2^-8 / sqrt(3) ~ 4.5e-3 at most (TOL_PRODUCT).  (The individual singular
vectors inside the subspace agree only to FP32 precision over the gaps between
singular values, so the two sides' BF16 factors need not round the same values.)
Where the spectrum is flat (random weights), the singular vectors are ill
conditioned but the singular values are not: they match to TOL_SIGMA = 2e-3
(FP32, plus the BF16 rounding of L2's columns, whose norms carry them).  In
every case the output is checked against itself: W_res' + beta L2' L1' returns
W to the BF16 rounding of W_res' (half a BF16 step, at most 2^-8 of the value,
per element, plus FP32 noise) and L1' has orthonormal rows to BF16 precision."""
TOL_PRODUCT = 4.5e-3
TOL_SIGMA = 2e-3
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


def test_realign_rejects_bad_arguments(F):
    L = F.lib()
    fake, info = 1 << 20, 1 << 21
    call = lambda r=16, s=32, q=2, beta=1.0, ws=1 << 40: L.fp4_lora_realign(
        fake, 512, 256, 256, fake, fake, r, beta, fake, s, q, fake, fake, fake, info, fake, ws, None)
    assert call(s=8) == F.FP4_ERR_UNSUPPORTED_SHAPE      # s < r
    assert call(s=136) == F.FP4_ERR_UNSUPPORTED_SHAPE    # s > 128
    assert call(s=40) == F.FP4_ERR_UNSUPPORTED_SHAPE     # not a multiple of 16
    assert call(q=9) == F.FP4_ERR_INVALID_ARG
    assert call(beta=0.0) == F.FP4_ERR_INVALID_ARG
    assert call(ws=1024) == F.FP4_ERR_WORKSPACE


def f64(oracle_mod, u):
    return oracle_mod.bf16_to_f32(u).astype(np.float64)


def run(F, W_res, L1, L2, Omega, beta, q):
    d = lambda u: S.bits_to_torch(u, DEV)
    Wo, L1o, L2o, info = F.fp4_lora_realign(d(W_res), d(L1), d(L2), d(Omega), beta=beta, q=q)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert int(info.item()) == 0
    return S.torch_to_bits(Wo), S.torch_to_bits(L1o), S.torch_to_bits(L2o)


def check_self(oracle_mod, W, Wo, L1o, L2o, beta):
    wres = f64(oracle_mod, Wo)
    low = beta * f64(oracle_mod, L2o) @ f64(oracle_mod, L1o)
    # the split returns W to the rounding of W_res' (plus FP32 noise far below it)
    assert np.all(np.abs(wres + low - W) <= 2.0 ** -8 * np.abs(wres) + 1e-6 * (np.abs(W).max() + np.abs(low).max()))
    l1 = f64(oracle_mod, L1o)
    assert np.abs(l1 @ l1.T - np.eye(l1.shape[0])).max() < 2e-2


def inputs(oracle_mod, N, K, r, s, kind, seed):
    if kind == "gapped":
        W0 = S.gapped_weight(N, K, r, seed)
    else:
        W0 = S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, seed)
    W_res, L1, L2 = oracle_mod.lora_svd_split(W0, r)
    # the residual drifts away from the split (as under training), so the realignment has work to do
    drift = S.normal((N, K), 0.004, seed + 1)
    W_res = S.to_bf16_bits((oracle_mod.bf16_to_f32(W_res) + oracle_mod.bf16_to_f32(drift)).astype(np.float32))
    return W_res, L1, L2, S.gaussian_test_matrix(K, s, seed + 2)


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,r,s,q,beta", [
    (384, 512, 16, 32, 2, 1.0), (1024, 768, 32, 48, 2, 0.5), (640, 1280, 48, 64, 1, 1.0), (768, 512, 64, 128, 3, 2.0),
    (648, 392, 32, 48, 2, 1.0),  # ragged 128-row tiles and 32-wide K stages in the tensor-core products
    (512, 256, 16, 16, 2, 1.0),  # sketch width 16: the narrowest tensor-core product (N = 16)
    (514, 384, 16, 32, 2, 1.0),  # N not a multiple of 4: the W^T products fall back to the FP32 GEMM
])
def test_realign_gapped_matches_oracle(F, oracle_mod, N, K, r, s, q, beta):
    W_res, L1, L2, Om = inputs(oracle_mod, N, K, r, s, "gapped", N + K + r)
    Wo, L1o, L2o = run(F, W_res, L1, L2, Om, beta, q)
    L2n, L1n, _, W = oracle_mod.lora_realign_f64(W_res, L1, L2, beta, Om, q)
    want = beta * L2n @ L1n
    got = beta * f64(oracle_mod, L2o) @ f64(oracle_mod, L1o)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < TOL_PRODUCT
    check_self(oracle_mod, W, Wo, L1o, L2o, beta)


@pytest.mark.gpu
@pytest.mark.parametrize("N,K,r,s,q", [(512, 384, 16, 32, 2), (1536, 1024, 64, 80, 2)])
def test_realign_flat_spectrum_properties(F, oracle_mod, N, K, r, s, q):
    W_res, L1, L2, Om = inputs(oracle_mod, N, K, r, s, "flat", 3 * N + K)
    Wo, L1o, L2o = run(F, W_res, L1, L2, Om, 1.0, q)
    L2n, L1n, sig, W = oracle_mod.lora_realign_f64(W_res, L1, L2, 1.0, Om, q)
    got_sig = np.linalg.norm(f64(oracle_mod, L2o), axis=0)   # L1' rows are unit, so |L2' col j| = sigma_j
    assert np.max(np.abs(got_sig - sig) / sig) < TOL_SIGMA
    check_self(oracle_mod, W, Wo, L1o, L2o, 1.0)


@pytest.mark.gpu
def test_realign_reports_a_failed_factorisation_and_writes_nothing(F, oracle_mod):
    N, K, r, s = 256, 256, 16, 32
    W_res, L1, L2, Om = inputs(oracle_mod, N, K, r, s, "flat", 5)
    W_res[7, 9] = 0x7FC0  # a NaN: the first Gram matrix has a NaN pivot
    d = lambda u: S.bits_to_torch(u, DEV)
    outs = (torch.full((N, K), 3.0, dtype=torch.bfloat16, device=DEV),
            torch.full((r, K), 3.0, dtype=torch.bfloat16, device=DEV),
            torch.full((N, r), 3.0, dtype=torch.bfloat16, device=DEV))
    _, _, _, info = F.fp4_lora_realign(d(W_res), d(L1), d(L2), d(Om), out=outs)
    torch.cuda.synchronize()
    assert int(info.item()) != 0
    assert all(bool((o == 3.0).all()) for o in outs)


@pytest.mark.gpu
def test_realign_full_size_gate_up(F, oracle_mod):
    # the 3B block's gate_up weight (16384 x 3072) at rank 64 with 16 columns of oversampling
    N, K, r, s, q = 16384, 3072, 64, 80, 2
    W0 = S.weight_with_outlier_columns(N, K, 0.02, 4, 20.0, 61)
    zeros1, zeros2 = np.zeros((r, K), np.uint16), np.zeros((N, r), np.uint16)
    Om = S.gaussian_test_matrix(K, s, 62)
    Wo, L1o, L2o = run(F, W0, zeros1, zeros2, Om, 1.0, q)
    L2n, L1n, sig, W = oracle_mod.lora_realign_f64(W0, zeros1, zeros2, 1.0, Om, q)
    got_sig = np.linalg.norm(f64(oracle_mod, L2o), axis=0)
    assert np.max(np.abs(got_sig - sig) / sig) < TOL_SIGMA
    check_self(oracle_mod, W, Wo, L1o, L2o, 1.0)
