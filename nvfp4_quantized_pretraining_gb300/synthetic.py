"""Seeded synthetic inputs shaped like the workloads of the NVFP4 linear
projection (Full-Stack FP4 pages, section 4: a 3B-parameter transformer; the
pages publish no data, so every tensor here is synthetic).

This module only draws random numbers and rounds them to BF16 storage; it
holds none of the quantization or GEMM arithmetic.  Both the CUDA path and
the oracle take their inputs from here, as BF16 bit patterns (numpy uint16),
so the two sides see identical bytes.

Recipes (all from numpy's PCG64 with an explicit seed):
  - activations X ~ N(0, 1), or Student-t(df=3) / sqrt(3) (unit variance);
  - weights W ~ N(0, 0.02^2), optionally with a few columns scaled x20;
  - gradients dY ~ N(0, (1e-3)^2) (1e-3 read as the standard deviation);
  - quantize-sweep tensors ~ N(0, 1) with 0.1% of entries scaled x50;
  - AdamW second moments v = (a_i b_j)^2 z_ij: row and column scales a, b
    ~ lognormal(0, 0.5), z the mean of 8 squared Student-t(3) draws / 3 (a
    heavy-tailed mean-1 factor), times 1e-6;
  - Newton-Schulz iterates X = U diag(s) V^T (m x n) with U, V from the QR
    factorisation of Gaussian matrices and s ~ Uniform[s_lo, s_hi]: a matrix
    part-way to orthogonality.
"""
from __future__ import annotations

import numpy as np
import torch


def to_bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Store float32 values as BF16 (round to nearest even); returns uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_torch(u16: np.ndarray, device=None) -> torch.Tensor:
    """View BF16 bit patterns as a torch.bfloat16 tensor (optionally moved)."""
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def torch_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def normal(shape, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def student_t(shape, df: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    x = rng.standard_t(df, size=shape).astype(np.float32)
    if df > 2:
        x /= np.float32(np.sqrt(df / (df - 2.0)))
    return to_bf16_bits(x)


def with_outlier_entries(shape, frac: float, factor: float, seed: int) -> np.ndarray:
    """N(0,1) with a seeded fraction of entries multiplied by `factor`."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(shape, dtype=np.float32)
    n = x.size
    k = max(1, int(round(frac * n)))
    idx = rng.choice(n, size=k, replace=False)
    x.reshape(-1)[idx] *= np.float32(factor)
    return to_bf16_bits(x)


def weight_with_outlier_columns(n_out: int, n_in: int, std: float, n_cols: int,
                                factor: float, seed: int) -> np.ndarray:
    """W (n_out x n_in) ~ N(0, std^2) with `n_cols` seeded input-feature columns x factor."""
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((n_out, n_in), dtype=np.float32) * np.float32(std)
    cols = rng.choice(n_in, size=n_cols, replace=False)
    w[:, cols] *= np.float32(factor)
    return to_bf16_bits(w)


def gapped_weight(n_out: int, n_in: int, r: int, seed: int) -> np.ndarray:
    """N x K weight with a spectral gap after r: singular values 4..2 for the first r, then
    0.5..0 (random singular vectors), scaled like N(0, 0.02) weights."""
    rng = np.random.default_rng(seed)
    m = min(n_out, n_in)
    U, _ = np.linalg.qr(rng.standard_normal((n_out, m)))
    V, _ = np.linalg.qr(rng.standard_normal((n_in, m)))
    s = np.concatenate([np.linspace(4.0, 2.0, r), np.linspace(0.5, 0.0, m - r)])
    return to_bf16_bits(((U * (s * 0.02 * np.sqrt(m) / 3.0)) @ V.T).astype(np.float32))


def gaussian_test_matrix(n_in: int, s: int, seed: int) -> np.ndarray:
    """The randomized SVD's test matrix Omega (K x s), N(0, 1) stored in BF16."""
    return normal((n_in, s), 1.0, seed)


def spectrum_matrix(m: int, n: int, s_lo: float, s_hi: float, seed: int) -> np.ndarray:
    """m x n with min(m, n) singular values ~ Uniform[s_lo, s_hi] and random singular vectors."""
    rng = np.random.default_rng(seed)
    k = min(m, n)
    U, _ = np.linalg.qr(rng.standard_normal((m, k)))
    V, _ = np.linalg.qr(rng.standard_normal((n, k)))
    s = rng.uniform(s_lo, s_hi, size=k)
    return to_bf16_bits(((U * s) @ V.T).astype(np.float32))


def adam_second_moment(rows: int, cols: int, seed: int) -> np.ndarray:
    """FP32 [rows, cols] non-negative state shaped like AdamW's v_t (see the recipe above)."""
    rng = np.random.default_rng(seed)
    a = np.exp(rng.normal(0.0, 0.5, (rows, 1)))
    b = np.exp(rng.normal(0.0, 0.5, (1, cols)))
    z = np.mean(rng.standard_t(3, (8, rows, cols)) ** 2, axis=0) / 3.0
    return ((a * b) ** 2 * z * 1e-6).astype(np.float32)


# Workload shapes.  Names describe what each is.
SINGLE_FWD_256x512x512 = dict(name="single_fwd_256x512x512_r16", M=256, K=512, N=512, r=16,
                              x="normal", seed=0)
MLP_UP_1B = dict(name="mlp_up_T8192_d2048_f5632_r32", M=8192, K=2048, N=5632, r=32, seed=1)
BLOCK_3B_PROJECTIONS = [
    # (name, N out, K in) for T=16384 tokens, d_model 3072, d_ff 8192
    ("qkv", 9216, 3072),
    ("o", 3072, 3072),
    ("gate_up", 16384, 3072),
    ("down", 3072, 8192),
]
BLOCK_3B = dict(name="block3b_T16384_d3072_ff8192_r64", T=16384, r=64,
                projections=BLOCK_3B_PROJECTIONS)
QUANT_SWEEP_ELEMS = [1 << 20, 1 << 24, 1 << 26, 1 << 28]
# Q-Root Newton-Schulz: the weight-gradient shapes of the 3B block, oriented m <= n
NS_SHAPES_3B = [("qkv", 3072, 9216), ("o", 3072, 3072), ("gate_up", 3072, 16384), ("down", 3072, 8192)]
GEMM_SWEEP = [(2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192),
              (16384, 16384, 16384), (16384, 3072, 8192), (3072, 8192, 16384)]


# Device-side generators for the benchmark's large tensors (seeded torch
# generators on the GPU; same distributions as above, not bit-identical to
# the NumPy versions, which the parity tests use).
def normal_device(shape, std: float, seed: int, device="cuda") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def student_t_device(shape, df: int, seed: int, device="cuda") -> torch.Tensor:
    """Student-t with integer df, t = z / sqrt(chi2_df / df) with chi2_df the sum
    of df squared standard normals; scaled to unit variance."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(int(df)):
        chi2 += torch.randn(shape, generator=g, device=device, dtype=torch.float32) ** 2
    t = z / torch.sqrt(chi2 / df)
    if df > 2:
        t = t / (df / (df - 2.0)) ** 0.5
    return t.to(torch.bfloat16)
