"""Q-Root Newton-Schulz with NVFP4 products through the C ABI against the oracle.

Bit-exact: the normalisation X_0 = bf16(G / ||G||_F) (the FP64 norm reduces in a
different order on the two sides; the BF16 result differs only if a quotient lies
within ~1e-12 relative of a BF16 midpoint) and the p99 clip (integer selection).

A full step compares within TOL_STEP relative Frobenius error.  The two sides
differ only in the products' accumulation (FP32 in the tensor cores, FP64 in the
oracle, each then rounded to BF16): an element of A = Q(X)Q(X)^T or of B X moves
by one BF16 ulp (2^-8 relative) where the accumulation error straddles a rounding
boundary, and the quantization of B sees such a move only for an element on an
E2M1 or E4M3 boundary.  Those are a small fraction of the elements, each off by at
most about 2^-8 of its value, so the relative Frobenius error stays near 1e-4;
TOL_STEP = 2e-3 leaves room for a flipped block scale.

Chains of steps re-quantize at every step, so a single flipped code early on makes
the two chains diverge at the level of the NVFP4 noise (which the oracle pins put
at ~12% of the FP64 iteration after 12 steps).  Chains are therefore checked by
properties: the same distance to the FP64 iteration as the oracle chain, singular
values near the scalar map of the initial spectrum, and bit-for-bit repeatability.
"""
TOL_STEP = 2e-3
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


def f64(oracle_mod, bits):
    return oracle_mod.bf16_to_f32(bits).astype(np.float64)


def padded(bits, pad):
    """A device BF16 view of `bits` with the row pitch widened by `pad` columns."""
    m, n = bits.shape
    full = torch.zeros((m, n + pad), dtype=torch.bfloat16, device=DEV)
    full[:, :n] = S.bits_to_torch(bits, DEV)
    return full[:, :n]


def test_newton_schulz_rejects_bad_arguments(F):
    # host-side checks only; nothing is launched
    L = F.lib()
    fake, big = 1 << 20, 1 << 40
    args = lambda m=128, n=256, steps=1, norm=1, clip=1, ws=big: (fake, m, n, n, norm, steps, 1.5, -0.5, 0.0, clip,
                                                                  fake, n, fake, ws, None)
    assert L.fp4_newton_schulz(*args(m=100)) == F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_newton_schulz(*args(n=200)) == F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_newton_schulz(*args(steps=-1)) == F.FP4_ERR_INVALID_ARG
    assert L.fp4_newton_schulz(*args(clip=2)) == F.FP4_ERR_INVALID_ARG
    assert L.fp4_newton_schulz(*args(ws=64)) == F.FP4_ERR_WORKSPACE
    # the quintic needs room for A's NVFP4 form and A^2
    assert L.fp4_newton_schulz_workspace(256, 512, -4.775) > L.fp4_newton_schulz_workspace(256, 512, 0.0)


@pytest.mark.gpu
@pytest.mark.parametrize("m,n,pad,kind", [
    (128, 256, 0, "normal"), (256, 384, 64, "normal"),
    (128, 512, 0, "outlier"),   # one huge entry: most quotients fall below 2^-100 (the FP64 path)
    (256, 256, 0, "huge"),      # ||G|| > 2^100: squares beyond binary32, the FP64 quotient throughout
    (384, 1024, 8, "tiny"),     # ||G|| < 1e-7: the clamped norm
])
def test_normalize_bit_exact(F, oracle_mod, m, n, pad, kind):
    G = S.normal((m, n), 1e-3, m + n)
    if kind == "outlier":
        g = oracle_mod.bf16_to_f32(G).copy()
        g[3, 5] = 1e34
        G = S.to_bf16_bits(g)
    elif kind == "huge":
        G = S.normal((m, n), 1e36, m + n)
    elif kind == "tiny":
        G = S.normal((m, n), 1e-12, m + n)
    X = F.fp4_newton_schulz(padded(G, pad), steps=0)
    torch.cuda.synchronize()
    F.fp4_check_status()
    want = oracle_mod.ns_normalize(G)
    got = S.torch_to_bits(X)
    assert np.array_equal(got, want), int(np.sum(got != want))


@pytest.mark.gpu
@pytest.mark.parametrize("m,n", [(128, 256), (256, 640)])
def test_p99_clip_bit_exact(F, oracle_mod, m, n):
    # one step with a = 1 and a negligible b: X_1 = bf16(X_c + tiny) = X_c, the clipped iterate
    X0 = S.with_outlier_entries((m, n), 0.003, 30.0, m * n)
    coeffs = (1.0, 2.0 ** -60, 0.0)
    X = F.fp4_newton_schulz(S.bits_to_torch(X0, DEV), steps=1, coeffs=coeffs, normalize=False)
    torch.cuda.synchronize()
    F.fp4_check_status()
    got = S.torch_to_bits(X)
    assert np.array_equal(got, oracle_mod.p99_clip(X0))
    assert np.array_equal(got, oracle_mod.ns_step(X0, *coeffs, clip=True))
    assert not np.array_equal(got, X0)  # the outliers were clipped


@pytest.mark.gpu
@pytest.mark.parametrize("m,n,coeffs,clip", [
    (128, 256, (1.5, -0.5, 0.0), True),
    (256, 512, (1.5, -0.5, 0.0), False),
    (384, 768, (1.5, -0.5, 0.0), True),
    (256, 512, (15 / 8, -10 / 8, 3 / 8), True),     # quintic: the A^2 product and its lincomb
    (128, 384, (3.4445, -4.7750, 2.0315), False),
    (384, 256, (1.5, -0.5, 0.0), True),              # m > n: a tall iterate (m x m Gram matrix of rank n)
])
def test_one_step_matches_oracle(F, oracle_mod, m, n, coeffs, clip):
    X0 = S.spectrum_matrix(m, n, 0.3, 1.1, m + 7 * n)
    X = F.fp4_newton_schulz(S.bits_to_torch(X0, DEV), steps=1, coeffs=coeffs, clip=clip, normalize=False)
    torch.cuda.synchronize()
    F.fp4_check_status()
    want = f64(oracle_mod, oracle_mod.ns_step(X0, *coeffs, clip=clip))
    got = f64(oracle_mod, S.torch_to_bits(X))
    assert rel(got, want) < TOL_STEP


def scalar_map(s, coeffs, steps):
    a, b, c = coeffs
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


@pytest.mark.gpu
@pytest.mark.parametrize("m,n", [(128, 256), (256, 512)])
def test_chain_properties(F, oracle_mod, m, n):
    G = S.normal((m, n), 1e-3, 5 * m + n)
    Gd = S.bits_to_torch(G, DEV)
    X = F.fp4_newton_schulz(Gd)
    X2 = F.fp4_newton_schulz(Gd)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert torch.equal(X, X2)  # deterministic
    got = f64(oracle_mod, S.torch_to_bits(X))
    g = f64(oracle_mod, G)
    ref = oracle_mod.newton_schulz_fp64(g)
    orc = f64(oracle_mod, oracle_mod.newton_schulz(G))
    # as close to the FP64 iteration as the oracle's own NVFP4 chain (within its pinned bound)
    assert rel(got, ref) < max(0.2, 1.25 * rel(orc, ref))
    sv = np.linalg.svd(got, compute_uv=False)
    want_sv = np.sort(scalar_map(np.linalg.svd(g / np.linalg.norm(g), compute_uv=False), F.NS_COEFFS,
                                 F.NS_STEPS))[::-1]
    assert 0.5 < sv.min() and sv.max() < 1.3
    assert np.max(np.abs(sv - want_sv)) < 0.25


@pytest.mark.gpu
def test_full_size_down_projection_gradient(F, oracle_mod):
    # the 3B block's down-projection gradient shape, as timed by the benchmark: the
    # normalisation bit-exact on every element, the chain by its spectrum
    m, n = 3072, 8192
    G = S.normal((m, n), 1e-3, 77)
    Gd = S.bits_to_torch(G, DEV)
    X0 = F.fp4_newton_schulz(Gd, steps=0)
    X = F.fp4_newton_schulz(Gd)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert np.array_equal(S.torch_to_bits(X0), oracle_mod.ns_normalize(G))
    got = f64(oracle_mod, S.torch_to_bits(X))
    assert np.all(np.isfinite(got))
    sv = np.sqrt(np.clip(np.linalg.eigvalsh(got @ got.T), 0.0, None))
    g = f64(oracle_mod, G)
    s0 = np.sqrt(np.clip(np.linalg.eigvalsh(g @ g.T), 0.0, None)) / np.linalg.norm(g)
    want_sv = scalar_map(s0, F.NS_COEFFS, F.NS_STEPS)
    assert np.max(np.abs(np.sort(sv) - np.sort(want_sv))) < 0.25
    assert sv.max() < 1.3
