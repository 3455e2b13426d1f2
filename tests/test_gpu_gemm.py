"""GPU parity of the block-scaled NVFP4 GEMM (with the fused BF16 branch) and
of the BF16 branch-factor GEMM against the oracle's FP64 products of the same
operands.  Tolerance: relative Frobenius error 1e-3 (FP32 output against the
FP64 result; BF16 output against the FP64 result rounded to BF16), and every
element and every 32-column chunk within the bounds of parity_util (one BF16
step plus (K + r) 2^-24 sum |a||b|; 8e-3 per chunk)."""
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


def quantize_both(F, oracle_mod, x, mode=0, seed=0, stream=0):
    g = F.fp4_quantize(dev(x), round_mode=mode, seed=seed, sr_stream=stream)
    o = oracle_mod.quantize(x, mode, seed=seed, stream=stream)
    torch.cuda.synchronize()
    assert np.array_equal(g.codes.cpu().numpy(), o.codes)
    assert np.array_equal(g.scales.cpu().numpy(), oracle_mod.scales_to_mma(o.scales))
    return g, o


def check_gemm(F, oracle_mod, M, N, K, r, out_dtype, beta, seed, rows=None, a_kind="normal", split=False):
    A = S.normal((M, K), 1.0, seed) if a_kind == "normal" else S.with_outlier_entries((M, K), 0.001, 50.0, seed)
    B = S.normal((N, K), 1.0, seed + 1)
    ga, oa = quantize_both(F, oracle_mod, A)
    gb, ob = quantize_both(F, oracle_mod, B)
    P = S.normal((M, r), 1.0, seed + 2) if r else None
    Q = S.normal((N, r), 1.0, seed + 3) if r else None
    gemm = F.fp4_gemm_blockscaled_ws if split else F.fp4_gemm_blockscaled
    C = gemm(ga, gb, None if P is None else dev(P), None if Q is None else dev(Q), beta=beta, out_dtype=out_dtype)
    torch.cuda.synchronize()
    F.fp4_check_status()
    sel = slice(None) if rows is None else rows
    dA, dB = oa.dequantize(rows), ob.dequantize()
    Psel = None if P is None else np.ascontiguousarray(P[sel])
    exact = oracle_mod.gemm(dA, dB, Psel, Q, beta, oa.S_t, ob.S_t)
    got = C.float().cpu().numpy().astype(np.float64)[sel]
    bf16_out = out_dtype == torch.bfloat16
    ref = oracle_mod.bf16_to_f32(oracle_mod.bf16_rn(exact)).astype(np.float64) if bf16_out else exact
    e = rel(got, ref)
    assert e < TOL, (M, N, K, r, e)
    abs_sum = np.abs(dA) @ np.abs(dB).T
    if r:
        abs_sum += abs(beta) * (np.abs(oracle_mod.bf16_to_f32(Psel).astype(np.float64))
                                @ np.abs(oracle_mod.bf16_to_f32(Q).astype(np.float64)).T)
    assert_elementwise(got, exact, abs_sum, K + r, bf16_out, f"GEMM {M}x{N}x{K} r={r}", rounded=ref)
    return e


@pytest.mark.parametrize("M,N,K,r", [
    (128, 128, 64, 0), (128, 128, 256, 0), (128, 128, 512, 16), (256, 384, 512, 16),
    (384, 256, 320, 32),      # K not a multiple of the 256-wide stage
    (128, 256, 1024, 48), (512, 512, 2048, 64),
    (2048, 2560, 512, 0),     # more tiles than SMs: persistent schedule wraps
    (256, 512, 512, 16),      # single-forward shape (X 256x512, W 512x512, rank 16)
    (256, 256, 128, 16),      # 2-SM kernel with K below one 256-wide stage (B scales by bulk copies)
])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_small(F, oracle_mod, M, N, K, r, out_dtype):
    check_gemm(F, oracle_mod, M, N, K, r, out_dtype, beta=0.75 if r else 1.0, seed=M + N + K + r)


def test_gemm_outliers_and_rank0_equivalence(F, oracle_mod):
    check_gemm(F, oracle_mod, 256, 256, 1024, 0, torch.float32, 1.0, seed=3, a_kind="outliers")
    # r > 0 with a zero branch gives the same output as r = 0 (bit for bit)
    A = S.normal((256, 512), 1.0, 4)
    B = S.normal((128, 512), 1.0, 5)
    ga, gb = F.fp4_quantize(dev(A)), F.fp4_quantize(dev(B))
    c0 = F.fp4_gemm_blockscaled(ga, gb, out_dtype=torch.float32)
    Z1 = torch.zeros((256, 32), dtype=torch.bfloat16, device=DEV)
    Z2 = torch.zeros((128, 32), dtype=torch.bfloat16, device=DEV)
    c1 = F.fp4_gemm_blockscaled(ga, gb, Z1, Z2, beta=3.0, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1)


@pytest.mark.parametrize("M,N,K,r", [(512, 512, 2048, 64), (384, 256, 512, 32), (256, 256, 320, 16)])
def test_gemm_prefolded_branch_equals_in_kernel_fold(F, M, N, K, r):
    # fp4_gemm_blockscaled_ws writes P~ by a launch of its own and the GEMM loads it as it is
    # (the 2-SM kernel and, for 384 x 256, the one-CTA kernel); no split at these sizes, so the
    # output equals the in-kernel fold's bit for bit
    ga = F.fp4_quantize(dev(S.normal((M, K), 1.0, M + r)))
    gb = F.fp4_quantize(dev(S.normal((N, K), 1.0, N + r)))
    P = dev(S.normal((M, r), 1.0, 5))
    Q = dev(S.normal((N, r), 1.0, 6))
    for out_dtype in (torch.bfloat16, torch.float32):
        c0 = F.fp4_gemm_blockscaled(ga, gb, P, Q, beta=0.3, out_dtype=out_dtype)
        n0 = F.fp4_launch_count()
        c1 = F.fp4_gemm_blockscaled_ws(ga, gb, P, Q, beta=0.3, out_dtype=out_dtype)
        assert F.fp4_launch_count() - n0 == 2  # the fold and the GEMM
        torch.cuda.synchronize()
        F.fp4_check_status()
        assert torch.equal(c0.view(torch.int16) if out_dtype == torch.bfloat16 else c0,
                           c1.view(torch.int16) if out_dtype == torch.bfloat16 else c1)


def test_gemm_strided_output(F, oracle_mod):
    A = S.normal((128, 256), 1.0, 6)
    B = S.normal((256, 256), 1.0, 7)
    ga, oa = quantize_both(F, oracle_mod, A)
    gb, ob = quantize_both(F, oracle_mod, B)
    big = torch.full((128, 384), 7.0, dtype=torch.float32, device=DEV)
    F.fp4_gemm_blockscaled(ga, gb, out=big[:, 64:320])
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(oa.dequantize(), ob.dequantize())
    got = big.cpu().numpy().astype(np.float64)
    assert rel(got[:, 64:320], ref) < TOL
    assert np.all(got[:, :64] == 7.0) and np.all(got[:, 320:] == 7.0)


def test_gemm_strided_bf16_output_pair_path(F, oracle_mod):
    # M, N multiples of 256 take the 2-SM kernel, whose BF16 tiles leave by TMA stores
    A = S.normal((512, 512), 1.0, 8)
    B = S.normal((512, 512), 1.0, 9)
    ga, oa = quantize_both(F, oracle_mod, A)
    gb, ob = quantize_both(F, oracle_mod, B)
    big = torch.full((512, 640), 7.0, dtype=torch.bfloat16, device=DEV)
    F.fp4_gemm_blockscaled(ga, gb, out=big[:, 64:576])
    torch.cuda.synchronize()
    ref = oracle_mod.gemm(oa.dequantize(), ob.dequantize())
    ref = oracle_mod.bf16_to_f32(oracle_mod.bf16_rn(ref)).astype(np.float64)
    got = big.float().cpu().numpy().astype(np.float64)
    assert rel(got[:, 64:576], ref) < TOL
    assert np.all(got[:, :64] == 7.0) and np.all(got[:, 576:] == 7.0)


# The block-scaled GEMM shape sweep at full size (M = N = K in {2048, 4096, 8192, 16384}, the
# 16384 x 3072 x 8192 skinny shape and the 3072 x 8192 x 16384 dW shape), rank 0 and rank 64,
# through the same launch configuration the benchmark times (the split-tail workspace given: the
# last shape splits its last wave); 48 sampled output rows, four of them in the last 256
# (where the split tiles of an M > N shape lie).
GEMM_SWEEP = [(2048, 2048, 2048), (4096, 4096, 4096), (8192, 8192, 8192), (16384, 16384, 16384),
              (16384, 3072, 8192), (3072, 8192, 16384)]


def sample_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    tail = np.array([M - 256, M - 150, M - 77, M - 1])
    rest = rng.choice(M - 256, n - tail.size, replace=False)
    return np.sort(np.concatenate([rest, tail]))


@pytest.mark.parametrize("r", [0, 64])
@pytest.mark.parametrize("M,N,K", GEMM_SWEEP)
def test_gemm_full_size_sampled_rows(F, oracle_mod, M, N, K, r):
    check_gemm(F, oracle_mod, M, N, K, r, torch.bfloat16, beta=1.0, seed=17, rows=sample_rows(M, 48, M + N + r),
               split=True)


# Split tail, whole output against the oracle: more 256 x 256 tiles than SM pairs with a partial
# last wave, and K of at least 48 stages of 256, so that the last wave's tiles are cut along K
# (M <= N: the tail is the last tile column; M > N: the last tile row; 12352 = 48.25 stages: a
# ragged last stage in the last piece).  The call launches the GEMM and the reduction (after the
# branch fold when r > 0).
@pytest.mark.parametrize("M,N,K,r,out_dtype", [
    (2304, 2304, 12288, 64, torch.bfloat16),
    (2560, 2048, 12288, 0, torch.float32),
    (2304, 2560, 12352, 48, torch.float32),
])
def test_gemm_split_tail_whole_output(F, oracle_mod, M, N, K, r, out_dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (M // 256) * (N // 256)
    assert tiles > sms // 2 and tiles % (sms // 2) != 0  # a partial last wave on this GPU
    n0 = F.fp4_launch_count()
    check_gemm(F, oracle_mod, M, N, K, r, out_dtype, beta=0.75 if r else 1.0, seed=M + K + r, split=True)
    # amax + quantize per operand; the branch fold (r > 0); the GEMM and the reduction
    assert F.fp4_launch_count() - n0 == 2 * 2 + (1 if r else 0) + 2


def test_gemm_split_tail_is_deterministic(F):
    # Outlier entries spread the block scales, so that FP32 accumulation rounds and the
    # summation order shows (with N(0, 1) operands every partial sum is exact in FP32 and the
    # split result equals the whole-tile one bit for bit).
    M, N, K = 2304, 2304, 12288
    ga = F.fp4_quantize(dev(S.with_outlier_entries((M, K), 0.01, 1000.0, 31)))
    gb = F.fp4_quantize(dev(S.with_outlier_entries((N, K), 0.01, 1000.0, 32)))
    ws = torch.empty(F.gemm_split_workspace(), dtype=torch.uint8, device=DEV)
    torch.cuda.synchronize()
    n0 = F.fp4_launch_count()
    c1 = F.fp4_gemm_blockscaled_ws(ga, gb, out_dtype=torch.float32, workspace=ws)
    assert F.fp4_launch_count() - n0 == 2  # the GEMM and the reduction of the split tail
    c2 = F.fp4_gemm_blockscaled_ws(ga, gb, out_dtype=torch.float32, workspace=ws)
    c0 = F.fp4_gemm_blockscaled(ga, gb, out_dtype=torch.float32)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert torch.equal(c1, c2)
    # the split changes only the FP32 summation order inside the tail tiles
    diff = (c1 != c0).reshape(M // 256, 256, N // 256, 256).any(dim=3).any(dim=1)
    tiles = (M // 256) * (N // 256)
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    assert int(diff.sum()) <= tiles % pairs
    assert float((c1 - c0).abs().max()) <= 1e-4 * float(c0.abs().max())


# 16384, 8320, 7168 and 19456 rows take h = ceil(M / 152) = 108, 55, 48 and 128 rows per CTA on
# 152 SMs (last CTA 76, 15, 16 and 128 rows); 7168 x 704 also ends K on a half stage; 19584 rows
# (153 blocks of 128) take one CTA per 128-row block
@pytest.mark.parametrize("M,K,r", [(128, 64, 16), (256, 512, 32), (384, 320, 48), (1024, 2048, 64),
                                   (16384, 3072, 64), (8320, 1024, 32), (7168, 704, 16), (19456, 512, 48),
                                   (19584, 256, 16)])
def test_branch_factor(F, oracle_mod, M, K, r):
    X = S.student_t((M, K), 3.0, M + K)
    L = S.normal((r, K), 0.05, r)
    amax = torch.full((1,), -1.0, dtype=torch.float32, device=DEV)  # the call must zero it first
    P = F.fp4_branch_factor(dev(X), dev(L), amax=amax)
    torch.cuda.synchronize()
    F.fp4_check_status()
    assert np.float32(amax.item()) == np.float32(oracle_mod.amax(X))
    P0 = F.fp4_branch_factor(dev(X), dev(L))  # without the amax output: the same factor
    torch.cuda.synchronize()
    assert torch.equal(P0.view(torch.int16), P.view(torch.int16))
    want = oracle_mod.branch_factor(X, L)
    got_bits = S.torch_to_bits(P)
    g = oracle_mod.bf16_to_f32(got_bits).astype(np.float64)
    w = oracle_mod.bf16_to_f32(want).astype(np.float64)
    assert rel(g, w) < TOL
    # FP32 accumulation may flip a BF16 rounding now and then: at most one BF16 step
    # (2^-7 relative) away, except for results that cancel to near zero
    assert np.mean(got_bits == want) > 0.98
    scale = np.abs(oracle_mod.bf16_to_f32(X).astype(np.float64)) @ np.abs(oracle_mod.bf16_to_f32(L).astype(np.float64)).T
    assert np.all(np.abs(g - w) <= 2.0 ** -7 * np.abs(w) + 2.0 ** -20 * scale)
