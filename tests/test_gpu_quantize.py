"""GPU parity of the quantize kernels against the oracle: codes, block scales
(in the MMA layout, padding included) and the tensor scale must match bit for
bit, for RTN and SR (same seed and counter), row-wise, transposed and dual."""
import numpy as np
import pytest
import torch

from nvfp4_quantized_pretraining_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_pretraining_gb300 as F
    return F


DEV = "cuda"


def dev(u16):
    return S.bits_to_torch(u16, DEV)


def assert_same_quant(F, got, want, oracle_mod):
    torch.cuda.synchronize()
    F.fp4_check_status()
    codes = got.codes.cpu().numpy()
    assert codes.shape == want.codes.shape
    mism = np.argwhere(codes != want.codes)
    assert mism.size == 0, f"{len(mism)} code bytes differ, first at {mism[:5].tolist()}"
    sc = got.scales.cpu().numpy()
    ws = oracle_mod.scales_to_mma(want.scales)
    assert sc.shape == ws.shape
    bad = np.flatnonzero(sc != ws)
    assert bad.size == 0, f"{bad.size} scale bytes differ, first at {bad[:5].tolist()}"
    st = got.scale.cpu().numpy()
    assert np.float32(st[0]) == np.float32(want.S_t) and np.float32(st[1]) == np.float32(want.amax)


def test_conversion_conventions(F, oracle_mod):
    # E2M1 RTN: midpoints, signed zeros, saturation; E4M3: ties, subnormals, saturation.
    vals = [0.0, -0.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 6.5, 7.0, 1e30, float("inf"),
            -0.1, -0.25, -1e-30, 0.2499, 0.2501, -5.0, -6.5, float("-inf")]
    rng = np.random.default_rng(0)
    y = np.concatenate([np.array(vals, np.float32), rng.uniform(-7, 7, 4096).astype(np.float32)])
    y = np.concatenate([y, np.zeros((-len(y)) % 8, np.float32)])
    e2m1, _ = F.fp4_debug_convert(torch.from_numpy(y).to(DEV))
    assert np.array_equal(e2m1.cpu().numpy(), oracle_mod.e2m1_rtn(y))
    s = np.concatenate([np.array([0.0, 2.0 ** -10, 3 * 2.0 ** -11, 432.0, 440.0, 448.0, 449.0, 500.0, 1e30],
                                 np.float32),
                        np.exp(rng.uniform(-16, 6.2, 4087)).astype(np.float32)])
    s = np.concatenate([s, np.zeros((-len(s)) % 8, np.float32)])
    _, e4m3 = F.fp4_debug_convert(torch.from_numpy(s).to(DEV))
    assert np.array_equal(e4m3.cpu().numpy(), oracle_mod.e4m3_encode(s))


def sr_cases(rng):
    """Inputs and 16-bit draws that hit every branch of the SR rule: all three
    gap sizes, saturation, signed zeros, denormals, and exact ties
    rnd16 == frac * 2^16 (which must round down)."""
    y = [rng.uniform(-7, 7, 200000), rng.uniform(-2, 2, 100000), rng.uniform(-1, 1, 50000) * 1e-3,
         rng.standard_normal(20000) * 1e-39,
         np.array([0.0, -0.0, 0.5, 1.0, 1.5, 2, 3, 4, 6, 7, -6.5, 0.25, 0.75, 5.999999, 1e-40, 0.4999999,
                   0.9999999, 1.9999999, 3.9999999, 5.0, 4.0000005, 1e30, -1e30])]
    y = np.concatenate(y).astype(np.float32)
    rnd = rng.integers(0, 65536, y.size).astype(np.uint32)
    rnd[:46] = np.array([0, 65535] * 23, np.uint32)
    k = rng.integers(0, 6 * 131072, 100000)           # magnitudes on a 2^-17 grid
    yt = (k / 131072.0).astype(np.float32) * rng.choice(np.array([-1, 1], np.float32), k.size)
    a = np.abs(yt).astype(np.float64)
    sp = np.where(a >= 4, 2.0, np.where(a >= 2, 1.0, 0.5))
    tie = (np.round((a - np.floor(a / sp) * sp) / sp * 65536).astype(np.int64) & 0xFFFF).astype(np.uint32)
    return np.concatenate([y, yt]), np.concatenate([rnd, tie])


def test_sr_rounding_rule(F, oracle_mod):
    y, rnd = sr_cases(np.random.default_rng(11))
    got = F.fp4_debug_sr_round(torch.from_numpy(y).to(DEV), torch.from_numpy(rnd.astype(np.int32)).to(DEV))
    want = oracle_mod.e2m1_sr(y, rnd)
    g = got.cpu().numpy()
    bad = np.flatnonzero(g != want)
    assert bad.size == 0, f"{bad.size} of {y.size} differ, e.g. y={y[bad[:4]]} rnd={rnd[bad[:4]]}"


SHAPES = [  # rows % 16 == 0 (the transposed form needs whole 16-row blocks); ragged vs 128-row tiles
    (16, 16), (128, 64), (256, 512), (208, 48), (96, 1040), (1008, 4096), (512, 512),
]
ROW_ONLY_SHAPES = [(200, 48), (1, 16), (1000, 4096), (129, 1040)]  # any row count for the row form


def make_input(shape, kind, seed):
    if kind == "normal":
        return S.normal(shape, 1.0, seed)
    if kind == "outliers":
        return S.with_outlier_entries(shape, 0.001, 50.0, seed)
    if kind == "student":
        return S.student_t(shape, 3.0, seed)
    if kind == "grad":
        return S.normal(shape, 1e-3, seed)
    if kind == "tiny":  # amax near 4e-36: denormal S_t, the 1/d cap, scale underflow
        return S.to_bf16_bits((np.random.default_rng(seed).standard_normal(shape) * 1e-36).astype(np.float32))
    raise ValueError(kind)


@pytest.mark.parametrize("shape", SHAPES + ROW_ONLY_SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_rows(F, oracle_mod, shape, mode):
    x = make_input(shape, "outliers", seed=shape[0] * 7 + shape[1])
    got = F.fp4_quantize(dev(x), round_mode=mode, seed=123456789012345, sr_stream=0)
    want = oracle_mod.quantize(x, mode, seed=123456789012345, stream=0)
    assert_same_quant(F, got, want, oracle_mod)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_transposed(F, oracle_mod, shape, mode):
    x = make_input(shape, "student", seed=shape[0] * 3 + shape[1])
    got = F.fp4_quantize_transposed(dev(x), round_mode=mode, seed=42, sr_stream=1)
    want = oracle_mod.quantize(x, mode, seed=42, stream=1, transposed=True)
    assert_same_quant(F, got, want, oracle_mod)


@pytest.mark.parametrize("shape", [(64, 128), (256, 512), (208, 48), (1024, 2048)])
@pytest.mark.parametrize("mode", [0, 1])
def test_quantize_dual(F, oracle_mod, shape, mode):
    x = make_input(shape, "grad", seed=5)
    r, c = F.fp4_quantize_dual(dev(x), round_mode=mode, seed=1, sr_stream_row=0, sr_stream_col=1)
    assert_same_quant(F, r, oracle_mod.quantize(x, mode, seed=1, stream=0), oracle_mod)
    assert_same_quant(F, c, oracle_mod.quantize(x, mode, seed=1, stream=1, transposed=True), oracle_mod)


@pytest.mark.parametrize("shape", [(208, 48), (1024, 2048)])
def test_sr_counter_forms_agree(F, oracle_mod, shape):
    # the SR kernels' 32-bit counter form (every tensor below 2^35 elements) and the general
    # form that computes counter word 1: both bit-exact against the oracle, so equal
    x = make_input(shape, "grad", seed=11)
    want_r = oracle_mod.quantize(x, 1, seed=7, stream=0)
    want_c = oracle_mod.quantize(x, 1, seed=7, stream=1, transposed=True)
    outs = []
    for force64 in (0, 1):
        F.lib().fp4_debug_force_counter64(force64)
        try:
            r, c = F.fp4_quantize_dual(dev(x), round_mode=1, seed=7, sr_stream_row=0, sr_stream_col=1)
            torch.cuda.synchronize()
        finally:
            F.lib().fp4_debug_force_counter64(0)
        assert_same_quant(F, r, want_r, oracle_mod)
        assert_same_quant(F, c, want_c, oracle_mod)
        outs.append((r, c))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)


@pytest.mark.parametrize("kind", ["tiny", "normal"])
def test_quantize_edge_values(F, oracle_mod, kind):
    x = make_input((128, 256), kind, seed=9)
    for mode in (0, 1):
        assert_same_quant(F, F.fp4_quantize(dev(x), round_mode=mode, seed=3), oracle_mod.quantize(x, mode, seed=3),
                          oracle_mod)
        assert_same_quant(F, F.fp4_quantize_transposed(dev(x), round_mode=mode, seed=3, sr_stream=1),
                          oracle_mod.quantize(x, mode, seed=3, stream=1, transposed=True), oracle_mod)


def test_all_zero_and_single_nonzero(F, oracle_mod):
    x = np.zeros((128, 64), np.uint16)
    x[5, 7] = 0x8000
    assert_same_quant(F, F.fp4_quantize(dev(x)), oracle_mod.quantize(x), oracle_mod)
    x[17, 33] = S.to_bf16_bits(np.array([-3.0], np.float32))[0]
    assert_same_quant(F, F.fp4_quantize(dev(x)), oracle_mod.quantize(x), oracle_mod)
    assert_same_quant(F, F.fp4_quantize_transposed(dev(x)), oracle_mod.quantize(x, transposed=True), oracle_mod)


def test_worked_blocks_on_gpu(F, oracle_mod):
    import json, os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_blocks.json")))
    x = S.to_bf16_bits(np.array([float(v) for v in g["x"]], np.float32)).reshape(1, -1)
    q = F.fp4_quantize(dev(x))
    torch.cuda.synchronize()
    codes = q.codes.cpu().numpy()[0]
    got = [(codes[i // 2] >> (4 * (i % 2))) & 0xF for i in range(x.shape[1])]
    assert got == g["codes"]
    sc = q.scales.cpu().numpy()
    assert [int(sc[oracle_mod.mma_scale_offset(0, k, 5)]) for k in range(5)] == g["scales"]
    assert float(q.scale[0]) == g["S_t"]


def test_amax_and_supplied_amax(F, oracle_mod):
    x = make_input((512, 1024), "outliers", seed=11)
    a = F.fp4_amax(dev(x))
    torch.cuda.synchronize()
    assert float(a[0]) == oracle_mod.amax(x)
    # a supplied amax (here 2x the true one) is used as given
    amax2 = torch.tensor([2.0 * oracle_mod.amax(x)], dtype=torch.float32, device=DEV)
    got = F.fp4_quantize(dev(x), amax=amax2)
    want = oracle_mod.quantize(x, amax_value=float(amax2[0]))
    assert_same_quant(F, got, want, oracle_mod)


def test_strided_input(F, oracle_mod):
    full = make_input((256, 1024), "normal", seed=12)
    xt = dev(full)[:, 128:640]  # row pitch 1024, 512 columns
    want = oracle_mod.quantize(np.ascontiguousarray(full[:, 128:640]), 1, seed=8)
    assert_same_quant(F, F.fp4_quantize(xt, round_mode=1, seed=8), want, oracle_mod)
    r, c = F.fp4_quantize_dual(xt, round_mode=1, seed=8)
    assert_same_quant(F, r, want, oracle_mod)
    assert_same_quant(F, c, oracle_mod.quantize(np.ascontiguousarray(full[:, 128:640]), 1, seed=8, stream=1,
                                                transposed=True), oracle_mod)


@pytest.mark.parametrize("name,shape,kind,mode", [
    ("mlp_up_X", (8192, 2048), "normal", 0),
    ("mlp_up_W", (5632, 2048), "normal", 0),
    ("mlp_up_dY_sr", (8192, 5632), "grad", 1),
    ("sweep_16M", (4096, 4096), "outliers", 0),
    ("sweep_16M_sr", (4096, 4096), "outliers", 1),
    ("sweep_64M", (16384, 4096), "outliers", 0),
    ("sweep_64M_sr", (16384, 4096), "outliers", 1),
    ("sweep_256M", (65536, 4096), "outliers", 0),
    ("sweep_256M_sr", (65536, 4096), "outliers", 1),
    ("block3b_gate_up_dY_sr", (16384, 16384), "grad", 1),
])
def test_quantize_full_size(F, oracle_mod, name, shape, kind, mode):
    # every code and scale of the full tensor, in the dual form and the single-orientation forms
    x = make_input(shape, kind, seed=21)
    xd = dev(x)
    r, c = F.fp4_quantize_dual(xd, round_mode=mode, seed=1)
    assert_same_quant(F, r, oracle_mod.quantize(x, mode, seed=1, stream=0), oracle_mod)
    assert_same_quant(F, c, oracle_mod.quantize(x, mode, seed=1, stream=1, transposed=True), oracle_mod)
    r2 = F.fp4_quantize(xd, round_mode=mode, seed=1)
    c2 = F.fp4_quantize_transposed(xd, round_mode=mode, seed=1)
    torch.cuda.synchronize()
    assert torch.equal(r2.codes, r.codes) and torch.equal(r2.scales, r.scales) and torch.equal(r2.scale, r.scale)
    assert torch.equal(c2.codes, c.codes) and torch.equal(c2.scales, c.scales) and torch.equal(c2.scale, c.scale)


def test_transposed_rejects_partial_row_blocks(F):
    x = make_input((200, 48), "normal", seed=1)
    with pytest.raises(F.FP4Error) as e:
        F.fp4_quantize_transposed(dev(x))
    assert e.value.status == F.FP4_ERR_UNSUPPORTED_SHAPE


@pytest.mark.gpu
def test_quantize_waits_for_a_copy_queued_after_the_previous_call(F, oracle_mod):
    # A quantization queued right behind another call and a device copy into its input: the copy
    # (not a kernel) must land before the quantizer reads the tensor.
    big = S.bits_to_torch(S.normal((8192, 4096), 1.0, 90), DEV)
    src = S.bits_to_torch(S.normal((256, 4096), 1.0, 91), DEV)
    want = F.fp4_quantize(src)
    torch.cuda.synchronize()
    want_codes, want_scales = want.codes.clone(), want.scales.clone()
    for i in range(4):
        x = torch.full_like(src, float(i + 3))
        torch.cuda.synchronize()
        F.fp4_quantize_dual(big)
        x.copy_(src)
        got = F.fp4_quantize(x)
        torch.cuda.synchronize()
        assert torch.equal(got.codes, want_codes) and torch.equal(got.scales, want_scales)
