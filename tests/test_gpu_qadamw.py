"""Q-AdamW second-moment codec through the C ABI against the oracle: the encoder's
codes, block scales (MMA layout, padding included), tensor scale and BF16 tile
means bit for bit, and the decoder's FP32 output bit for bit.  Every step is one
FP32 operation in a fixed order on both sides (square root, pairwise-tree mean,
the Walsh-Hadamard butterfly), so the two sides take every rounding and every
quantization decision on the same value."""
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


def test_qadamw_codec_rejects_bad_arguments(F):
    # host-side checks only; nothing is launched
    L = F.lib()
    fake = 1 << 20
    t = F.CTensor(fake, fake, fake, 64, 256)
    import ctypes
    assert L.fp4_qadamw_v_encode(fake, 64, 250, 256, ctypes.byref(t), fake, None) == F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_qadamw_v_encode(fake, 64, 256, 258, ctypes.byref(t), fake, None) == F.FP4_ERR_MISALIGNED
    assert L.fp4_qadamw_v_encode(fake, 32, 256, 256, ctypes.byref(t), fake, None) == F.FP4_ERR_INVALID_ARG
    assert L.fp4_qadamw_v_encode(fake, 64, 256, 256, ctypes.byref(t), None, None) == F.FP4_ERR_INVALID_ARG
    assert L.fp4_qadamw_v_decode(ctypes.byref(t), fake, fake, 128, None) == F.FP4_ERR_INVALID_ARG


def padded_f32(v, pad):
    R, C = v.shape
    full = torch.zeros((R, C + pad), dtype=torch.float32, device=DEV)
    full[:, :C] = torch.from_numpy(v).to(DEV)
    return full[:, :C]


def check_encode(F, oracle_mod, q, mean, v):
    torch.cuda.synchronize()
    F.fp4_check_status()
    want, want_mean = oracle_mod.vt_encode(v)
    got_mean = S.torch_to_bits(mean)
    assert np.array_equal(got_mean, want_mean), int(np.sum(got_mean != want_mean))
    st = q.scale.cpu().numpy()
    assert np.float32(st[0]) == np.float32(want.S_t) and np.float32(st[1]) == np.float32(want.amax)
    codes = q.codes.cpu().numpy()
    assert np.array_equal(codes, want.codes), int(np.sum(codes != want.codes))
    assert np.array_equal(q.scales.cpu().numpy(), oracle_mod.scales_to_mma(want.scales))
    return want, want_mean


def worked_blocks():
    H = np.array([[1.0]])
    while H.shape[0] < 16:
        H = np.block([[H, H], [H, -H]])
    u = 1.0 + (21.0 / 128.0) * H[[1, 5, 15]]
    return (u * u).astype(np.float32)


@pytest.mark.gpu
@pytest.mark.parametrize("R,C,pad,kind", [
    (64, 256, 0, "adam"), (200, 1040, 12, "adam"),  # ragged rows and scale columns (padded atoms)
    (1, 16, 0, "adam"), (130, 64, 4, "wide"),        # one block; 1e-30 .. 1e10 magnitudes
    (32, 128, 0, "zero"), (3, 16, 0, "worked"), (16, 96, 0, "constant"),
])
def test_encode_and_decode_match_oracle(F, oracle_mod, R, C, pad, kind):
    if kind == "adam":
        v = S.adam_second_moment(R, C, R + C)
    elif kind == "wide":
        rng = np.random.default_rng(9)
        v = np.exp(rng.uniform(np.log(1e-30), np.log(1e10), (R, C))).astype(np.float32)
        v[0, :7] = 0.0
    elif kind == "zero":
        v = np.zeros((R, C), np.float32)
    elif kind == "worked":
        v = worked_blocks()
    else:
        v = np.repeat(np.array([[4.0], [2.25], [0.7]], np.float32), C, axis=1)
        v = np.tile(v, (R // 3 + 1, 1))[:R]
    q, mean = F.fp4_qadamw_v_encode(padded_f32(v, pad))
    want, want_mean = check_encode(F, oracle_mod, q, mean, v)
    # decode: the GPU's own encoding, and the oracle's encoding uploaded
    out = torch.full((R, C + 4), -1.0, dtype=torch.float32, device=DEV)[:, :C]
    F.fp4_qadamw_v_decode(q, mean, out=out)
    qo = F.NVFP4Tensor.empty(R, C, DEV)
    qo.codes.copy_(torch.from_numpy(want.codes))
    qo.scales.copy_(torch.from_numpy(oracle_mod.scales_to_mma(want.scales)))
    qo.scale.copy_(torch.tensor([want.S_t, want.amax], dtype=torch.float32))
    out2 = F.fp4_qadamw_v_decode(qo, S.bits_to_torch(want_mean, DEV))
    torch.cuda.synchronize()
    F.fp4_check_status()
    ref = oracle_mod.vt_decode(want, want_mean)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert np.array_equal(out2.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    if kind in ("worked", "constant", "zero"):
        assert np.array_equal(ref, v)  # exactly representable: the codec is lossless here


@pytest.mark.gpu
def test_codec_full_size_gate_up_state(F, oracle_mod):
    # the second moment of the 3B block's gate_up weight (16384 x 3072 FP32, 201 MB)
    R, C = 16384, 3072
    v = S.adam_second_moment(R, C, 31)
    vd = torch.from_numpy(v).to(DEV)
    q, mean = F.fp4_qadamw_v_encode(vd)
    want, want_mean = check_encode(F, oracle_mod, q, mean, v)
    out = F.fp4_qadamw_v_decode(q, mean)
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(R, 256, replace=False)
    got = out.cpu().numpy()
    qs = oracle_mod.QTensor(want.codes[rows], want.scales[rows], want.S_t, want.amax, len(rows), C)
    ref = oracle_mod.vt_decode(qs, want_mean[rows])
    assert np.array_equal(got[rows].view(np.uint32), ref.view(np.uint32))
