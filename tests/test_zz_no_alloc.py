"""The workspace-free forward (fp4_linear_fwd_noalloc) against fp4_linear_fwd:
same launches on the library's static scratch instead of a caller workspace,
so Y and the saved column form of X must match bit for bit, call after call.
Named to be collected last, after every other test has used the library."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_quantized_pretraining_gb300 import synthetic as S

DEV = "cuda"
SCRATCH_BYTES = 32 << 20


@pytest.fixture(scope="module")
def F():
    import __graft_entry__
    __graft_entry__.build()
    import nvfp4_quantized_pretraining_gb300 as F
    return F


def test_noalloc_rejects_oversized_shape(F):
    # host-side check only: no pointer is dereferenced and nothing is launched
    M, K, N, r = 16384, 8192, 128, 64
    assert F.linear_fwd_workspace(M, N, K, r) > SCRATCH_BYTES
    fake = 1 << 20  # 256-byte aligned, never touched
    wq = F.CTensor(codes=fake, scales=fake, scale=fake, rows=N, cols=K)
    xq = F.CTensor(codes=fake, scales=fake, scale=fake, rows=K, cols=M)
    st = F.lib().fp4_linear_fwd_noalloc(fake, M, K, K, ctypes.byref(wq), fake, fake, r, 1.0, fake, N,
                                        ctypes.byref(xq), None)
    assert st == F.FP4_ERR_WORKSPACE
    msg = F.lib().fp4_last_error().decode()
    assert "static scratch" in msg and str(SCRATCH_BYTES) in msg


def layer(F, M, K, N, r, seed):
    X = S.bits_to_torch(S.normal((M, K), 1.0, seed), DEV)
    W = S.bits_to_torch(S.normal((N, K), 0.02, seed + 1), DEV)
    Wq = F.fp4_quantize(W)
    L1 = S.bits_to_torch(S.normal((r, K), 0.02, seed + 2), DEV) if r else None
    L2 = S.bits_to_torch(S.normal((N, r), 0.02, seed + 3), DEV) if r else None
    return X, Wq, L1, L2


def same_tensor(a, b):
    return (torch.equal(a.codes, b.codes) and torch.equal(a.scales, b.scales)
            and torch.equal(a.scale, b.scale))


@pytest.mark.gpu
def test_noalloc_matches_workspace_forward_twice_in_a_row(F):
    cases = [(256, 512, 384, 16, 1), (512, 1024, 256, 64, 2), (384, 256, 128, 0, 3),
             (16384, 3072, 256, 64, 4)]  # the last one is 30.4 MB of scratch, close to the limit
    for (M, K, N, r, seed) in cases:
        assert F.linear_fwd_workspace(M, N, K, r) <= SCRATCH_BYTES
    layers = [layer(F, M, K, N, r, 10 * seed) for (M, K, N, r, seed) in cases]
    outs = []
    for (M, K, N, r, _), (X, Wq, L1, L2) in zip(cases, layers):
        outs.append((torch.empty((M, N), dtype=torch.bfloat16, device=DEV), F.NVFP4Tensor.empty(K, M, DEV)))
    F.fp4_linear_fwd_noalloc(*layers[0], 0.75, *outs[0])  # first call per device: address look-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    # consecutive calls on one stream reuse the scratch; each must still be exact
    for (X, Wq, L1, L2), (Y, xqT) in zip(layers, outs):
        F.fp4_linear_fwd_noalloc(X, Wq, L1, L2, 0.75, Y, xqT)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    F.fp4_check_status()
    for (X, Wq, L1, L2), (Y, xqT) in zip(layers, outs):
        Y_ref, xqT_ref = F.fp4_linear_fwd(X, Wq, L1, L2, beta=0.75)
        torch.cuda.synchronize()
        assert torch.equal(Y.view(torch.int16), Y_ref.view(torch.int16))
        assert same_tensor(xqT, xqT_ref)
    F.fp4_check_status()
