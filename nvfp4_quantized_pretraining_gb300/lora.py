"""Host-side set-up of the LoRA-SVD weight split (Full-Stack FP4, section 2.1:
W = W_res + beta L2 L1; the subspace is (re)aligned with a randomized SVD).

This runs once per weight (and at each realignment), not in the per-step hot
path: a randomized range finder (Halko, Martinsson, Tropp 2011) with a few
power iterations, in NumPy FP32/FP64 on the host.  Returns BF16 bit patterns
ready to upload: L2 = bf16(U_r Sigma_r) (N x r), L1 = bf16(V_r^T) (r x K),
W_res = bf16(W - L2 L1).
"""
from __future__ import annotations

import numpy as np

from . import synthetic as S


def lora_svd_split_randomized(W_bf16: np.ndarray, r: int, oversample: int = 16, power_iters: int = 2,
                              seed: int = 0):
    W = (W_bf16.astype(np.uint32) << 16).view(np.float32)
    N, K = W.shape
    if r == 0:
        return W_bf16.copy(), np.zeros((0, K), np.uint16), np.zeros((N, 0), np.uint16)
    rng = np.random.default_rng(seed)
    k = min(r + oversample, min(N, K))
    Y = W @ rng.standard_normal((K, k), dtype=np.float32)
    for _ in range(power_iters):
        Q, _ = np.linalg.qr(Y)
        Z, _ = np.linalg.qr(W.T @ Q)
        Y = W @ Z
    Q, _ = np.linalg.qr(Y.astype(np.float64))
    B = Q.T @ W.astype(np.float64)                 # k x K
    Ub, s, Vt = np.linalg.svd(B, full_matrices=False)
    U = Q @ Ub[:, :r]
    L2 = S.to_bf16_bits((U * s[:r]).astype(np.float32))
    L1 = S.to_bf16_bits(Vt[:r].astype(np.float32))
    low = ((L2.astype(np.uint32) << 16).view(np.float32) @ (L1.astype(np.uint32) << 16).view(np.float32))
    W_res = S.to_bf16_bits(W - low)
    return W_res, L1, L2
