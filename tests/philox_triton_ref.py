"""Philox4x32-10 computed by Triton's own implementation (``tl.random.philox``),
run on the CPU by Triton's interpreter: an implementation of the generator
written independently of this repository, used to pin the oracle's.

Test infrastructure, run as a child process with TRITON_INTERPRET=1 set (the
interpreter must be chosen before Triton is imported):

    TRITON_INTERPRET=1 python philox_triton_ref.py IN.npz OUT.npz

IN.npz holds ``seeds`` (uint64, one per row) and ``ctr`` (uint32, rows x 4);
OUT.npz receives ``out`` (uint32, rows x 4).  Triton's key is (seed lo 32 bits,
seed hi 32 bits) and its counter the four 32-bit words as given.
"""
import sys

import numpy as np
import torch
import triton
import triton.language as tl


@triton.jit
def _philox_kernel(seed, c_ptr, out_ptr, n, BLOCK: tl.constexpr):
    i = tl.program_id(0) * BLOCK + tl.arange(0, BLOCK)
    m = i < n
    c0 = tl.load(c_ptr + 4 * i, mask=m)
    c1 = tl.load(c_ptr + 4 * i + 1, mask=m)
    c2 = tl.load(c_ptr + 4 * i + 2, mask=m)
    c3 = tl.load(c_ptr + 4 * i + 3, mask=m)
    o0, o1, o2, o3 = tl.random.philox(seed, c0, c1, c2, c3, 10)
    tl.store(out_ptr + 4 * i, o0, mask=m)
    tl.store(out_ptr + 4 * i + 1, o1, mask=m)
    tl.store(out_ptr + 4 * i + 2, o2, mask=m)
    tl.store(out_ptr + 4 * i + 3, o3, mask=m)


def main(src: str, dst: str) -> None:
    d = np.load(src)
    seeds, ctr = d["seeds"].astype(np.uint64), d["ctr"].astype(np.uint32)
    out = np.zeros_like(ctr)
    block = 1024
    for seed in np.unique(seeds):
        rows = np.nonzero(seeds == seed)[0]
        c = torch.from_numpy(np.ascontiguousarray(ctr[rows]).view(np.int32).reshape(-1))
        o = torch.zeros_like(c)
        n = len(rows)
        _philox_kernel[(triton.cdiv(n, block),)](int(seed.view(np.int64)), c, o, n, BLOCK=block)
        out[rows] = o.numpy().view(np.uint32).reshape(n, 4)
    np.savez(dst, out=out)


if __name__ == "__main__":
    main(sys.argv[1], sys.argv[2])
