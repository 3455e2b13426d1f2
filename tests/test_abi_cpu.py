"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, reports sizes consistent with the oracle's layout, and
rejects bad arguments on the host before anything is launched.  Every bad
argument here fails validation (NULL / misaligned / bad shape), so no call
reaches the device even on a machine that has one."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def F():
    from nvfp4_quantized_pretraining_gb300 import build
    build.build()
    import nvfp4_quantized_pretraining_gb300 as F
    F.lib()
    return F


def header_functions():
    text = open(os.path.join(ROOT, "include", "nvfp4_gb300.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = header_functions()
    for n in ["fp4_quantize", "fp4_quantize_transposed", "fp4_gemm_blockscaled", "fp4_linear_fwd", "fp4_linear_bwd"]:
        assert n in names


def test_library_exports_every_declared_symbol(F):
    L = F.lib()
    for name in header_functions():
        assert hasattr(L, name), name
    assert sorted(F.EXPORTS) == header_functions()


def test_scale_bytes_match_oracle_layout(F, oracle_mod):
    for rows, cols in [(128, 64), (200, 48), (1, 16), (4096, 4096), (5632, 2048), (129, 1040)]:
        assert F.scale_bytes(rows, cols) == oracle_mod.mma_scale_bytes(rows, cols // 16)


def test_workspace_sizes(F):
    M, N, K, r = 16384, 3072, 8192, 64
    fw = F.linear_fwd_workspace(M, N, K, r)
    assert fw >= M * K // 2 + F.scale_bytes(M, K) + M * r * 2
    bw = F.linear_bwd_workspace(M, N, K, r)
    assert bw >= 2 * (M * N // 2 + F.scale_bytes(M, N)) + (M + N + K) * r * 2
    assert F.linear_fwd_workspace(M, N, K, 0) < fw


def _t(codes=0x1000, scales=0x2000, scale=0x3000, rows=128, cols=128):
    import nvfp4_quantized_pretraining_gb300 as F
    return F.CTensor(codes, scales, scale, rows, cols)


def test_invalid_arguments_rejected_on_host(F):
    L = F.lib()
    s = None
    t = _t()
    # NULL input
    assert L.fp4_quantize(None, 128, 128, 128, 0, 0, 0, None, ctypes.byref(t), s) == F.FP4_ERR_INVALID_ARG
    # misaligned input
    assert L.fp4_quantize(0x1008, 128, 128, 128, 0, 0, 0, None, ctypes.byref(t), s) == F.FP4_ERR_MISALIGNED
    # pitch not 16-byte aligned
    assert L.fp4_quantize(0x1000, 128, 128, 130, 0, 0, 0, None, ctypes.byref(t), s) == F.FP4_ERR_MISALIGNED
    # cols not a multiple of 16
    t2 = _t(cols=120)
    assert L.fp4_quantize(0x1000, 128, 120, 128, 0, 0, 0, None, ctypes.byref(t2), s) == F.FP4_ERR_UNSUPPORTED_SHAPE
    # bad rounding mode
    assert L.fp4_quantize(0x1000, 128, 128, 128, 7, 0, 0, None, ctypes.byref(t), s) == F.FP4_ERR_INVALID_ARG
    # output shape mismatch
    t3 = _t(rows=64)
    assert L.fp4_quantize(0x1000, 128, 128, 128, 0, 0, 0, None, ctypes.byref(t3), s) == F.FP4_ERR_INVALID_ARG
    # transposed needs rows % 16
    t4 = _t(rows=128, cols=40)
    assert L.fp4_quantize_transposed(0x1000, 40, 128, 128, 0, 0, 0, None, ctypes.byref(t4), s) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE
    # misaligned output buffer
    t5 = _t(codes=0x1004)
    assert L.fp4_quantize(0x1000, 128, 128, 128, 0, 0, 0, None, ctypes.byref(t5), s) == F.FP4_ERR_MISALIGNED
    assert "16-byte" in F.fp4_last_error()


def test_gemm_argument_checks(F):
    L = F.lib()
    A, B = _t(rows=128, cols=128), _t(rows=128, cols=128)
    ok_c = 0x4000
    assert L.fp4_gemm_blockscaled(None, ctypes.byref(B), None, None, 0, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_INVALID_ARG
    Bk = _t(rows=128, cols=192)
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(Bk), None, None, 0, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_INVALID_ARG
    Am = _t(rows=100, cols=128)
    assert L.fp4_gemm_blockscaled(ctypes.byref(Am), ctypes.byref(B), None, None, 0, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE
    Ak = _t(rows=128, cols=96)
    Bk2 = _t(rows=128, cols=96)
    assert L.fp4_gemm_blockscaled(ctypes.byref(Ak), ctypes.byref(Bk2), None, None, 0, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(B), 0x5000, 0x6000, 80, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_UNSUPPORTED_SHAPE
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(B), None, None, 16, 1.0, ok_c, 0, 128, None) == \
        F.FP4_ERR_INVALID_ARG
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(B), None, None, 0, 1.0, ok_c, 0, 100, None) == \
        F.FP4_ERR_INVALID_ARG
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(B), None, None, 0, 1.0, ok_c + 8, 0, 128, None) == \
        F.FP4_ERR_MISALIGNED
    assert L.fp4_gemm_blockscaled(ctypes.byref(A), ctypes.byref(B), None, None, 0, 1.0, ok_c, 5, 128, None) == \
        F.FP4_ERR_INVALID_ARG


def test_linear_argument_checks(F):
    L = F.lib()
    W = _t(rows=256, cols=128)
    xT = _t(rows=128, cols=256)
    # workspace too small
    assert L.fp4_linear_fwd(0x1000, 256, 128, 128, ctypes.byref(W), None, None, 0, 1.0, 0x2000, 256,
                            ctypes.byref(xT), 0x8000, 16, None) == F.FP4_ERR_WORKSPACE
    # K mismatch
    W2 = _t(rows=256, cols=64)
    assert L.fp4_linear_fwd(0x1000, 256, 128, 128, ctypes.byref(W2), None, None, 0, 1.0, 0x2000, 256,
                            ctypes.byref(xT), 0x8000, 1 << 30, None) == F.FP4_ERR_INVALID_ARG
    # rank without factors
    assert L.fp4_linear_fwd(0x1000, 256, 128, 128, ctypes.byref(W), None, None, 16, 1.0, 0x2000, 256,
                            ctypes.byref(xT), 0x8000, 1 << 30, None) == F.FP4_ERR_INVALID_ARG
    WT = _t(rows=128, cols=256)
    assert L.fp4_linear_bwd(0x1000, 256, 256, 256, ctypes.byref(WT), ctypes.byref(xT), None, None, 0, 1.0, 0,
                            0x2000, 128, 0x3000, 0, 128, 0x8000, 16, None) == F.FP4_ERR_WORKSPACE
    xT2 = _t(rows=128, cols=128)
    assert L.fp4_linear_bwd(0x1000, 256, 256, 256, ctypes.byref(WT), ctypes.byref(xT2), None, None, 0, 1.0, 0,
                            0x2000, 128, 0x3000, 0, 128, 0x8000, 1 << 30, None) == F.FP4_ERR_INVALID_ARG


def test_header_is_plain_c_and_a_c_host_links_the_library(F, tmp_path):
    # The boundary is a C ABI: the header must compile as C99 (no C++), and a C program that
    # takes the address of every declared call must link against the shared library.
    names = header_functions()
    src = tmp_path / "abi_host.c"
    src.write_text('#include "nvfp4_gb300.h"\n#include <stdio.h>\n'
                   "typedef void (*any_fn)(void);\n"
                   "int main(void) {\n  any_fn fns[] = {\n" +
                   "".join(f"    (any_fn)&{n},\n" for n in names) +
                   "  };\n  printf(\"%d\\n\", (int)(sizeof(fns) / sizeof(fns[0])));\n"
                   "  return fp4_scale_bytes(128, 64) == 512 ? 0 : 1;  /* 128 rows x 4 scale bytes */\n}\n")
    lib_dir = os.path.dirname(F.LIB_PATH)
    exe = tmp_path / "abi_host"
    import subprocess
    cc = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                         str(src), "-L", lib_dir, "-lnvfp4_gb300", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                        capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == str(len(names)), run.stdout + run.stderr
