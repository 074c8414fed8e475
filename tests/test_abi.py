"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every entry point include/nvfp4rl.h declares, and
reject bad arguments with the documented status codes before any CUDA call.
"""

import ctypes
import os
import re

import pytest
import torch

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "nvfp4rl.h")


@pytest.fixture(scope="module")
def lib():
    from nvfp4_quantized_dit_gb300 import build as b
    b.build()
    import nvfp4_quantized_dit_gb300 as pkg
    return pkg.library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^(?:nvfp4_status|const char\*|int|size_t)\s+(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_five_calls():
    names = _declared_functions()
    for n in ["nvfp4_requant", "nvfp4_act_quant", "nvfp4_gemm", "bf16_gemm", "select_contrastive"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    import nvfp4_quantized_dit_gb300 as pkg
    for code, name in pkg.STATUS.items():
        assert pkg.nvfp4_status_string(code) == name
    assert pkg.nvfp4_version() >= 100


def test_sf_helpers_match_header_layout():
    import nvfp4_quantized_dit_gb300 as pkg
    K = 256
    assert pkg.sf_bytes(1, K) == 128 * 16 and pkg.sf_bytes(129, K) == 256 * 16
    seen = set()
    for row in range(256):
        for kb in range(K // 16):
            off = pkg.sf_offset(row, kb, K)
            assert off not in seen
            seen.add(off)
    assert seen == set(range(pkg.sf_bytes(256, K)))
    # tile (R, C) is 512 contiguous bytes; inside: (row%32)*16 + ((row/32)%4)*4 + kb%4
    assert pkg.sf_offset(0, 0, K) == 0 and pkg.sf_offset(1, 0, K) == 16
    assert pkg.sf_offset(32, 0, K) == 4 and pkg.sf_offset(0, 3, K) == 3
    assert pkg.sf_offset(0, 4, K) == 512 and pkg.sf_offset(128, 0, K) == (K // 64) * 512


A16 = 0x10000  # aligned fake addresses: never dereferenced, validation fails first
BAD = 0x10001


def test_act_quant_validation(lib):
    P = ctypes.c_void_p
    assert lib.nvfp4_act_quant(P(A16), 4, 100, P(A16), P(A16), P(A16), None) == 2  # K % 64
    assert lib.nvfp4_act_quant(P(A16), -1, 64, P(A16), P(A16), P(A16), None) == 2
    assert lib.nvfp4_act_quant(P(A16), 4, 64 * 1024, P(A16), P(A16), P(A16), None) == 2
    assert lib.nvfp4_act_quant(None, 4, 64, P(A16), P(A16), P(A16), None) == 1
    assert lib.nvfp4_act_quant(P(BAD), 4, 64, P(A16), P(A16), P(A16), None) == 3
    assert lib.nvfp4_act_quant(None, 0, 64, None, None, None, None) == 0  # empty: no-op


def test_act_quant_tensor_validation(lib):
    P = ctypes.c_void_p
    assert lib.nvfp4_act_quant_tensor(P(A16), 4, 100, P(A16), P(A16), P(A16), None) == 2  # K % 64
    assert lib.nvfp4_act_quant_tensor(P(A16), -1, 64, P(A16), P(A16), P(A16), None) == 2
    assert lib.nvfp4_act_quant_tensor(None, 4, 64, P(A16), P(A16), P(A16), None) == 1
    assert lib.nvfp4_act_quant_tensor(P(A16), 4, 64, P(A16), P(A16), None, None) == 1  # s_t
    assert lib.nvfp4_act_quant_tensor(P(BAD), 4, 64, P(A16), P(A16), P(A16), None) == 3
    assert lib.nvfp4_act_quant_tensor(None, 0, 64, None, None, None, None) == 1  # s_t always written
    assert lib.nvfp4_act_quant_tensor(None, 0, 64, None, None, P(BAD), None) == 3


def test_requant_validation(lib):
    P = ctypes.c_void_p
    f = ctypes.c_float(32.0)
    assert lib.nvfp4_requant(P(A16), 2, None, None, 0, f, 8, 64, P(A16), P(A16), P(A16), None, 0, None) == 2
    assert lib.nvfp4_requant(P(A16), 0, P(A16), P(A16), 65, f, 8, 64, P(A16), P(A16), P(A16), None, 0, None) == 2
    assert lib.nvfp4_requant(P(A16), 0, None, None, 0, f, 8, 96, P(A16), P(A16), P(A16), None, 0, None) == 2
    assert lib.nvfp4_requant(P(A16), 0, None, None, 0, f, 8, 64, P(A16), P(A16), None, None, 0, None) == 1
    assert lib.nvfp4_requant(None, 0, None, None, 0, f, 8, 64, P(A16), P(A16), P(A16), None, 0, None) == 1
    assert lib.nvfp4_requant(P(A16), 0, P(BAD), P(A16), 32, f, 8, 64, P(A16), P(A16), P(A16), None, 0, None) == 3
    assert lib.nvfp4_requant(P(A16), 0, None, None, 0, f, 8, 64, P(BAD), P(A16), P(A16), None, 0, None) == 3


def test_requant_workspace_bytes(lib):
    """The tensor-core merge's workspace: A' (256 bytes per column of A), the row
    norms (rows padded to 256), 16 bytes of column norms per 128 columns and a
    counter, each piece rounded up to 256 bytes; 0 where that path does not apply."""
    ws = lib.nvfp4_requant_workspace_bytes
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    up = lambda x: (x + 255) // 256 * 256
    assert ws(0, 32, 300, 192) == up(192 * 256) + up(512 * 4) + up(2 * 16) + 256
    assert ws(0, 32, 12288, 3072) == 3072 * 256 + 12288 * 4 + 512 + 256
    assert ws(1, 32, 300, 192) == 0     # fp32 W: CUDA-core merge
    assert ws(0, 16, 300, 192) == 0     # rank other than 32
    assert ws(0, 32, 300, 100) == 0     # K % 64
    assert ws(0, 32, 0, 64) == 0


def test_gemm_validation(lib):
    P = ctypes.c_void_p
    a = [P(A16)] * 6
    assert lib.nvfp4_gemm(*a, None, P(A16), 16, 12, 64, None) == 2   # N % 8
    assert lib.nvfp4_gemm(*a, None, P(A16), 16, 16, 96, None) == 2   # K % 64
    assert lib.nvfp4_gemm(*a, None, None, 16, 16, 64, None) == 1
    assert lib.nvfp4_gemm(*a, P(BAD), P(A16), 16, 16, 64, None) == 3  # bias alignment
    assert lib.nvfp4_gemm(*a, None, P(A16), 0, 16, 64, None) == 0     # empty
    assert lib.bf16_gemm(P(A16), P(A16), None, P(A16), 16, 16, 12, None) == 2
    assert lib.bf16_gemm(P(A16), None, None, P(A16), 16, 16, 64, None) == 1
    assert lib.bf16_gemm(P(BAD), P(A16), None, P(A16), 16, 16, 64, None) == 3
    assert lib.bf16_gemm(P(A16), P(A16), None, P(A16), 16, 0, 64, None) == 0


def test_select_validation(lib):
    P = ctypes.c_void_p
    assert lib.select_contrastive(P(A16), 1, 96, 23, 1, P(A16), None, None) == 2
    assert lib.select_contrastive(P(A16), 1, 96, 98, 1, P(A16), None, None) == 2
    assert lib.select_contrastive(P(A16), 1, 2000, 24, 1, P(A16), None, None) == 2
    assert lib.select_contrastive(None, 1, 96, 24, 1, P(A16), None, None) == 1
    assert lib.select_contrastive(P(BAD + 1), 1, 96, 24, 1, P(A16), None, None) == 3
    assert lib.select_contrastive(None, 0, 96, 24, 1, None, None, None) == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="needs a machine without a usable GPU")
def test_well_formed_call_without_gpu_reports_cuda_error(lib):
    P = ctypes.c_void_p
    rc = lib.nvfp4_act_quant(P(A16), 4, 64, P(A16), P(A16), P(A16), None)
    assert rc in (4, 5)
    out = ctypes.c_int(-1)
    assert lib.nvfp4_device_status(ctypes.byref(out), 0) in (4, 5)


def test_binding_refuses_cpu_tensors(lib):
    import nvfp4_quantized_dit_gb300 as pkg
    with pytest.raises(ValueError):
        pkg.nvfp4_act_quant(torch.zeros(4, 64, dtype=torch.bfloat16),
                            codes=torch.zeros(4, 32, dtype=torch.uint8),
                            sf=torch.zeros(pkg.sf_bytes(4, 64), dtype=torch.uint8),
                            s_row=torch.zeros(4))


def test_requant_noalloc_checks_arguments_before_anything_else(lib):
    """nvfp4_requant_noalloc runs nvfp4_requant's argument checks first (before its
    size limit, the device's architecture and the scratch lookup)."""
    P, F = ctypes.c_void_p, ctypes.c_float
    f = lib.nvfp4_requant_noalloc
    # misaligned codes on a shape whose workspace would also exceed the scratch
    assert f(P(A16), 0, P(A16), P(A16), 32, F(32.0), 64, 65536, P(BAD), P(A16), P(A16), None) == 3
    assert f(P(A16), 0, P(A16), P(A16), 32, F(32.0), 64, 65536, P(A16), P(A16), None, None) == 1
    assert f(P(A16), 7, P(A16), P(A16), 32, F(32.0), 64, 128, P(A16), P(A16), P(A16), None) == 2
    # the same codes as nvfp4_requant for the same bad arguments
    g = lib.nvfp4_requant
    for args in [(P(A16), 0, P(A16), P(A16), 32, F(32.0), 64, 100, P(A16), P(A16), P(A16)),
                 (P(A16), 0, P(BAD), P(A16), 32, F(32.0), 64, 128, P(A16), P(A16), P(A16)),
                 (None, 0, P(A16), P(A16), 32, F(32.0), 64, 128, P(A16), P(A16), P(A16))]:
        assert f(*args, None) == g(*args, None, 0, None)


def test_gemm_withhold_hook_validation(lib):
    P = ctypes.c_void_p
    f = lib.nvfp4_test_gemm_withhold
    ok = [P(A16)] * 7
    assert f(*ok, 256, 256, 512, 2, 50_000_000, None) == 2   # stage 2 of a 2-stage K
    assert f(*ok, 256, 256, 512, -1, 50_000_000, None) == 2
    assert f(*ok, 256, 256, 512, 1, 10, None) == 2           # limit below 1 ms
    assert f(*ok, 256, 256, 100, 0, 50_000_000, None) == 2   # K % 64
    bad = list(ok)
    bad[6] = P(BAD)
    assert f(*bad, 256, 256, 512, 1, 50_000_000, None) == 3


def test_requant_exact_counts_validation(lib):
    """The diagnostic checks its arguments before any CUDA call."""
    P = ctypes.c_void_p
    f = lib.nvfp4_requant_exact_counts
    need = lib.nvfp4_requant_workspace_bytes(0, 32, 256, 1024)
    out = (ctypes.c_uint32 * 2)()
    assert f(None, need, 256, 1024, out, None) == 1
    assert f(P(A16), need, 256, 1024, None, None) == 1
    assert f(P(A16 + 16), need, 256, 1024, out, None) == 3       # workspace not 256-aligned
    assert f(P(A16), need - 1, 256, 1024, out, None) == 2        # too small
    assert f(P(A16), need, 256, 100, out, None) == 2             # K % 64
    assert f(P(A16), need, 0, 1024, out, None) == 2


def test_prescaled_and_rowamax_validation(lib):
    P = ctypes.c_void_p
    f = lib.nvfp4_act_quant_prescaled
    assert f(P(A16), 4, 100, P(A16), P(A16), P(A16), P(A16), None) == 2     # K % 64
    assert f(P(A16), 4, 64, None, P(A16), P(A16), P(A16), None) == 1        # row_amax
    assert f(P(A16), 4, 64, P(BAD), P(A16), P(A16), P(A16), None) == 3
    assert f(None, 0, 64, None, None, None, None, None) == 0                # nothing to do
    g = lib.nvfp4_gemm_rowamax
    ok = [P(A16)] * 8
    assert g(*ok, None, 4, 256, 256, None) == 1                              # y_row_amax
    assert g(*ok, P(BAD), 4, 256, 256, None) == 3
    assert g(*ok, P(A16), 4, 256, 100, None) == 2
    assert g(*ok, None, 0, 256, 256, None) == 0                              # M == 0


def test_block_entry_points_validation(lib):
    """The synthetic DiT block's entry points check shapes, pointers and alignment before
    any CUDA call (shape rules: D % 64, dh = D/H in {64, 128}, S % 64)."""
    P = ctypes.c_void_p
    W = (ctypes.c_void_p * 16)(*([A16] * 16))  # 4 x {codes, sf, s_t, bias}
    blk, att = lib.nvfp4_dit_block, lib.nvfp4_dit_attention
    need = lib.nvfp4_dit_block_workspace_bytes(2, 128, 256, 2)
    # shapes
    assert blk(P(A16), 2, 100, 256, 2, W, P(A16), P(A16), need, None) == 2      # S % 64
    assert blk(P(A16), 1, 128, 384, 2, W, P(A16), P(A16), need, None) == 2      # dh = 192
    assert blk(P(A16), 2, 128, 256, 2, W, P(A16), P(A16), need - 256, None) == 2  # workspace too small
    # pointers and alignment
    assert blk(None, 2, 128, 256, 2, W, P(A16), P(A16), need, None) == 1
    assert blk(P(A16), 2, 128, 256, 2, None, P(A16), P(A16), need, None) == 1
    W0 = (ctypes.c_void_p * 16)(*([A16] * 16))
    W0[2] = None  # the first linear's s_t
    assert blk(P(A16), 2, 128, 256, 2, W0, P(A16), P(A16), need, None) == 1
    assert blk(P(BAD), 2, 128, 256, 2, W, P(A16), P(A16), need, None) == 3
    assert blk(P(A16), 2, 128, 256, 2, W, P(A16), P(A16 + 16), need, None) == 3  # workspace 256-aligned
    need_a = lib.nvfp4_dit_attention_workspace_bytes(2, 128, 256, 2)
    assert att(P(A16), 2, 100, 256, 2, P(A16), P(A16), need_a, None) == 2
    assert att(None, 2, 128, 256, 2, P(A16), P(A16), need_a, None) == 1
    assert att(P(A16), 2, 128, 256, 2, P(BAD), P(A16), need_a, None) == 3
    assert att(P(A16), 2, 128, 256, 2, P(A16), P(A16), need_a - 1, None) == 2
    # the streaming steps
    assert lib.bf16_softmax_rows(P(A16), 4, 12, ctypes.c_float(1.0), P(A16), None) == 2   # cols % 8
    assert lib.bf16_softmax_rows(None, 0, 16, ctypes.c_float(1.0), None, None) == 0      # empty
    assert lib.bf16_softmax_rows(None, 4, 16, ctypes.c_float(1.0), P(A16), None) == 1
    assert lib.bf16_softmax_rows(P(BAD), 4, 16, ctypes.c_float(1.0), P(A16), None) == 3
    assert lib.bf16_gelu(P(A16), 12, P(A16), None) == 2
    assert lib.bf16_gelu(None, 0, None, None) == 0
    assert lib.bf16_gelu(P(A16), 16, None, None) == 1
    assert lib.bf16_add(P(A16), P(BAD), 16, P(A16), None) == 3
    assert lib.bf16_add(P(A16), P(A16), -8, P(A16), None) == 2


def test_block_workspace_sizes(lib):
    """0 for shapes outside the rules; otherwise 256-byte multiples that hold at least
    the block's bf16 intermediates (qkv, the MLP hidden, h1: 8 T D values), growing
    with the batch; the attention's scratch is V transposed (T D values)."""
    blk, att = lib.nvfp4_dit_block_workspace_bytes, lib.nvfp4_dit_attention_workspace_bytes
    for bad in [(1, 100, 256, 2), (1, 128, 256, 3), (1, 128, 384, 2), (0, 128, 256, 2), (1, 128, 96, 1)]:
        assert blk(*bad) == 0 and att(*bad) == 0
    prev = 0
    for B in (1, 2, 8):
        T, D = B * 4608, 3072
        n = blk(B, 4608, D, 24)
        assert n % 256 == 0 and n >= 2 * 8 * T * D and n > prev
        prev = n
        assert att(B, 4608, D, 24) == 2 * T * D
    assert blk(2, 128, 256, 4) > 0  # dh = 64


def test_attention_withhold_hook_validation(lib):
    P = ctypes.c_void_p
    f = lib.nvfp4_test_attention_withhold
    need = lib.nvfp4_dit_attention_workspace_bytes(2, 512, 256, 2)
    assert f(P(A16), 2, 512, 256, 2, P(A16), P(A16), need, 2, 50_000_000, None) == 2   # 2 tiles of 256 keys
    assert f(P(A16), 2, 512, 256, 2, P(A16), P(A16), need, -1, 50_000_000, None) == 2
    assert f(P(A16), 2, 512, 256, 2, P(A16), P(A16), need, 1, 10, None) == 2           # timeout range
    assert f(P(A16), 2, 500, 256, 2, P(A16), P(A16), need, 1, 50_000_000, None) == 2   # S % 64
    assert f(None, 2, 512, 256, 2, P(A16), P(A16), need, 1, 50_000_000, None) == 1


def test_header_is_plain_c(tmp_path):
    """The boundary is a C ABI: the header compiles as C99 and C11 (pedantic, all
    warnings as errors), structs and inline helpers included."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "nvfp4rl.h"\n'
                   "int main(void) {\n"
                   "    nvfp4_linear_weights w[4] = {{0}};\n"
                   "    (void)w;\n"
                   "    return nvfp4_sf_bytes(128, 64) == 512 && nvfp4_sf_offset(1, 0, 64) == 16 ? 0 : 1;\n"
                   "}\n")
    for std in ("c99", "c11"):
        exe = tmp_path / f"use_header_{std}"
        subprocess.run([gcc, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
        assert subprocess.run([str(exe)]).returncode == 0
