"""CPU oracle for the NVFP4 FP4-explore hot path (TEST INFRASTRUCTURE ONLY).

A thin ctypes wrapper over ``oracle.c``: a plain, slow, obviously correct CPU
restatement of what the hot path computes (see that file's header for the
sources and the readings).  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference legs may import this package.  The CUDA
library and its Python binding never import it, and it imports nothing from
them.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-std=c11", "-Wall"]


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (plain C11, OpenMP, no FP contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            F = ctypes.c_float
            L.orc_num_threads.restype = I
            L.orc_set_num_threads.argtypes = [I]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [I]
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [I]
            L.orc_e2m1_rne_sat.restype = I
            L.orc_e2m1_rne_sat.argtypes = [F]
            L.orc_e4m3_rne_sat.restype = I
            L.orc_e4m3_rne_sat.argtypes = [F]
            L.orc_e2m1_rne_sat_array.argtypes = [P, I64, P]
            L.orc_e4m3_rne_sat_array.argtypes = [P, I64, P]
            L.orc_merge.argtypes = [P, I, P, P, I, F, I64, I64, P]
            L.orc_quantize.restype = I
            L.orc_quantize.argtypes = [P, I64, I64, I, P, P, P]
            L.orc_dequantize.argtypes = [P, P, P, I, I64, I64, P]
            L.orc_gemm_nvfp4.argtypes = [P, P, P, P, P, F, P, I64, I64, I64, P, I64, P, P]
            L.orc_gemm_nvfp4_exact.argtypes = [P, P, P, P, I64, I64, P, I64, P]
            L.orc_gemm_bf16.argtypes = [P, P, P, I64, I64, I64, P, I64, P, P]
            L.orc_select_contrastive.restype = I
            L.orc_select_contrastive.argtypes = [P, I, I, I, I, P, P]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    lib().orc_set_num_threads(int(n))


# ---------------------------------------------------------------- formats

def e2m1_decode(code: int) -> float:
    return lib().orc_e2m1_decode(int(code))


def e4m3_decode(code: int) -> float:
    return lib().orc_e4m3_decode(int(code))


def e2m1_rne(q) -> np.ndarray:
    """RNE to E2M1 (sign kept, saturating at 6) of fp32 values; one code per byte."""
    q = _c(q, np.float32).reshape(-1)
    out = np.empty(q.size, np.uint8)
    lib().orc_e2m1_rne_sat_array(_p(q), q.size, _p(out))
    return out


def e4m3_rne(v) -> np.ndarray:
    """RNE to E4M3 (saturating at 448) of non-negative fp32 values."""
    v = _c(v, np.float32).reshape(-1)
    out = np.empty(v.size, np.uint8)
    lib().orc_e4m3_rne_sat_array(_p(v), v.size, _p(out))
    return out


# ---------------------------------------------------------------- merge / quantize

def merge(W, A, B, alpha: float) -> np.ndarray:
    """W' = W + (alpha/r) B A as an fmaf chain.  W: float32 array, or uint16 bf16 bits."""
    W = np.ascontiguousarray(W)
    if W.dtype == np.uint16:
        w_dtype = 0
    elif W.dtype == np.float32:
        w_dtype = 1
    else:
        raise TypeError("W must be float32 or bf16 bits (uint16)")
    N, K = W.shape
    if A is None or B is None:
        r = 0
        A_ = B_ = None
    else:
        A_ = _c(A, np.float32)
        B_ = _c(B, np.float32)
        r = A_.shape[0]
        assert A_.shape == (r, K) and B_.shape == (N, r)
    out = np.empty((N, K), np.float32)
    lib().orc_merge(_p(W), w_dtype, _p(A_), _p(B_), r, ctypes.c_float(alpha), N, K, _p(out))
    return out


def quantize(x, scope: str):
    """NVFP4-quantize float32 x [rows, K]; scope 'tensor' or 'row'.

    Returns (codes [rows, K/2] uint8, sf [rows, K/16] uint8 row-major, s float32
    [1] or [rows])."""
    x = _c(x, np.float32)
    rows, K = x.shape
    codes = np.empty((rows, K // 2), np.uint8)
    sf = np.empty((rows, K // 16), np.uint8)
    s = np.empty(1 if scope == "tensor" else rows, np.float32)
    rc = lib().orc_quantize(_p(x), rows, K, 0 if scope == "tensor" else 1, _p(codes), _p(sf), _p(s))
    if rc != 0:
        raise ValueError(f"orc_quantize: bad shape {x.shape}")
    return codes, sf, s


def dequantize(codes, sf, s, scope: str) -> np.ndarray:
    codes = _c(codes, np.uint8)
    sf = _c(sf, np.uint8)
    s = _c(s, np.float32).reshape(-1)
    rows = codes.shape[0]
    K = codes.shape[1] * 2
    out = np.empty((rows, K), np.float64)
    lib().orc_dequantize(_p(codes), _p(sf), _p(s), 0 if scope == "tensor" else 1, rows, K, _p(out))
    return out


def requant(W, A, B, alpha: float):
    """Merge then per-tensor NVFP4 quantize: (codes, sf row-major, s_t[1])."""
    return quantize(merge(W, A, B, alpha), "tensor")


def act_quant(x_bits):
    """Per-row NVFP4 quantize of bf16 activations given as uint16 bits [M, K]."""
    x_bits = _c(x_bits, np.uint16)
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    return quantize(x, "row")


# ---------------------------------------------------------------- GEMMs

def _rows(rows, M):
    if rows is None:
        rows = np.arange(M, dtype=np.int64)
    return _c(rows, np.int64)


def gemm_nvfp4(a_codes, a_sf, a_s, w_codes, w_sf, w_s, bias_bits=None, rows=None):
    """fp64 reference y[rows, N] and S[rows, N] for the NVFP4 GEMM (sf row-major)."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    a_s = _c(a_s, np.float32).reshape(-1)
    w_codes = _c(w_codes, np.uint8)
    w_sf = _c(w_sf, np.uint8)
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    rows = _rows(rows, M)
    bias_bits = None if bias_bits is None else _c(bias_bits, np.uint16)
    y = np.empty((rows.size, N), np.float64)
    S = np.empty((rows.size, N), np.float64)
    lib().orc_gemm_nvfp4(_p(a_codes), _p(a_sf), _p(a_s), _p(w_codes), _p(w_sf),
                         ctypes.c_float(float(np.float32(np.asarray(w_s).reshape(-1)[0]))),
                         _p(bias_bits), M, N, K, _p(rows), rows.size, _p(y), _p(S))
    return y, S


def gemm_nvfp4_exact(a_codes, a_sf, w_codes, w_sf, rows=None) -> np.ndarray:
    """Integer T[rows, N] with sum_k a_hat*w_hat = a_s * w_s * 2^-20 * T exactly."""
    a_codes = _c(a_codes, np.uint8)
    a_sf = _c(a_sf, np.uint8)
    w_codes = _c(w_codes, np.uint8)
    w_sf = _c(w_sf, np.uint8)
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    rows = _rows(rows, M)
    T = np.empty((rows.size, N), np.int64)
    lib().orc_gemm_nvfp4_exact(_p(a_codes), _p(a_sf), _p(w_codes), _p(w_sf), N, K, _p(rows),
                               rows.size, _p(T))
    return T


def gemm_bf16(x_bits, w_bits, bias_bits=None, rows=None):
    """fp64 reference y[rows, N] and S[rows, N] for Y = X W^T (+ bias), bf16 inputs as bits."""
    x_bits = _c(x_bits, np.uint16)
    w_bits = _c(w_bits, np.uint16)
    M, K = x_bits.shape
    N = w_bits.shape[0]
    rows = _rows(rows, M)
    bias_bits = None if bias_bits is None else _c(bias_bits, np.uint16)
    y = np.empty((rows.size, N), np.float64)
    S = np.empty((rows.size, N), np.float64)
    lib().orc_gemm_bf16(_p(x_bits), _p(w_bits), _p(bias_bits), M, N, K, _p(rows), rows.size,
                        _p(y), _p(S))
    return y, S


# ---------------------------------------------------------------- selection

def select_contrastive(rewards, K: int, global_std: bool = True, with_transform: bool = True):
    """Returns (idx [P,K] int32, r [P,K] float32 or None)."""
    rewards = _c(rewards, np.float32)
    P, N = rewards.shape
    idx = np.empty((P, K), np.int32)
    r = np.empty((P, K), np.float32) if with_transform else None
    rc = lib().orc_select_contrastive(_p(rewards), P, N, K, int(bool(global_std)), _p(idx), _p(r))
    if rc != 0:
        raise ValueError(f"select_contrastive: bad shape P={P} N={N} K={K}")
    return idx, r
