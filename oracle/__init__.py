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
            L.orc_bf16_rne.restype = ctypes.c_uint16
            L.orc_bf16_rne.argtypes = [ctypes.c_double]
            L.orc_bf16_rne_array.argtypes = [P, I64, P]
            L.orc_softmax_bf16.argtypes = [P, I64, I64, ctypes.c_double, P]
            L.orc_gelu_f64.argtypes = [P, I64, P]
            L.orc_gelu_bf16.argtypes = [P, I64, P]
            L.orc_add_bf16.argtypes = [P, P, I64, P]
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


# ---------------------------------------------------------------- DiT block (reading R15 of oracle.c's header)

def bf16_rne(x) -> np.ndarray:
    """Nearest bf16 (ties to even) of float64 values, as uint16 bits (same shape)."""
    x = np.asarray(x, np.float64)
    flat = _c(x, np.float64).reshape(-1)
    out = np.empty(flat.size, np.uint16)
    lib().orc_bf16_rne_array(_p(flat), flat.size, _p(out))
    return out.reshape(x.shape)


def bf16_value(bits) -> np.ndarray:
    """float64 values of bf16 bit patterns."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def softmax_bf16(L_bits, scale: float) -> np.ndarray:
    """bf16(softmax(scale * L)) per row of bf16 logits [rows, cols] (exact in double)."""
    L_bits = _c(L_bits, np.uint16)
    rows, cols = L_bits.shape
    out = np.empty((rows, cols), np.uint16)
    lib().orc_softmax_bf16(_p(L_bits), rows, cols, ctypes.c_double(scale), _p(out))
    return out


def gelu_f64(x) -> np.ndarray:
    x = _c(x, np.float64)
    y = np.empty_like(x)
    lib().orc_gelu_f64(_p(x), x.size, _p(y))
    return y


def gelu_bf16(x_bits) -> np.ndarray:
    x_bits = _c(x_bits, np.uint16)
    y = np.empty_like(x_bits)
    lib().orc_gelu_bf16(_p(x_bits), x_bits.size, _p(y))
    return y


def add_bf16(a_bits, b_bits) -> np.ndarray:
    a_bits = _c(a_bits, np.uint16)
    b_bits = _c(b_bits, np.uint16)
    assert a_bits.shape == b_bits.shape
    y = np.empty_like(a_bits)
    lib().orc_add_bf16(_p(a_bits), _p(b_bits), a_bits.size, _p(y))
    return y


def attention_head(q_bits, k_bits, v_bits) -> np.ndarray:
    """One head: O = bf16(P V) with P = bf16(softmax(bf16(q k^T) * scale)), scale the
    fp32 value of 1 / sqrt(dh); q, k, v [S, dh] bf16 bits.  Returns O [S, dh] bits."""
    q_bits, k_bits, v_bits = (_c(t, np.uint16) for t in (q_bits, k_bits, v_bits))
    dh = q_bits.shape[1]
    logits, _ = gemm_bf16(q_bits, k_bits)
    # The scale is the fp32 value 1 / sqrt(dh) (two fp32 operations, IEEE rounding).
    scale = float(np.float32(1.0) / np.sqrt(np.float32(dh)))
    P = softmax_bf16(bf16_rne(logits), scale)
    o, _ = gemm_bf16(P, np.ascontiguousarray(v_bits.T))
    return bf16_rne(o)


def attention(qkv_bits, B: int, S: int, H: int) -> np.ndarray:
    """Multi-head attention of the block: qkv [B*S, 3D] bf16 bits (q, k, v side by
    side, head h in columns h*dh .. of each); returns o [B*S, D] bits."""
    qkv_bits = _c(qkv_bits, np.uint16)
    T, D3 = qkv_bits.shape
    D = D3 // 3
    dh = D // H
    o = np.empty((T, D), np.uint16)
    for b in range(B):
        rs = slice(b * S, (b + 1) * S)
        for h in range(H):
            c = slice(h * dh, (h + 1) * dh)
            o[rs, c] = attention_head(qkv_bits[rs, c], qkv_bits[rs, D + h * dh:D + (h + 1) * dh],
                                      qkv_bits[rs, 2 * D + h * dh:2 * D + (h + 1) * dh])
    return o


def nvfp4_linear(x_bits, w, bias_bits=None) -> np.ndarray:
    """bf16(NVFP4 GEMM) of bf16 activations x [T, K] (quantized per row) with weights
    w = (codes, sf row-major, s_t) from requant; returns [T, N] bits."""
    ac, asf, a_s = act_quant(x_bits)
    y, _ = gemm_nvfp4(ac, asf, a_s, *w, bias_bits)
    return bf16_rne(y)


def dit_block(x_bits, w, bias, B: int, S: int, H: int) -> dict:
    """The synthetic DiT block (reading R15 of oracle.c's header) on bf16 x [B*S, D]:
    qkv = lin(x, qkv); o = attention(qkv); h1 = bf16(lin(o, o) + x);
    out = bf16(lin(gelu(lin(h1, up)), dn) + h1), every lin an NVFP4 linear (per-row
    activation quantization) with bias.  w and bias: dicts keyed 'qkv', 'o', 'up',
    'dn' (weights as returned by requant, bias as bf16 bits or None).  Returns every
    intermediate (bits)."""
    r = {}
    r["qkv"] = nvfp4_linear(x_bits, w["qkv"], bias.get("qkv"))
    r["o"] = attention(r["qkv"], B, S, H)
    r["h1"] = add_bf16(nvfp4_linear(r["o"], w["o"], bias.get("o")), x_bits)
    r["u"] = nvfp4_linear(r["h1"], w["up"], bias.get("up"))
    r["g"] = gelu_bf16(r["u"])
    r["out"] = add_bf16(nvfp4_linear(r["g"], w["dn"], bias.get("dn")), r["h1"])
    return r


def linear_unquantized(x_bits, w, bias_bits=None) -> np.ndarray:
    """bf16(x W^T + bias) with the NVFP4 weights w = (codes, sf row-major, s_t)
    dequantized and the bf16 activations x [T, K] used as they are (no activation
    quantization), the product in fp64 (a library matmul).  Returns [T, N] bits.  The
    distance of a block built on it from the NVFP4 block measures what the activation
    quantizer's decisions do to the result."""
    codes, sf, s_t = w
    W = dequantize(codes, sf, np.asarray(s_t, np.float32).reshape(-1)[:1], "tensor")
    y = bf16_value(_c(x_bits, np.uint16)) @ W.T
    if bias_bits is not None:
        y = y + bf16_value(_c(bias_bits, np.uint16))[None, :]
    return bf16_rne(y)


def dit_block_rows(x_bits, w, bias, B: int, S: int, H: int, rows,
                   quantize_activations: bool = True) -> np.ndarray:
    """dit_block's output at the token rows `rows` only, for inputs too large to run
    whole.  Every step of the block but the attention maps a row to the same row (the
    activation quantization is per row), so those steps run on the chosen rows alone;
    the attention of a row reads the keys and values of every token of its image, so
    those (columns D..3D of the qkv linear) are formed for each image that holds a
    chosen row.  With quantize_activations=False every linear is linear_unquantized
    instead (the same weights, activations not quantized).  Returns out[rows]
    [len(rows), D] bits."""
    x_bits = _c(x_bits, np.uint16)
    T, D = x_bits.shape
    dh = D // H
    rows = np.asarray(rows, np.int64).reshape(-1)
    lin = nvfp4_linear if quantize_activations else linear_unquantized
    codes, sf, s_t = w["qkv"]
    bq = bias.get("qkv")
    bq = None if bq is None else _c(bq, np.uint16)
    if quantize_activations:
        ac, asf, a_s = act_quant(x_bits)
    o = np.empty((rows.size, D), np.uint16)
    for b in np.unique(rows // S):
        sel = np.nonzero(rows // S == b)[0]
        img = slice(int(b) * S, (int(b) + 1) * S)
        w_kv = (codes[D:3 * D], sf[D:3 * D], s_t)
        w_q = (codes[:D], sf[:D], s_t)
        b_kv = None if bq is None else bq[D:3 * D]
        b_q = None if bq is None else bq[:D]
        if quantize_activations:
            kv = bf16_rne(gemm_nvfp4(ac[img], asf[img], a_s[img], *w_kv, b_kv)[0])
            q = bf16_rne(gemm_nvfp4(ac, asf, a_s, *w_q, b_q, rows=rows[sel])[0])
        else:
            kv = linear_unquantized(x_bits[img], w_kv, b_kv)
            q = linear_unquantized(x_bits[rows[sel]], w_q, b_q)
        for h in range(H):
            c = slice(h * dh, (h + 1) * dh)
            o[sel, c] = attention_head(q[:, c], kv[:, c], kv[:, D + h * dh:D + (h + 1) * dh])
    h1 = add_bf16(lin(o, w["o"], bias.get("o")), x_bits[rows])
    g = gelu_bf16(lin(h1, w["up"], bias.get("up")))
    return add_bf16(lin(g, w["dn"], bias.get("dn")), h1)
