"""Python binding of libnvfp4rl, the NVFP4 FP4-explore hot path for GB300 (sm_103a).

Argument marshalling only: every function here checks tensor placement, dtype
and contiguity, allocates outputs with torch when the caller does not pass
them, and calls the C entry point of the same name (declared and documented in
include/nvfp4rl.h) with raw device pointers and the current CUDA stream.  All
arithmetic runs in the library's CUDA kernels; there is no fallback.  Importing
works without the library; the first call raises if ``libnvfp4rl.so`` has not
been built (``python -m nvfp4_quantized_dit_gb300.build``).
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "NVFP4Error", "library", "sf_bytes", "sf_offset",
    "nvfp4_requant", "requant_workspace_bytes", "nvfp4_requant_noalloc", "nvfp4_act_quant",
    "nvfp4_act_quant_tensor", "nvfp4_gemm", "bf16_gemm", "select_contrastive",
    "nvfp4_device_status", "nvfp4_status_string", "nvfp4_version",
    "nvfp4_test_e2m1", "nvfp4_test_e4m3", "nvfp4_test_e2m1_quotient", "nvfp4_test_e4m3_quotient",
    "nvfp4_test_e4m3_decode", "nvfp4_test_merge", "nvfp4_test_wait_timeout", "nvfp4_test_gemm_withhold", "nvfp4_test_attention_withhold",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libnvfp4rl.so")
_lock = threading.Lock()
_lib = None

STATUS = {0: "NVFP4_OK", 1: "NVFP4_ERR_NULL", 2: "NVFP4_ERR_SHAPE", 3: "NVFP4_ERR_ALIGN",
          4: "NVFP4_ERR_ARCH", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_TIMEOUT"}
W_BF16, W_FP32 = 0, 1


class NVFP4Error(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {STATUS.get(code, code)}")
        self.code = code


def library() -> ctypes.CDLL:
    """The loaded libnvfp4rl.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m nvfp4_quantized_dit_gb300.build` (nvcc, sm_103a)")
            L = ctypes.CDLL(LIB_PATH)
            P, I64, I, F = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
            sig = {
                "nvfp4_requant": [P, I, P, P, I, F, I64, I64, P, P, P, P, ctypes.c_size_t, P],
                "nvfp4_requant_noalloc": [P, I, P, P, I, F, I64, I64, P, P, P, P],
                "nvfp4_requant_exact_counts": [P, ctypes.c_size_t, I64, I64, P, P],
                "nvfp4_act_quant": [P, I64, I64, P, P, P, P],
                "nvfp4_act_quant_tensor": [P, I64, I64, P, P, P, P],
                "nvfp4_gemm": [P, P, P, P, P, P, P, P, I64, I64, I64, P],
                "nvfp4_gemm_rowamax": [P, P, P, P, P, P, P, P, P, I64, I64, I64, P],
                "nvfp4_act_quant_prescaled": [P, I64, I64, P, P, P, P, P],
                "nvfp4_dit_block": [P, I64, I64, I64, I64, P, P, P, ctypes.c_size_t, P],
                "nvfp4_dit_attention": [P, I64, I64, I64, I64, P, P, ctypes.c_size_t, P],
                "bf16_softmax_rows": [P, I64, I64, F, P, P],
                "bf16_gelu": [P, I64, P, P],
                "bf16_add": [P, P, I64, P, P],
                "bf16_gemm": [P, P, P, P, I64, I64, I64, P],
                "select_contrastive": [P, I, I, I, I, P, P, P],
                "nvfp4_device_status": [ctypes.POINTER(ctypes.c_int), I],
                "nvfp4_test_e2m1": [P, P, I64, P],
                "nvfp4_test_e4m3": [P, P, I64, P],
                "nvfp4_test_e2m1_quotient": [P, P, P, I64, P],
                "nvfp4_test_e4m3_quotient": [P, P, P, I64, P],
                "nvfp4_test_e4m3_decode": [P, P, I64, P],
                "nvfp4_test_merge": [P, I, P, P, I, F, I64, I64, P, P],
                "nvfp4_test_wait_timeout": [I64, P],
                "nvfp4_test_gemm_withhold": [P, P, P, P, P, P, P, I64, I64, I64, I, I64, P],
                "nvfp4_test_attention_withhold": [P, I64, I64, I64, I64, P, P, ctypes.c_size_t, I, I64, P],
            }
            for name, args in sig.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = I
            L.nvfp4_requant_workspace_bytes.argtypes = [I, I, I64, I64]
            L.nvfp4_requant_workspace_bytes.restype = ctypes.c_size_t
            for name in ("nvfp4_dit_block_workspace_bytes", "nvfp4_dit_attention_workspace_bytes"):
                getattr(L, name).argtypes = [I64, I64, I64, I64]
                getattr(L, name).restype = ctypes.c_size_t
            L.nvfp4_status_string.argtypes = [I]
            L.nvfp4_status_string.restype = ctypes.c_char_p
            L.nvfp4_version.argtypes = []
            L.nvfp4_version.restype = I
            _lib = L
    return _lib


def sf_bytes(rows: int, K: int) -> int:
    """Bytes of a scale-factor buffer for a [rows, K] NVFP4 tensor (128-row padded)."""
    return (rows + 127) // 128 * 128 * (K // 16)


def sf_offset(row: int, kblk: int, K: int) -> int:
    """Byte offset of the scale of (row, kblk) in the 128x4 blocked layout."""
    return ((row // 128) * (K // 64) + kblk // 4) * 512 + (row % 32) * 16 + ((row // 32) % 4) * 4 + kblk % 4


def _call(name: str, *args) -> None:
    rc = getattr(library(), name)(*args)
    if rc != 0:
        raise NVFP4Error(name, rc)


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, name, dtype=None):
    return None if t is None else _dev(t, name, dtype)


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def nvfp4_status_string(code: int) -> str:
    return library().nvfp4_status_string(int(code)).decode()


def nvfp4_version() -> int:
    return library().nvfp4_version()


def requant_workspace_bytes(w_dtype: int, r: int, N: int, K: int) -> int:
    """Workspace bytes that select the tensor-core merge of nvfp4_requant (0: n/a)."""
    return int(library().nvfp4_requant_workspace_bytes(int(w_dtype), int(r), int(N), int(K)))


def nvfp4_requant(W, A=None, B=None, alpha: float = 32.0, codes=None, sf=None, s_t=None,
                  stream=None, workspace=None):
    """W' = W + (alpha/r) B A, then per-tensor NVFP4.  Returns (codes, sf, s_t).

    ``workspace`` (uint8 CUDA tensor) is the call's scratch; when omitted and the
    tensor-core merge applies, one of nvfp4_requant_workspace_bytes is allocated."""
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    w_dtype = {torch.bfloat16: W_BF16, torch.float32: W_FP32}.get(W.dtype)
    if w_dtype is None:
        raise TypeError("W must be bfloat16 or float32")
    r = 0 if (A is None or B is None) else A.shape[0]
    if r and (tuple(A.shape) != (r, K) or tuple(B.shape) != (N, r)):
        raise ValueError(f"LoRA shapes A {tuple(A.shape)} / B {tuple(B.shape)} do not match W {tuple(W.shape)}")
    dev = W.device
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    sf = torch.empty(sf_bytes(N, K), dtype=torch.uint8, device=dev) if sf is None else sf
    s_t = torch.empty(1, dtype=torch.float32, device=dev) if s_t is None else s_t
    if workspace is None and r:
        need = requant_workspace_bytes(w_dtype, r, N, K)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = _opt(workspace, "workspace", torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel()
    _call("nvfp4_requant", _dev(W, "W"), w_dtype, _opt(A, "A", torch.float32), _opt(B, "B", torch.float32),
          r, ctypes.c_float(alpha), N, K, _dev(codes, "codes", torch.uint8), _dev(sf, "sf", torch.uint8),
          _dev(s_t, "s_t", torch.float32), ws_ptr, ws_bytes, _stream(stream))
    return codes, sf, s_t


def nvfp4_requant_noalloc(W, A=None, B=None, alpha: float = 32.0, codes=None, sf=None, s_t=None,
                          stream=None):
    """nvfp4_requant with the library's fixed device scratch instead of a workspace
    (outputs are still allocated here when the caller does not pass them)."""
    if W.dim() != 2:
        raise ValueError("W must be [N, K]")
    N, K = W.shape
    w_dtype = {torch.bfloat16: W_BF16, torch.float32: W_FP32}.get(W.dtype)
    if w_dtype is None:
        raise TypeError("W must be bfloat16 or float32")
    r = 0 if (A is None or B is None) else A.shape[0]
    if r and (tuple(A.shape) != (r, K) or tuple(B.shape) != (N, r)):
        raise ValueError(f"LoRA shapes A {tuple(A.shape)} / B {tuple(B.shape)} do not match W {tuple(W.shape)}")
    dev = W.device
    codes = torch.empty(N, K // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    sf = torch.empty(sf_bytes(N, K), dtype=torch.uint8, device=dev) if sf is None else sf
    s_t = torch.empty(1, dtype=torch.float32, device=dev) if s_t is None else s_t
    _call("nvfp4_requant_noalloc", _dev(W, "W"), w_dtype, _opt(A, "A", torch.float32),
          _opt(B, "B", torch.float32), r, ctypes.c_float(alpha), N, K, _dev(codes, "codes", torch.uint8),
          _dev(sf, "sf", torch.uint8), _dev(s_t, "s_t", torch.float32), _stream(stream))
    return codes, sf, s_t


def nvfp4_requant_exact_counts(workspace, N: int, K: int, stream=None):
    """(quantize-phase, amax-phase) element counts that the last tensor-core
    nvfp4_requant with this workspace merged by the exact fp32 chain."""
    out = (ctypes.c_uint32 * 2)()
    _call("nvfp4_requant_exact_counts", _dev(workspace, "workspace", torch.uint8), workspace.numel(),
          N, K, out, _stream(stream))
    return int(out[0]), int(out[1])


def nvfp4_act_quant(X, codes=None, sf=None, s_row=None, stream=None):
    """Per-row NVFP4 of bf16 activations X [M, K].  Returns (codes, sf, s_row)."""
    if X.dim() != 2:
        raise ValueError("X must be [M, K]")
    M, K = X.shape
    dev = X.device
    codes = torch.empty(M, K // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    sf = torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=dev) if sf is None else sf
    s_row = torch.empty(M, dtype=torch.float32, device=dev) if s_row is None else s_row
    _call("nvfp4_act_quant", _dev(X, "X", torch.bfloat16), M, K, _dev(codes, "codes", torch.uint8),
          _dev(sf, "sf", torch.uint8), _dev(s_row, "s_row", torch.float32), _stream(stream))
    return codes, sf, s_row


def nvfp4_act_quant_tensor(X, codes=None, sf=None, s_t=None, stream=None):
    """NVFP4 of bf16 activations X [M, K] with one per-tensor scale.  Returns
    (codes, sf, s_t)."""
    if X.dim() != 2:
        raise ValueError("X must be [M, K]")
    M, K = X.shape
    dev = X.device
    codes = torch.empty(M, K // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    sf = torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=dev) if sf is None else sf
    s_t = torch.empty(1, dtype=torch.float32, device=dev) if s_t is None else s_t
    _call("nvfp4_act_quant_tensor", _dev(X, "X", torch.bfloat16), M, K, _dev(codes, "codes", torch.uint8),
          _dev(sf, "sf", torch.uint8), _dev(s_t, "s_t", torch.float32), _stream(stream))
    return codes, sf, s_t


def nvfp4_gemm(a, w, bias=None, out=None, stream=None):
    """Y[M,N] bf16 from NVFP4 activations a = (codes, sf, s_row) and weights
    w = (codes, sf, s_t), plus an optional bf16 bias [N]."""
    a_codes, a_sf, a_s = a
    w_codes, w_sf, w_s = w
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    if w_codes.shape[1] * 2 != K:
        raise ValueError("activation and weight K differ")
    out = torch.empty(M, N, dtype=torch.bfloat16, device=a_codes.device) if out is None else out
    _call("nvfp4_gemm", _dev(a_codes, "a_codes", torch.uint8), _dev(a_sf, "a_sf", torch.uint8),
          _dev(a_s, "a_srow", torch.float32), _dev(w_codes, "w_codes", torch.uint8),
          _dev(w_sf, "w_sf", torch.uint8), _dev(w_s, "w_st", torch.float32),
          _opt(bias, "bias", torch.bfloat16), _dev(out, "Y", torch.bfloat16), M, N, K, _stream(stream))
    return out


def nvfp4_gemm_rowamax(a, w, bias=None, out=None, row_amax=None, stream=None):
    """nvfp4_gemm that also returns amax|Y[m, :]| per row (fp32 [M]): (Y, row_amax)."""
    a_codes, a_sf, a_s = a
    w_codes, w_sf, w_s = w
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    if w_codes.shape[1] * 2 != K:
        raise ValueError("activation and weight K differ")
    dev = a_codes.device
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev) if out is None else out
    row_amax = torch.empty(M, dtype=torch.float32, device=dev) if row_amax is None else row_amax
    _call("nvfp4_gemm_rowamax", _dev(a_codes, "a_codes", torch.uint8), _dev(a_sf, "a_sf", torch.uint8),
          _dev(a_s, "a_srow", torch.float32), _dev(w_codes, "w_codes", torch.uint8),
          _dev(w_sf, "w_sf", torch.uint8), _dev(w_s, "w_st", torch.float32),
          _opt(bias, "bias", torch.bfloat16), _dev(out, "Y", torch.bfloat16),
          _dev(row_amax, "row_amax", torch.float32), M, N, K, _stream(stream))
    return out, row_amax


def nvfp4_act_quant_prescaled(X, row_amax, codes=None, sf=None, s_row=None, stream=None):
    """nvfp4_act_quant of X [M, K] given amax|X[m, :]| per row (fp32 [M]), e.g. from
    nvfp4_gemm_rowamax.  Returns (codes, sf, s_row)."""
    if X.dim() != 2:
        raise ValueError("X must be [M, K]")
    M, K = X.shape
    if row_amax.numel() != M:
        raise ValueError("row_amax must hold one value per row of X")
    dev = X.device
    codes = torch.empty(M, K // 2, dtype=torch.uint8, device=dev) if codes is None else codes
    sf = torch.empty(sf_bytes(M, K), dtype=torch.uint8, device=dev) if sf is None else sf
    s_row = torch.empty(M, dtype=torch.float32, device=dev) if s_row is None else s_row
    _call("nvfp4_act_quant_prescaled", _dev(X, "X", torch.bfloat16), M, K,
          _dev(row_amax, "row_amax", torch.float32), _dev(codes, "codes", torch.uint8),
          _dev(sf, "sf", torch.uint8), _dev(s_row, "s_row", torch.float32), _stream(stream))
    return codes, sf, s_row


def bf16_gemm(X, W, bias=None, out=None, stream=None):
    """Y = X W^T (+ bias), bf16 in and out, fp32 accumulation."""
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("X and W K differ")
    out = torch.empty(M, N, dtype=torch.bfloat16, device=X.device) if out is None else out
    _call("bf16_gemm", _dev(X, "X", torch.bfloat16), _dev(W, "W", torch.bfloat16),
          _opt(bias, "bias", torch.bfloat16), _dev(out, "Y", torch.bfloat16), M, N, K, _stream(stream))
    return out


def select_contrastive(rewards, K: int, global_std: bool = True, with_transform: bool = True,
                       idx=None, r=None, stream=None):
    """Top K/2 and bottom K/2 seeds per prompt plus the NFT reward transform.
    Returns (idx [P,K] int32, r [P,K] float32 or None)."""
    P, N = rewards.shape
    dev = rewards.device
    idx = torch.empty(P, K, dtype=torch.int32, device=dev) if idx is None else idx
    if with_transform and r is None:
        r = torch.empty(P, K, dtype=torch.float32, device=dev)
    if not with_transform:
        r = None
    _call("select_contrastive", _dev(rewards, "rewards", torch.float32), P, N, K, int(bool(global_std)),
          _dev(idx, "idx", torch.int32), _opt(r, "r_out", torch.float32), _stream(stream))
    return idx, r


def nvfp4_device_status(clear: bool = True) -> int:
    """Device status word (0 or NVFP4_ERR_TIMEOUT); synchronizes the device."""
    out = ctypes.c_int(-1)
    _call("nvfp4_device_status", ctypes.byref(out), int(bool(clear)))
    return out.value


def nvfp4_test_e2m1(q, out=None, stream=None):
    out = torch.empty(q.numel(), dtype=torch.uint8, device=q.device) if out is None else out
    _call("nvfp4_test_e2m1", _dev(q, "q", torch.float32), _dev(out, "codes", torch.uint8), q.numel(),
          _stream(stream))
    return out


def nvfp4_test_e4m3(v, out=None, stream=None):
    out = torch.empty(v.numel(), dtype=torch.uint8, device=v.device) if out is None else out
    _call("nvfp4_test_e4m3", _dev(v, "v", torch.float32), _dev(out, "codes", torch.uint8), v.numel(),
          _stream(stream))
    return out


def nvfp4_test_e4m3_decode(codes, out=None, stream=None):
    out = torch.empty(codes.numel(), dtype=torch.float32, device=codes.device) if out is None else out
    _call("nvfp4_test_e4m3_decode", _dev(codes, "codes", torch.uint8), _dev(out, "out", torch.float32),
          codes.numel(), _stream(stream))
    return out


def nvfp4_test_e2m1_quotient(x, den, out=None, stream=None):
    out = torch.empty(x.numel(), dtype=torch.uint8, device=x.device) if out is None else out
    _call("nvfp4_test_e2m1_quotient", _dev(x, "x", torch.float32), _dev(den, "den", torch.float32),
          _dev(out, "codes", torch.uint8), x.numel(), _stream(stream))
    return out


def nvfp4_test_e4m3_quotient(v, d, out=None, stream=None):
    out = torch.empty(v.numel(), dtype=torch.uint8, device=v.device) if out is None else out
    _call("nvfp4_test_e4m3_quotient", _dev(v, "v", torch.float32), _dev(d, "d", torch.float32),
          _dev(out, "codes", torch.uint8), v.numel(), _stream(stream))
    return out


def nvfp4_test_merge(W, A=None, B=None, alpha: float = 32.0, out=None, stream=None):
    """The merged weights W' [N, K] (fp32) exactly as nvfp4_requant forms them."""
    N, K = W.shape
    w_dtype = {torch.bfloat16: W_BF16, torch.float32: W_FP32}.get(W.dtype)
    if w_dtype is None:
        raise TypeError("W must be bfloat16 or float32")
    r = 0 if (A is None or B is None) else A.shape[0]
    out = torch.empty(N, K, dtype=torch.float32, device=W.device) if out is None else out
    _call("nvfp4_test_merge", _dev(W, "W"), w_dtype, _opt(A, "A", torch.float32),
          _opt(B, "B", torch.float32), r, ctypes.c_float(alpha), N, K,
          _dev(out, "out", torch.float32), _stream(stream))
    return out


def nvfp4_test_wait_timeout(timeout_ns: int, stream=None) -> None:
    _call("nvfp4_test_wait_timeout", int(timeout_ns), _stream(stream))


def nvfp4_test_gemm_withhold(a, w, withhold_kb: int, timeout_ns: int, out=None, stream=None):
    """nvfp4_gemm with one K-stage of the first CTA pair never loaded (test hook of the
    GEMM's abort path); returns the (incomplete) output."""
    a_codes, a_sf, a_s = a
    w_codes, w_sf, w_s = w
    M, K = a_codes.shape[0], a_codes.shape[1] * 2
    N = w_codes.shape[0]
    out = torch.empty(M, N, dtype=torch.bfloat16, device=a_codes.device) if out is None else out
    _call("nvfp4_test_gemm_withhold", _dev(a_codes, "a_codes", torch.uint8), _dev(a_sf, "a_sf", torch.uint8),
          _dev(a_s, "a_srow", torch.float32), _dev(w_codes, "w_codes", torch.uint8),
          _dev(w_sf, "w_sf", torch.uint8), _dev(w_s, "w_st", torch.float32), _dev(out, "Y", torch.bfloat16),
          M, N, K, int(withhold_kb), int(timeout_ns), _stream(stream))
    return out


# ---------------------------------------------------------------- synthetic DiT block

class _LinearWeights(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("s_t", ctypes.c_void_p),
                ("bias", ctypes.c_void_p)]


def dit_block_workspace_bytes(B: int, S: int, D: int, H: int) -> int:
    return int(library().nvfp4_dit_block_workspace_bytes(B, S, D, H))


def dit_attention_workspace_bytes(B: int, S: int, D: int, H: int) -> int:
    return int(library().nvfp4_dit_attention_workspace_bytes(B, S, D, H))


def _workspace(nbytes: int, dev, workspace):
    if nbytes == 0:
        raise NVFP4Error("workspace size", 2)  # NVFP4_ERR_SHAPE: the shape rules of the block
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    return workspace


def nvfp4_dit_block(x, B: int, S: int, H: int, weights, out=None, workspace=None, stream=None):
    """The synthetic DiT block on bf16 x [B*S, D]; weights: 4 tuples (codes, sf, s_t,
    bias or None) for qkv, o, up, dn, as nvfp4_requant returns them.  Returns out."""
    T, D = x.shape
    if T != B * S:
        raise ValueError("x must be [B*S, D]")
    if len(weights) != 4:
        raise ValueError("weights: qkv, o, up, dn")
    arr = (_LinearWeights * 4)()
    for i, wt in enumerate(weights):
        codes, sf, s_t, bias = wt
        arr[i] = _LinearWeights(_dev(codes, "codes", torch.uint8), _dev(sf, "sf", torch.uint8),
                                _dev(s_t, "s_t", torch.float32), _opt(bias, "bias", torch.bfloat16))
    out = torch.empty_like(x) if out is None else out
    workspace = _workspace(dit_block_workspace_bytes(B, S, D, H), x.device, workspace)
    _call("nvfp4_dit_block", _dev(x, "x", torch.bfloat16), B, S, D, H, arr, _dev(out, "out", torch.bfloat16),
          _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    return out


def nvfp4_dit_attention(qkv, B: int, S: int, H: int, o=None, workspace=None, stream=None):
    """The block's attention: qkv [B*S, 3D] bf16 -> o [B*S, D] bf16."""
    T, D3 = qkv.shape
    D = D3 // 3
    o = torch.empty(T, D, dtype=torch.bfloat16, device=qkv.device) if o is None else o
    workspace = _workspace(dit_attention_workspace_bytes(B, S, D, H), qkv.device, workspace)
    _call("nvfp4_dit_attention", _dev(qkv, "qkv", torch.bfloat16), B, S, D, H, _dev(o, "o", torch.bfloat16),
          _dev(workspace, "workspace", torch.uint8), workspace.numel(), _stream(stream))
    return o


def nvfp4_test_attention_withhold(qkv, B: int, S: int, H: int, withhold_tile: int, timeout_ns: int, stream=None):
    """nvfp4_dit_attention with one K tile of the first CTA pair never loaded (test hook
    of the attention's abort path); returns the (incomplete) output."""
    T, D3 = qkv.shape
    D = D3 // 3
    o = torch.empty(T, D, dtype=torch.bfloat16, device=qkv.device)
    workspace = _workspace(dit_attention_workspace_bytes(B, S, D, H), qkv.device, None)
    _call("nvfp4_test_attention_withhold", _dev(qkv, "qkv", torch.bfloat16), B, S, D, H, _dev(o, "o", torch.bfloat16),
          _dev(workspace, "workspace", torch.uint8), workspace.numel(), int(withhold_tile), int(timeout_ns),
          _stream(stream))
    return o


def bf16_softmax_rows(L, scale: float, P=None, stream=None):
    rows, cols = L.shape
    P = torch.empty_like(L) if P is None else P
    _call("bf16_softmax_rows", _dev(L, "L", torch.bfloat16), rows, cols, ctypes.c_float(scale),
          _dev(P, "P", torch.bfloat16), _stream(stream))
    return P


def bf16_gelu(x, y=None, stream=None):
    y = torch.empty_like(x) if y is None else y
    _call("bf16_gelu", _dev(x, "x", torch.bfloat16), x.numel(), _dev(y, "y", torch.bfloat16), _stream(stream))
    return y


def bf16_add(a, b, y=None, stream=None):
    if a.shape != b.shape:
        raise ValueError("a and b differ in shape")
    y = torch.empty_like(a) if y is None else y
    _call("bf16_add", _dev(a, "a", torch.bfloat16), _dev(b, "b", torch.bfloat16), a.numel(),
          _dev(y, "y", torch.bfloat16), _stream(stream))
    return y
