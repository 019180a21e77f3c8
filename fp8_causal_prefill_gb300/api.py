"""Thin Python binding of libzyfa.so (argument marshalling only; every step runs in the CUDA library).

``zyfa_attn_fwd_causal`` mirrors the C entry point (raw device addresses and sizes);
``flash_attn_func`` is the tensor-level call in the flash_attn_func style the pages describe
(spbcomputers.ru ZYFA article, intro: a drop-in flash_attn_func-compatible interface).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libzyfa.so")
_lib = None
_lock = threading.Lock()

ZYFA_DTYPE_E4M3 = 0
ZYFA_DTYPE_BF16 = 1
STATUS = {0: "ZYFA_OK", 1: "ZYFA_ERR_INVALID_ARG", 2: "ZYFA_ERR_UNSUPPORTED", 3: "ZYFA_ERR_MISALIGNED",
          4: "ZYFA_ERR_CUDA", 5: "ZYFA_ERR_TIMEOUT"}
EXPORTED = ("zyfa_attn_fwd_causal", "zyfa_attn_fwd_causal_ex", "zyfa_attn_fwd_causal_host", "zyfa_check_errors",
            "zyfa_status_string",
            "zyfa_kernel_launches", "zyfa_selftest_stalled_pipeline", "zyfa_hadamard_quantize_e4m3",
            "zyfa_hadamard_quantize_e4m3_noalloc", "zyfa_hadamard_quantize_qk_e4m3", "zyfa_hadamard_workspace_bytes",
            "zyfa_probe_mma_rate",
            "zyfa_probe_mma_flops_per_iter", "zyfa_probe_mma_form_rate", "zyfa_probe_mma_form_flops_per_iter")
ZYFA_P_LEAN = 0
ZYFA_P_EXACT = 1
ZYFA_P_EXACT_NO_BLOCK_SCALE = 2
_P_MODES = {"lean": ZYFA_P_LEAN, "exact": ZYFA_P_EXACT, "exact-noblock": ZYFA_P_EXACT_NO_BLOCK_SCALE}


class FwdOptions(ctypes.Structure):
    """zyfa_fwd_options_t: p_mode, descale_per_kv_head, lse (device pointer or None)."""
    _fields_ = [("p_mode", ctypes.c_int), ("descale_per_kv_head", ctypes.c_int), ("lse", ctypes.c_void_p)]


class ZyfaError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


def library_path() -> str:
    return _LIB_PATH


def load_library() -> ctypes.CDLL:
    """Load libzyfa.so; raises if it has not been built (there is no fallback path)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ZyfaError(4, f"{_LIB_PATH} is missing; build it with `python -m fp8_causal_prefill_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, ci, cf = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.zyfa_attn_fwd_causal.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, vp, vp, vp]
        lib.zyfa_attn_fwd_causal.restype = ci
        lib.zyfa_attn_fwd_causal_ex.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci, vp, vp, vp,
                                                ctypes.POINTER(FwdOptions), vp]
        lib.zyfa_attn_fwd_causal_ex.restype = ci
        lib.zyfa_attn_fwd_causal_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, cf, ci,
                                                  vp, vp, vp, ci, vp]
        lib.zyfa_attn_fwd_causal_host.restype = ci
        lib.zyfa_selftest_stalled_pipeline.argtypes = [vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, ci, vp]
        lib.zyfa_selftest_stalled_pipeline.restype = ci
        ll, sz = ctypes.c_longlong, ctypes.c_size_t
        lib.zyfa_hadamard_quantize_e4m3.argtypes = [vp, vp, vp, ll, ci, vp, sz, vp]
        lib.zyfa_hadamard_quantize_e4m3.restype = ci
        lib.zyfa_hadamard_quantize_qk_e4m3.argtypes = [vp, vp, vp, ll, vp, vp, vp, ll, ci, vp, sz, vp]
        lib.zyfa_hadamard_quantize_qk_e4m3.restype = ci
        lib.zyfa_hadamard_quantize_e4m3_noalloc.argtypes = [vp, vp, vp, ll, ci, vp]
        lib.zyfa_hadamard_quantize_e4m3_noalloc.restype = ci
        lib.zyfa_hadamard_workspace_bytes.argtypes = [ll]
        lib.zyfa_hadamard_workspace_bytes.restype = sz
        lib.zyfa_check_errors.argtypes = [vp]
        lib.zyfa_check_errors.restype = ci
        lib.zyfa_status_string.argtypes = [ci]
        lib.zyfa_status_string.restype = ctypes.c_char_p
        lib.zyfa_kernel_launches.argtypes = [ci, ci, ci]
        lib.zyfa_kernel_launches.restype = ci
        lib.zyfa_probe_mma_rate.argtypes = [ci, ci, ci, vp, vp, vp]
        lib.zyfa_probe_mma_rate.restype = ci
        lib.zyfa_probe_mma_flops_per_iter.argtypes = [ci]
        lib.zyfa_probe_mma_flops_per_iter.restype = ll
        lib.zyfa_probe_mma_form_rate.argtypes = [ci, ci, ci, vp, vp, vp]
        lib.zyfa_probe_mma_form_rate.restype = ci
        lib.zyfa_probe_mma_form_flops_per_iter.argtypes = [ci]
        lib.zyfa_probe_mma_form_flops_per_iter.restype = ll
        _lib = lib
        return lib


def zyfa_attn_fwd_causal(q: int, k: int, v: int, out: int, B: int, S: int, H: int, H_kv: int, D_qk: int, D_v: int,
                         softmax_scale: float, dtype: int, q_descale: int = 0, k_descale: int = 0,
                         v_descale: int = 0, stream: int = 0) -> int:
    """Call the C entry point with raw addresses; returns the status code."""
    lib = load_library()
    return lib.zyfa_attn_fwd_causal(q, k, v, out, B, S, H, H_kv, D_qk, D_v, float(softmax_scale), dtype,
                                    q_descale or None, k_descale or None, v_descale or None, stream or None)


def zyfa_attn_fwd_causal_ex(q: int, k: int, v: int, out: int, B: int, S: int, H: int, H_kv: int, D_qk: int,
                            D_v: int, softmax_scale: float, dtype: int, q_descale: int = 0, k_descale: int = 0,
                            v_descale: int = 0, p_mode: int = ZYFA_P_LEAN, descale_per_kv_head: int = 0,
                            lse: int = 0, stream: int = 0) -> int:
    """Call the C entry point with options (raw addresses); returns the status code."""
    lib = load_library()
    opts = FwdOptions(p_mode, descale_per_kv_head, lse or None)
    return lib.zyfa_attn_fwd_causal_ex(q, k, v, out, B, S, H, H_kv, D_qk, D_v, float(softmax_scale), dtype,
                                       q_descale or None, k_descale or None, v_descale or None,
                                       ctypes.byref(opts), stream or None)


def zyfa_attn_fwd_causal_host(q_host: int, k_host: int, v_host: int, out_host: int, q_dev: int, k_dev: int,
                              v_dev: int, out_dev: int, B: int, S: int, H: int, H_kv: int, D_qk: int, D_v: int,
                              softmax_scale: float, dtype: int, q_descale: int = 0, k_descale: int = 0,
                              v_descale: int = 0, chunks: int = 0, stream: int = 0) -> int:
    """Call the host-buffer C entry point (transfers overlapped with compute); returns the status code."""
    return load_library().zyfa_attn_fwd_causal_host(q_host, k_host, v_host, out_host, q_dev, k_dev, v_dev, out_dev,
                                                    B, S, H, H_kv, D_qk, D_v, float(softmax_scale), dtype,
                                                    q_descale or None, k_descale or None, v_descale or None,
                                                    chunks, stream or None)


def zyfa_selftest_stalled_pipeline(q: int, k: int, v: int, out: int, B: int, S: int, H: int, H_kv: int, D_qk: int,
                                   D_v: int, dtype: int, stream: int = 0) -> int:
    """Enqueue the kernel with its loads withheld (tests of the timeout path); returns the status code."""
    return load_library().zyfa_selftest_stalled_pipeline(q, k, v, out, B, S, H, H_kv, D_qk, D_v, dtype,
                                                         stream or None)


def zyfa_check_errors(stream: int = 0) -> int:
    return load_library().zyfa_check_errors(stream or None)


def zyfa_kernel_launches(B: int, S: int, H: int) -> int:
    return load_library().zyfa_kernel_launches(B, S, H)


def _descale_ptr(t, per_head_numel):
    """(pointer, per_head) for a descale tensor: one float (per tensor) or per_head_numel floats
    ([batch][KV head], flash_attn_func's (batch, nheads_k) layout)."""
    if t is None:
        return 0, None
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.float32 and t.is_contiguous()):
        raise TypeError("descale must be a contiguous float32 CUDA tensor or None")
    if t.numel() == 1:
        return t.data_ptr(), False
    if t.numel() == per_head_numel:
        return t.data_ptr(), True
    raise ValueError(f"descale must hold 1 or batch*nheads_k = {per_head_numel} values, got {t.numel()}")


def flash_attn_func(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: float | None = None,
                    causal: bool = True, q_descale=None, k_descale=None, v_descale=None,
                    out: torch.Tensor | None = None, return_lse: bool = False, p_mode: str = "lean"):
    """Causal prefill attention on CUDA tensors q [B,S,H,D_qk], k [B,S,H_kv,D_qk], v [B,S,H_kv,D_v].

    FP8 inputs are ``torch.float8_e4m3fn`` (or ``torch.uint8`` holding e4m3 bit patterns) with optional
    descales: float32 CUDA tensors of one value (per tensor) or of B*H_kv values ([batch][KV head]); all
    three given descales must use the same form.  BF16 inputs are ``torch.bfloat16``.  ``p_mode`` picks
    how FP8 probabilities are produced ("lean": Lean P; "exact": exponential and e4m3 rounding;
    "exact-noblock": the same against the row's running reference, without per-block scaling).
    Returns a bfloat16 tensor [B,S,H,D_v], and with ``return_lse`` also the float32 log-sum-exp
    [B,H,S].  Runs on the current CUDA stream.
    """
    if not causal:
        raise NotImplementedError("only causal attention is implemented")
    if q.dtype in (torch.float8_e4m3fn, torch.uint8):
        dtype = ZYFA_DTYPE_E4M3
    elif q.dtype == torch.bfloat16:
        dtype = ZYFA_DTYPE_BF16
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, S, heads, D]")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous CUDA tensors")
    B, S, H, D_qk = q.shape
    _, _, H_kv, D_v = v.shape
    if k.shape != (B, S, H_kv, D_qk) or v.shape[:2] != (B, S):
        raise ValueError("inconsistent q/k/v shapes")
    if out is None:
        out = torch.empty((B, S, H, D_v), dtype=torch.bfloat16, device=q.device)
    elif out.shape != (B, S, H, D_v) or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 [B,S,H,D_v] tensor")
    if p_mode not in _P_MODES:
        raise ValueError("p_mode must be 'lean', 'exact' or 'exact-noblock'")
    descales = [_descale_ptr(t, B * H_kv) for t in (q_descale, k_descale, v_descale)]
    forms = {per for _, per in descales if per is not None}
    if len(forms) > 1:
        raise ValueError("descales must all be per tensor or all per (batch, KV head)")
    lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device) if return_lse else None
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = zyfa_attn_fwd_causal_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, H, H_kv, D_qk,
                                     D_v, 0.0 if softmax_scale is None else softmax_scale, dtype,
                                     descales[0][0], descales[1][0], descales[2][0],
                                     _P_MODES[p_mode],
                                     1 if forms == {True} else 0, lse.data_ptr() if lse is not None else 0, stream)
    if st != 0:
        raise ZyfaError(st, "zyfa_attn_fwd_causal_ex")
    return (out, lse) if return_lse else out


def zyfa_hadamard_quantize_e4m3(x: int, x8: int, descale: int, rows: int, D: int, workspace: int,
                                workspace_bytes: int, stream: int = 0) -> int:
    """Call the C pre-pass with raw addresses; returns the status code."""
    return load_library().zyfa_hadamard_quantize_e4m3(x or None, x8 or None, descale or None, rows, D,
                                                      workspace or None, workspace_bytes, stream or None)


def zyfa_hadamard_quantize_e4m3_noalloc(x: int, x8: int, descale: int, rows: int, D: int, stream: int = 0) -> int:
    """Call the allocation-free C pre-pass (scratch inside the library; calls must not overlap on the
    GPU); returns the status code."""
    return load_library().zyfa_hadamard_quantize_e4m3_noalloc(x or None, x8 or None, descale or None, rows, D,
                                                             stream or None)


def zyfa_hadamard_quantize_qk_e4m3(q: int, q8: int, q_descale: int, q_rows: int, k: int, k8: int, k_descale: int,
                                   k_rows: int, D: int, workspace: int, workspace_bytes: int, stream: int = 0) -> int:
    """Call the C pre-pass for Q and K together (one launch per pass) with raw addresses; returns the
    status code."""
    return load_library().zyfa_hadamard_quantize_qk_e4m3(q or None, q8 or None, q_descale or None, q_rows, k or None,
                                                         k8 or None, k_descale or None, k_rows, D, workspace or None,
                                                         workspace_bytes, stream or None)


def zyfa_hadamard_workspace_bytes(rows: int) -> int:
    return load_library().zyfa_hadamard_workspace_bytes(rows)


def hadamard_quantize_e4m3(x: torch.Tensor):
    """Rotate a bf16 CUDA tensor [..., D] by the block Hadamard matrix over its last axis and quantise
    it per tensor to e4m3.  Returns (codes as torch.float8_e4m3fn, same shape; descale, a 1-element
    float32 CUDA tensor).  Rotate Q and K (not V) and pass the codes and descales to flash_attn_func."""
    if x.dtype != torch.bfloat16 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous bfloat16 CUDA tensor")
    D = x.shape[-1]
    rows = x.numel() // D if D else 0
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    descale = torch.ones(1, dtype=torch.float32, device=x.device)
    ws = torch.empty(max(1, zyfa_hadamard_workspace_bytes(rows) // 4), dtype=torch.float32, device=x.device)
    stream = torch.cuda.current_stream(x.device).cuda_stream
    with torch.cuda.device(x.device):
        st = zyfa_hadamard_quantize_e4m3(x.data_ptr(), codes.data_ptr(), descale.data_ptr(), rows, D,
                                         ws.data_ptr(), ws.numel() * 4, stream)
    if st != 0:
        raise ZyfaError(st, "zyfa_hadamard_quantize_e4m3")
    return codes.view(torch.float8_e4m3fn), descale


def hadamard_quantize_qk_e4m3(q: torch.Tensor, k: torch.Tensor):
    """Rotate and quantise Q and K together (contiguous bf16 CUDA tensors with the same last dimension
    D): one launch per pass for both.  Returns (q codes, q descale, k codes, k descale) as
    hadamard_quantize_e4m3 does for each."""
    for t in (q, k):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise TypeError("q and k must be contiguous bfloat16 CUDA tensors")
    D = q.shape[-1]
    if k.shape[-1] != D or k.device != q.device:
        raise ValueError("q and k need the same head dimension and device")
    qr, kr = (q.numel() // D if D else 0), (k.numel() // D if D else 0)
    q8 = torch.empty(q.shape, dtype=torch.uint8, device=q.device)
    k8 = torch.empty(k.shape, dtype=torch.uint8, device=q.device)
    ds = torch.ones(2, dtype=torch.float32, device=q.device)
    nbytes = zyfa_hadamard_workspace_bytes(qr) + zyfa_hadamard_workspace_bytes(kr)
    ws = torch.empty(max(1, nbytes // 4), dtype=torch.float32, device=q.device)
    stream = torch.cuda.current_stream(q.device).cuda_stream
    with torch.cuda.device(q.device):
        st = zyfa_hadamard_quantize_qk_e4m3(q.data_ptr(), q8.data_ptr(), ds.data_ptr(), qr, k.data_ptr(),
                                            k8.data_ptr(), ds.data_ptr() + 4, kr, D, ws.data_ptr(), ws.numel() * 4,
                                            stream)
    if st != 0:
        raise ZyfaError(st, "zyfa_hadamard_quantize_qk_e4m3")
    return q8.view(torch.float8_e4m3fn), ds[0:1], k8.view(torch.float8_e4m3fn), ds[1:2]
