"""GB300 (sm_103a) fused multi-head attention: Python binding of libfmha.so.

Thin ctypes marshalling only: every step of attention, split-KV combine and NVFP4 quantisation
runs in the library's CUDA kernels.  torch tensors supply device memory and the current stream.
There is no CPU path: if libfmha.so is missing or cannot load, every call raises.

Function names match the C ABI in include/fmha.h.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfmha.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "fmha.h")

FMHA_OK = 0
FMHA_ERR_INVALID = 1
FMHA_ERR_UNSUPPORTED = 2
FMHA_ERR_WORKSPACE = 3
FMHA_ERR_CUDA = 4
FMHA_ERR_TIMEOUT = 5
FMHA_ERR_RACE = 6
FMHA_OUT_BF16 = 0
FMHA_OUT_F32 = 1
FMHA_OUT_NVFP4 = 2
FMHA_WIDE_AUTO = 0
FMHA_WIDE_INDEPENDENT = 1
FMHA_WIDE_PAIR = 2

_lock = threading.Lock()
_lib = None


class FmhaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


class fmha_opts(ctypes.Structure):
    _fields_ = [
        ("out_kind", ctypes.c_int),
        ("seqlens_k", ctypes.c_void_p),
        ("num_splits", ctypes.c_int),
        ("workspace", ctypes.c_void_p),
        ("workspace_bytes", ctypes.c_size_t),
        ("out_scales", ctypes.c_void_p),
        ("out_tensor_scale", ctypes.c_void_p),
        ("out_f32", ctypes.c_void_p),
        ("causal", ctypes.c_int),
        ("nvfp4_scale_in", ctypes.c_void_p),
        ("out_amax", ctypes.c_void_p),
        ("wide_variant", ctypes.c_int),
    ]


def header_functions() -> list[str]:
    """Names of the functions include/fmha.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(fmha_\w+|nvfp4_\w+)\s*\(", txt)) - {"fmha_fwd_ex_"})


def load(path: str | None = None):
    """Load libfmha.so (built by build.py / __graft_entry__.build()); raises if absent."""
    global _lib
    lib = _lib
    if lib is not None:
        return lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FmhaError(FMHA_ERR_CUDA, f"{p} not built: run attention_tensor_cores_gb300/build.py")
        lib = ctypes.CDLL(p)
        V, I, I64, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
        sig = {
            "fmha_fwd": ([V, V, V, V, V, I, I, I, I, I, I, F, V], I),
            "fmha_fwd_ex": ([V, V, V, V, V, I, I, I, I, I, I, F, V, ctypes.POINTER(fmha_opts)], I),
            "fmha_workspace_size": ([I, I, I, I, I, I, ctypes.POINTER(fmha_opts)], S),
            "fmha_fwd_host": ([V, V, V, V, V, I, I, I, I, I, I, F, V, ctypes.POINTER(fmha_opts), V, S], I),
            "fmha_host_buffer_size": ([I, I, I, I, I, I, ctypes.POINTER(fmha_opts)], S),
            "nvfp4_quantize": ([V, V, V, I64, V], I),
            "nvfp4_quantize_scaled": ([V, V, V, I64, V, V], I),
            "nvfp4_scales_bytes": ([I64], S),
            "fmha_qk_gemm": ([V, V, V, I, I, I, V], I),
            "fmha_selftest": ([I, V, V, S, I, V], I),
            "fmha_check_status": ([V], I),
            "fmha_set_wait_limit": ([ctypes.c_longlong], None),
            "fmha_error_string": ([I], ctypes.c_char_p),
            "fmha_last_error": ([], ctypes.c_char_p),
            "fmha_num_sms": ([], I),
            "fmha_launch_count": ([], ctypes.c_longlong),
            "fmha_time_next_call": ([V, V], None),
            "fmha_fwd_decode_noalloc": ([V, V, V, V, V, I, I, I, I, I, I, F, V, V], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name, None)
            if fn is None:
                continue
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def _check(rc: int, what: str):
    if rc != FMHA_OK:
        lib = load()
        raise FmhaError(rc, f"{what}: {lib.fmha_last_error().decode()} ({lib.fmha_error_string(rc).decode()})")


def _stream(stream=None):
    """Raw cudaStream_t of `stream`, else of the current stream on the current device."""
    import torch
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise FmhaError(FMHA_ERR_INVALID, "tensors must be on a CUDA device")
        if t is not None and not t.is_contiguous():
            raise FmhaError(FMHA_ERR_INVALID, "tensors must be contiguous")


# ------------------------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ------------------------------------------------------------------------------------------------
def fmha_fwd(q, k, v, out, lse, scale: float, stream=None):
    """O = softmax(scale Q K^T) V with BF16 output; q [B,Hq,Sq,D], k/v [B,Hkv,Skv,D]."""
    _need_cuda(q, k, v, out, lse)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    rc = load().fmha_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                         float(scale), _stream(stream))
    _check(rc, "fmha_fwd")


def make_opts(out_kind=FMHA_OUT_BF16, seqlens_k=None, num_splits=0, workspace=None,
              out_scales=None, out_tensor_scale=None, out_f32=None, causal=False,
              nvfp4_scale_in=None, out_amax=None, wide_variant=FMHA_WIDE_AUTO) -> fmha_opts:
    o = fmha_opts()
    o.wide_variant = wide_variant
    o.causal = 1 if causal else 0
    o.nvfp4_scale_in = None if nvfp4_scale_in is None else nvfp4_scale_in.data_ptr()
    o.out_amax = None if out_amax is None else out_amax.data_ptr()
    o.out_kind = out_kind
    o.seqlens_k = None if seqlens_k is None else seqlens_k.data_ptr()
    o.num_splits = num_splits
    o.workspace = None if workspace is None else workspace.data_ptr()
    o.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    o.out_scales = None if out_scales is None else out_scales.data_ptr()
    o.out_tensor_scale = None if out_tensor_scale is None else out_tensor_scale.data_ptr()
    o.out_f32 = None if out_f32 is None else out_f32.data_ptr()
    return o


def fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, opts: fmha_opts | None = None) -> int:
    return int(load().fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D,
                                          None if opts is None else ctypes.byref(opts)))


def fmha_fwd_ex(q, k, v, out, lse, scale: float, opts: fmha_opts | None = None, stream=None):
    """Attention with options (see make_opts); tensors as in fmha_fwd, `out` per opts.out_kind."""
    _need_cuda(q, k, v, out, lse)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    rc = load().fmha_fwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                            float(scale), _stream(stream), None if opts is None else ctypes.byref(opts))
    _check(rc, "fmha_fwd_ex")


def fmha_host_buffer_size(B, Hq, Hkv, Sq, Skv, D, opts: fmha_opts | None = None) -> int:
    return int(load().fmha_host_buffer_size(B, Hq, Hkv, Sq, Skv, D, None if opts is None else ctypes.byref(opts)))


def fmha_fwd_host(q, k, v, out, lse, scale: float, dev_buf, opts: fmha_opts | None = None, stream=None):
    """Attention from host memory: q/k/v/out/lse are CPU tensors (page-locked for asynchronous copies,
    lse may be None), dev_buf a CUDA byte tensor of at least fmha_host_buffer_size() bytes.  Returns
    once enqueued on `stream`; synchronise before reading out / lse."""
    for t in (q, k, v, out, lse):
        if t is not None and (t.is_cuda or not t.is_contiguous()):
            raise FmhaError(FMHA_ERR_INVALID, "q/k/v/out/lse must be contiguous host tensors")
    _need_cuda(dev_buf)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    rc = load().fmha_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D, float(scale),
                              _stream(stream), None if opts is None else ctypes.byref(opts), _ptr(dev_buf),
                              dev_buf.numel() * dev_buf.element_size())
    _check(rc, "fmha_fwd_host")


def nvfp4_scales_bytes(n: int) -> int:
    return int(load().nvfp4_scales_bytes(n))


def nvfp4_quantize(x, q, scales, stream=None):
    """x: FP32 [n] (n % 16 == 0), q: uint8 [n/2], scales: uint8 [nvfp4_scales_bytes(n)]."""
    _need_cuda(x, q, scales)
    rc = load().nvfp4_quantize(_ptr(x), _ptr(q), _ptr(scales), x.numel(), _stream(stream))
    _check(rc, "nvfp4_quantize")


def nvfp4_quantize_scaled(x, q, scales, tensor_scale, stream=None):
    """x: FP32 [n] (n % 16 == 0), q: uint8 [n/2], scales: uint8 [n/16], tensor_scale: FP32 [1] (s_g)."""
    _need_cuda(x, q, scales, tensor_scale)
    rc = load().nvfp4_quantize_scaled(_ptr(x), _ptr(q), _ptr(scales), x.numel(), _ptr(tensor_scale), _stream(stream))
    _check(rc, "nvfp4_quantize_scaled")


def fmha_qk_gemm(q, k, s, stream=None):
    """Raw S = Q K^T (FP32, no scale); q [Sq,D], k [Skv,D] BF16, s [Sq,Skv] FP32."""
    _need_cuda(q, k, s)
    Sq, D = q.shape
    Skv = k.shape[0]
    rc = load().fmha_qk_gemm(_ptr(q), _ptr(k), _ptr(s), Sq, Skv, D, _stream(stream))
    _check(rc, "fmha_qk_gemm")


def fmha_selftest(which: int, inp, out, param: int = 0, stream=None):
    _need_cuda(inp, out)
    rc = load().fmha_selftest(which, _ptr(inp), _ptr(out), out.numel() * out.element_size(), param,
                              _stream(stream))
    _check(rc, f"fmha_selftest({which})")


def fmha_check_status(stream=None) -> int:
    return int(load().fmha_check_status(_stream(stream)))


def fmha_set_wait_limit(cycles: int):
    load().fmha_set_wait_limit(int(cycles))


def fmha_num_sms() -> int:
    return int(load().fmha_num_sms())


def fmha_launch_count() -> int:
    return int(load().fmha_launch_count())


def fmha_time_next_call(start_event, stop_event):
    """torch.cuda.Event pair (enable_timing=True, already recorded once so the handle exists)."""
    load().fmha_time_next_call(ctypes.c_void_p(start_event.cuda_event), ctypes.c_void_p(stop_event.cuda_event))


def fmha_fwd_decode_noalloc(q, k, v, out, lse, scale: float, seqlens_k=None, stream=None):
    """Split-KV decode whose scratch is the library's fixed device array (nothing is allocated)."""
    _need_cuda(q, k, v, out, lse, seqlens_k)
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    rc = load().fmha_fwd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, Sq, Skv, D,
                                        float(scale), _ptr(seqlens_k), _stream(stream))
    _check(rc, "fmha_fwd_decode_noalloc")
