"""CPU FP64 oracle for fused attention and NVFP4 quantisation (test infrastructure only).

Only the test suite, the smoke check and the benchmark's CPU-baseline / reference arm use this
package.  The CUDA library never imports, links or calls it, and the two share no code; the
only thing both sides see is the seeded inputs (``attention_tensor_cores_gb300.inputs``).

The arithmetic lives in plain C (``attn_ref.c``, ``nvfp4_ref.c``), built with gcc -O2 (no
fast-math) and OpenMP; this module only builds it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SOURCES = ("attn_ref.c", "nvfp4_ref.c")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so in place (gcc, -O2, OpenMP, no fast-math)."""
    srcs = [os.path.join(_HERE, s) for s in _SOURCES]
    hdr = os.path.join(_HERE, "oracle.h")
    if not force and os.path.exists(_LIB_PATH):
        newest = max(os.path.getmtime(p) for p in srcs + [hdr])
        if os.path.getmtime(_LIB_PATH) >= newest:
            return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            # ORACLE_LIB names a prebuilt library to load instead: the mutation tests point it at
            # copies of this oracle built with one planted mistake, which the pins must reject.
            path = os.environ.get("ORACLE_LIB")
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            P = ctypes.c_void_p
            I = ctypes.c_int
            I64 = ctypes.c_int64
            lib.oracle_attention_f64.argtypes = [P, P, P, I, I, I, I, I, I, ctypes.c_double,
                                                 P, I, P, I64, P, P]
            lib.oracle_attention_f64.restype = I
            lib.oracle_qk_f64.argtypes = [P, P, I, I, I, P]
            lib.oracle_qk_f64.restype = I
            lib.oracle_nvfp4_quantize.argtypes = [P, I64, P, P, P]
            lib.oracle_nvfp4_quantize.restype = I
            lib.oracle_nvfp4_quantize_scaled.argtypes = [P, I64, ctypes.c_float, P, P]
            lib.oracle_nvfp4_quantize_scaled.restype = I
            lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_decode.restype = ctypes.c_double
            lib.oracle_e4m3_round.argtypes = [ctypes.c_double]
            lib.oracle_e4m3_round.restype = ctypes.c_uint8
            lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_decode.restype = ctypes.c_double
            lib.oracle_e2m1_round.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_round.restype = ctypes.c_uint8
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(t) -> np.ndarray:
    """Accept a torch bfloat16 tensor or a uint16 numpy array of BF16 bit patterns."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


def attention(q, k, v, scale: float, seqlens_k=None, rows=None, causal: bool = False):
    """FP64 attention for query rows `rows` (flat (b*Hq+hq)*Sq+i; None = all).

    q: [B,Hq,Sq,D], k/v: [B,Hkv,Skv,D] BF16 (torch bf16 or uint16 bits).  causal: bottom-right
    aligned mask (query i of Sq sees keys j <= i + n - Sq).
    Returns (o [nrows, D] float64, lse [nrows] float64)."""
    lib = _load()
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, Dk = k.shape
    assert Dk == D and tuple(v.shape) == tuple(k.shape) and k.shape[0] == B
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    sl = None
    if seqlens_k is not None:
        sl = np.ascontiguousarray(np.asarray(seqlens_k, dtype=np.int32))
        assert sl.shape == (B,)
    rr = None
    nrows = B * Hq * Sq
    if rows is not None:
        rr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rr.shape[0]
    o = np.zeros((nrows, D), dtype=np.float64)
    lse = np.zeros((nrows,), dtype=np.float64)
    rc = lib.oracle_attention_f64(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Sq, Skv, D,
                                  float(scale), _ptr(sl), 1 if causal else 0, _ptr(rr), nrows, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attention_f64: bad arguments")
    return o, lse


def qk(q, k):
    """Raw FP64 S = Q K^T (no scale); q [Sq,D], k [Skv,D] BF16."""
    lib = _load()
    qb, kb = _bf16_bits(q), _bf16_bits(k)
    Sq, D = qb.shape
    Skv, Dk = kb.shape
    assert D == Dk
    s = np.zeros((Sq, Skv), dtype=np.float64)
    rc = lib.oracle_qk_f64(_ptr(qb), _ptr(kb), Sq, Skv, D, _ptr(s))
    if rc != 0:
        raise ValueError("oracle_qk_f64: bad arguments")
    return s


def nvfp4_quantize(x):
    """NVFP4 quantisation of an FP32 array (n % 16 == 0).

    Returns (codes uint8[n/2], scales uint8[n/16], tensor_scale float32)."""
    lib = _load()
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    n = xf.shape[0]
    codes = np.zeros(n // 2, dtype=np.uint8)
    scales = np.zeros(n // 16, dtype=np.uint8)
    sg = np.zeros(1, dtype=np.float32)
    rc = lib.oracle_nvfp4_quantize(_ptr(xf), n, _ptr(codes), _ptr(scales), _ptr(sg))
    if rc != 0:
        raise ValueError("oracle_nvfp4_quantize: bad arguments (n % 16 != 0?)")
    return codes, scales, float(sg[0])


def nvfp4_quantize_scaled(x, tensor_scale: float):
    """NVFP4 encoding of an FP32 array (n % 16 == 0) with a given per-tensor scale s_g.

    Returns (codes uint8[n/2], scales uint8[n/16])."""
    lib = _load()
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    xf = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    n = xf.shape[0]
    codes = np.zeros(n // 2, dtype=np.uint8)
    scales = np.zeros(n // 16, dtype=np.uint8)
    rc = lib.oracle_nvfp4_quantize_scaled(_ptr(xf), n, float(np.float32(tensor_scale)), _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle_nvfp4_quantize_scaled: bad arguments (n % 16 != 0?)")
    return codes, scales


def e4m3_decode(code: int) -> float:
    return _load().oracle_e4m3_decode(code)


def e4m3_round(v: float) -> int:
    return _load().oracle_e4m3_round(v)


def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(code)


def e2m1_round(v: float) -> int:
    return _load().oracle_e2m1_round(v)


def num_threads() -> int:
    return _load().oracle_num_threads()


def nvfp4_dequantize(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """Values represented by an NVFP4 encoding (FP64); used by tests for error bounds."""
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=1).reshape(-1)
    mag = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])[c & 7]
    val = np.where(c & 8, -mag, mag)
    sc = np.array([e4m3_decode(int(s)) for s in range(256)])[scales]
    return val * np.repeat(sc, 16) * float(tensor_scale)
