"""CPU checks of the C ABI: the library builds and loads without a GPU, exports every function
include/fmha.h declares, and rejects bad arguments before touching a device."""
import ctypes

import pytest

import attention_tensor_cores_gb300 as F
from attention_tensor_cores_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return F.load()


def test_exports_every_declared_function(lib):
    names = F.header_functions()
    assert "fmha_fwd" in names and "nvfp4_quantize" in names and len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n


def test_error_strings(lib):
    for code in range(7):
        assert lib.fmha_error_string(code).decode().startswith("FMHA_")
    assert b"unknown" in lib.fmha_error_string(99)


def test_null_pointers_rejected_without_device(lib):
    assert lib.fmha_qk_gemm(None, None, None, 1, 128, 64, None) == F.FMHA_ERR_INVALID
    assert b"NULL" in lib.fmha_last_error()
    fake = ctypes.c_void_p(0x1000)
    assert lib.fmha_qk_gemm(fake, fake, fake, 1, 128, 48, None) == F.FMHA_ERR_INVALID
    assert lib.fmha_qk_gemm(ctypes.c_void_p(0x1008), fake, fake, 1, 128, 64, None) == F.FMHA_ERR_INVALID


def test_non_positive_or_non_finite_scale_rejected_without_device(lib):
    fake = ctypes.c_void_p(0x1000)
    for sc in (0.0, -0.125, float("nan"), float("inf")):
        assert lib.fmha_fwd(fake, fake, fake, fake, None, 1, 1, 1, 1, 16, 64, sc, None) == F.FMHA_ERR_INVALID
        assert b"scale" in lib.fmha_last_error()
        assert lib.fmha_fwd_decode_noalloc(fake, fake, fake, fake, None, 1, 1, 1, 1, 16, 64, sc, None, None) == F.FMHA_ERR_INVALID


def test_host_entry_rejects_before_device(lib):
    """fmha_fwd_host checks its pointers, options and device buffer before it touches a device."""
    fake = ctypes.c_void_p(0x1000)
    size = lib.fmha_host_buffer_size(2, 8, 2, 1, 256, 64, None)
    args = (2, 8, 2, 1, 256, 64, 0.125, None)
    assert lib.fmha_fwd_host(None, fake, fake, fake, None, *args, None, fake, size) == F.FMHA_ERR_INVALID
    seq = F.fmha_opts()
    seq.seqlens_k = 0x2000
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *args, ctypes.byref(seq), fake, size) == F.FMHA_ERR_UNSUPPORTED
    nv = F.fmha_opts()
    nv.out_kind = F.FMHA_OUT_NVFP4
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *args, ctypes.byref(nv), fake, size) == F.FMHA_ERR_UNSUPPORTED
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *args, None, None, size) == F.FMHA_ERR_WORKSPACE
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *args, None, ctypes.c_void_p(0x1040), size) == F.FMHA_ERR_WORKSPACE
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *args, None, fake, size - 1) == F.FMHA_ERR_WORKSPACE
    bad = (2, 8, 2, 1, 256, 64, float("nan"), None)
    assert lib.fmha_fwd_host(fake, fake, fake, fake, None, *bad, None, fake, size) == F.FMHA_ERR_INVALID
    assert lib.fmha_host_buffer_size(2, 8, 3, 1, 256, 64, None) == 0


def test_host_buffer_size_holds_the_staged_tensors(lib):
    """The device buffer holds Q, K, V, O and the LSE (each rounded up to 256 bytes) and the
    workspace of the largest batch chunk (up to four chunks of whole batch entries)."""
    def al(x):
        return (x + 255) // 256 * 256
    B, Hq, Hkv, Sq, Skv, D = 8, 32, 8, 1, 1000, 128
    for kind, esz in ((F.FMHA_OUT_BF16, 2), (F.FMHA_OUT_F32, 4)):
        o = F.fmha_opts()
        o.out_kind = kind
        staged = al(B * Hq * Sq * D * 2) + 2 * al(B * Hkv * Skv * D * 2) + al(B * Hq * Sq * D * esz) + al(B * Hq * Sq * 4)
        ws = lib.fmha_workspace_size(2, Hq, Hkv, Sq, Skv, D, ctypes.byref(o))
        assert ws > 0   # automatic split-KV for the decode shape
        assert lib.fmha_host_buffer_size(B, Hq, Hkv, Sq, Skv, D, ctypes.byref(o)) == staged + al(ws)
