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
