"""Pins for the NVFP4 quantisation oracle (CPU only).

The element tables are pinned to the OCP MX v1.0 encodings (tests/golden), the roundings to
CUDA's own host-side FP8/FP4 conversions and to torch's float8_e4m3fn cast, and the whole
quantiser to closed forms, exhaustive grids and a brute-force nearest-code search.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


@pytest.fixture(scope="module")
def cvt(tmp_path_factory):
    """CUDA's host conversions (cuda_fp8.h / cuda_fp4.h), compiled with g++ for the test."""
    out = tmp_path_factory.mktemp("cvt") / "libcvt.so"
    src = os.path.join(HERE, "helpers", "cuda_host_cvt.cpp")
    inc = os.environ.get("CUDA_HOME", "/usr/local/cuda") + "/include"
    if not os.path.exists(os.path.join(inc, "cuda_fp4.h")):
        pytest.skip("cuda_fp4.h not available")
    subprocess.run(["g++", "-O1", "-shared", "-fPIC", "-I", inc, "-o", str(out), src], check=True)
    lib = ctypes.CDLL(str(out))
    lib.host_cvt_e2m1_rn.argtypes = [ctypes.c_float]
    lib.host_cvt_e2m1_rn.restype = ctypes.c_uint8
    lib.host_cvt_e4m3_satfinite.argtypes = [ctypes.c_float]
    lib.host_cvt_e4m3_satfinite.restype = ctypes.c_uint8
    lib.host_cvt_e4m3_from_double_satfinite.argtypes = [ctypes.c_double]
    lib.host_cvt_e4m3_from_double_satfinite.restype = ctypes.c_uint8
    return lib


def test_golden_element_tables():
    path = os.path.join(HERE, "golden", "ocp_mx_element_tables.txt")
    n = 0
    for line in open(path):
        if not line.strip() or line.startswith("#"):
            continue
        fmt, code, val = line.split()
        code = int(code, 16)
        got = oracle.e2m1_decode(code) if fmt == "e2m1" else oracle.e4m3_decode(code)
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val) and np.signbit(got) == val.startswith("-")
        n += 1
    assert n == 21


def test_e4m3_round_matches_torch_cast():
    g = torch.Generator().manual_seed(0)
    x = torch.cat([torch.rand(20000, generator=g) * 448.0,
                   torch.exp2(torch.rand(20000, generator=g) * 18 - 10),  # 2^-10 .. 2^8
                   torch.rand(2000, generator=g) * 2 ** -8])
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_round(float(v)) for v in x])
    np.testing.assert_array_equal(got, ref)


def test_e4m3_round_matches_cuda_host_cvt(cvt):
    g = torch.Generator().manual_seed(1)
    x = torch.cat([torch.exp2(torch.rand(20000, generator=g, dtype=torch.float64) * 20 - 11),
                   torch.rand(2000, generator=g, dtype=torch.float64) * 600.0])
    for v in x.tolist():
        assert oracle.e4m3_round(v) == cvt.host_cvt_e4m3_from_double_satfinite(v), v


def test_e4m3_codes_midpoints_saturation():
    for c in range(0x7F):
        assert oracle.e4m3_round(oracle.e4m3_decode(c)) == c
    for c in range(0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_round(mid) == even
        assert oracle.e4m3_round(np.nextafter(mid, 0)) == c
        assert oracle.e4m3_round(np.nextafter(mid, np.inf)) == c + 1
    for v in (448.0, 463.99, 464.0, 480.0, 1e6, 1e300):
        assert oracle.e4m3_round(v) == 0x7E
    assert oracle.e4m3_round(2.0 ** -10) == 0x00          # half the least subnormal: tie to 0
    assert oracle.e4m3_round(2.0 ** -10 * 1.0001) == 0x01


def test_e2m1_grid_ties_saturation_sign():
    for c, v in enumerate(E2M1):
        assert oracle.e2m1_round(v) == c
        assert oracle.e2m1_round(-v) == (c | 8)
    ties = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6}
    for v, c in ties.items():
        assert oracle.e2m1_round(v) == c
        assert oracle.e2m1_round(-v) == c | 8
    for v in (6.0, 6.5, 7.0, 100.0, 1e30):
        assert oracle.e2m1_round(v) == 7
    assert oracle.e2m1_round(-0.1) == 0x8
    assert oracle.e2m1_round(0.2) == 0x0


def test_e2m1_round_matches_cuda_host_cvt(cvt):
    g = torch.Generator().manual_seed(2)
    xs = (torch.rand(30000, generator=g, dtype=torch.float64) * 16 - 8).tolist()
    xs += [m + d for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) for d in (-1e-7, 0.0, 1e-7)]
    for v in xs:
        f = float(np.float32(v))
        assert oracle.e2m1_round(f) == cvt.host_cvt_e2m1_rn(f), f


def test_quantize_zero_tensor():
    codes, scales, sg = oracle.nvfp4_quantize(np.zeros(64, np.float32))
    assert sg == 0.0 and not codes.any() and not scales.any()
    codes, scales, sg = oracle.nvfp4_quantize(-np.zeros(32, np.float32))
    assert sg == 0.0 and not codes.any() and not scales.any()


def test_quantize_tensor_scale_is_fp32_quotient():
    g = np.random.default_rng(3)
    for _ in range(200):
        x = (g.standard_normal(32) * 10.0 ** g.uniform(-3, 3)).astype(np.float32)
        _, _, sg = oracle.nvfp4_quantize(x)
        assert np.float32(sg) == np.float32(np.abs(x).max()) / np.float32(2688.0)


def test_quantize_exact_grid_and_nibble_order():
    """Values already on the grid x den (den = 1 when amax = 6*448 * s_g ...) come back exactly."""
    # one block whose amax is 6: s_g = 6/2688, block scale = 6/(6 s_g) = 448 (code 0x7E), den = 6/6 = 1
    x = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0, 0.0],
                 np.float32)
    codes, scales, sg = oracle.nvfp4_quantize(x)
    assert sg == np.float32(6.0) / np.float32(2688.0)
    assert scales[0] == 0x7E
    assert list(codes) == [0x10, 0x32, 0x54, 0x76, 0xA9, 0xCB, 0xED, 0x0F]
    deq = oracle.nvfp4_dequantize(codes, scales, sg)
    np.testing.assert_allclose(deq, x, rtol=2 ** -20)


def test_quantize_brute_force_nearest_code():
    """Every code is the nearest representable value given the block scale (ties: even code)."""
    g = np.random.default_rng(4)
    x = np.concatenate([g.standard_normal(16 * 64), g.standard_normal(16 * 8) * 1e-4,
                        g.uniform(-1, 1, 16 * 8) * 50]).astype(np.float32)
    codes, scales, sg = oracle.nvfp4_quantize(x)
    cvals = np.stack([codes & 0xF, codes >> 4], 1).reshape(-1)
    for blk in range(x.size // 16):
        xb = x[blk * 16:(blk + 1) * 16].astype(np.float64)
        den = oracle.e4m3_decode(int(scales[blk])) * sg
        # the block scale is the nearest E4M3 to amax_b / (6 s_g): no other code is closer
        target = np.abs(xb).max() / (6.0 * sg)
        errs = [abs(target - oracle.e4m3_decode(c)) for c in range(0x7F)]
        assert errs[scales[blk]] == min(errs)
        for i in range(16):
            c = int(cvals[blk * 16 + i])
            if den == 0:
                assert c == 0
                continue
            e = [abs(abs(xb[i]) - E2M1[m] * den) for m in range(8)]
            assert e[c & 7] == min(e)
            assert bool(c & 8) == bool(np.signbit(xb[i]))


def test_quantize_error_bound():
    g = np.random.default_rng(5)
    x = g.standard_normal(4096).astype(np.float32)
    codes, scales, sg = oracle.nvfp4_quantize(x)
    deq = oracle.nvfp4_dequantize(codes, scales, sg)
    for blk in range(x.size // 16):
        xb = x[blk * 16:(blk + 1) * 16]
        den = oracle.e4m3_decode(int(scales[blk])) * sg
        # within range every element is off by at most half a grid step (<= 1 den)
        assert np.all(np.abs(deq[blk * 16:(blk + 1) * 16] - xb) <= 1.0 * den + 1e-30)


def test_quantize_rejects_bad_length():
    with pytest.raises(ValueError):
        oracle.nvfp4_quantize(np.zeros(17, np.float32))
