"""Single-pass NVFP4 output (a given per-tensor scale s_g, encoded in the attention epilogues with
no amax pass and no FP32 staging), on every kernel path, against the oracle's encoding with the
same s_g of the same FP32 O (the NVFP4 step of the kernel plan in
"NVFP4-1.1_RAW_CUDA_CPP_APPROACH.md", item 7, with the scale supplied instead of measured)."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


CASES = [
    # B, Hq, Hkv, Sq, Skv, D, sigma, ragged, num_splits, causal
    (4, 8, 2, 1, 1500, 128, 1.0, True, 0, False),     # decode path, split-KV: codes from the combine
    (2, 8, 2, 1, 700, 64, 1.0, False, 1, False),      # decode path, whole units: codes from the epilogue
    (2, 2, 2, 300, 700, 64, 1.0, False, 0, False),    # row-tile path, fixed order
    (3, 4, 2, 300, 700, 64, 1.0, True, 0, False),     # row-tile path, ragged (counter order)
    (1, 2, 2, 520, 520, 128, 1.0, False, 0, True),    # row-tile path, causal, D = 128
    (2, 16, 1, 1, 300, 512, 0.5, False, 0, False),    # wide-head path, whole units
    (1, 32, 1, 1, 4000, 512, 0.5, False, 0, False),   # wide-head path, split over pairs (combine)
]


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,sigma,ragged,ns,causal", CASES)
@pytest.mark.parametrize("factor", [1.0, 0.2])
def test_single_pass_matches_oracle(F, B, Hq, Hkv, Sq, Skv, D, sigma, ragged, ns, causal, factor):
    """s_g = factor * max|O| / 2688: factor 1 is the two-pass scale, 0.2 saturates the largest
    blocks.  Codes and scales bit-exact against the oracle on the kernel's own FP32 O."""
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "nvfp4", 91, ragged=ragged)
    q, k, v, sl = w.make("cuda")
    ref = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=ns, want_f32=True, causal=causal)
    sg = float(np.float32(ref["tensor_scale"] * factor))
    a = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=ns, want_f32=True, causal=causal,
                      nvfp4_scale=sg, want_amax=True)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=None if sl is None else sl.cpu().numpy(),
                                    causal=causal)
    check_o_lse(a["o"], a["lse"], o_ref, l_ref, "single-pass fp32 O")
    codes, scales = oracle.nvfp4_quantize_scaled(a["o"].reshape(-1), sg)
    np.testing.assert_array_equal(a["scales"], scales)
    np.testing.assert_array_equal(a["codes"], codes)
    assert a["tensor_scale"] == sg
    assert a["amax"] == float(np.abs(a["o"]).max())
    if factor == 1.0:   # the same FP32 O and the same s_g as the two-pass run: the same encoding
        np.testing.assert_array_equal(a["codes"], ref["codes"])
        np.testing.assert_array_equal(a["scales"], ref["scales"])
    # without the FP32 copy: same encoding, and no NVFP4 workspace beyond the path's own
    b = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=ns, causal=causal, nvfp4_scale=sg)
    np.testing.assert_array_equal(b["codes"], a["codes"])
    np.testing.assert_array_equal(b["scales"], a["scales"])


@pytest.mark.parametrize("sg", [0.0, -1.0, float("nan"), float("inf")])
def test_unusable_scale_gives_zero_encoding(F, sg):
    w = inputs.Workload("t", 2, 8, 2, 1, 700, 128, 1.0, "nvfp4", 92)
    q, k, v, _ = w.make("cuda")
    a = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", num_splits=0, nvfp4_scale=sg)
    assert not a["codes"].any() and not a["scales"].any()


@pytest.mark.parametrize("log2_sg", [-100, -30, 0, 40, 110])
def test_standalone_scaled_quantiser(F, log2_sg):
    """nvfp4_quantize_scaled, including scales outside [2^-90, 2^100] (the FP64 route), against the
    oracle; values scaled with s_g so that blocks fit, saturate and underflow."""
    rng = np.random.default_rng(log2_sg + 200)
    n = 16 * 4096
    mag = np.repeat(2.0 ** rng.uniform(-12, 12, n // 16), 16)
    x = (rng.standard_normal(n) * mag * 2.0 ** log2_sg * 2688 / 4096).astype(np.float32)
    sg = float(np.float32(2.0 ** log2_sg * 1.37))
    xt = torch.from_numpy(x).cuda()
    q = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(n // 16, dtype=torch.uint8, device="cuda")
    F.nvfp4_quantize_scaled(xt, q, sc, torch.tensor([sg], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    np.testing.assert_array_equal(sc.cpu().numpy(), scales)
    np.testing.assert_array_equal(q.cpu().numpy(), codes)
    assert (scales == 0x7E).any() and (scales == 0).any() and ((scales > 0) & (scales < 0x7E)).any()


def test_standalone_scaled_quantiser_ties(F):
    """Elements planted exactly on E2M1 and E4M3 rounding midpoints (ties to the even code)."""
    sg = 2.0 ** -7 * 1.5
    rows = []
    for sc_val in (0.25, 1.0, 13.0, 448.0):                     # block scales to plant around
        den = sc_val * sg
        blk = np.array([m * den for m in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)] + [6 * den], np.float64)
        blk = np.concatenate([blk, -blk]).astype(np.float32)
        assert np.all(blk.astype(np.float64) == np.concatenate([blk[:8], -blk[:8]]))
        rows.append(blk)
    for mid in (13.5, 432.0, 1.5 * 2.0 ** -9, 0.5 * (0.25 + 0.28125)):   # E4M3 midpoints: scale ties
        top = 6 * sg * mid
        blk = np.array([top, -top / 3, top / 7, 0.0] + [top * (i + 1) / 17 for i in range(12)], np.float64)
        assert float(np.float32(top)) == top
        rows.append(blk.astype(np.float32))
    x = np.concatenate(rows * 64).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    n = x.size
    q = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(n // 16, dtype=torch.uint8, device="cuda")
    F.nvfp4_quantize_scaled(xt, q, sc, torch.tensor([sg], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    np.testing.assert_array_equal(sc.cpu().numpy(), scales)
    np.testing.assert_array_equal(q.cpu().numpy(), codes)


def _e4m3_value(c):
    e, m = c >> 3, c & 7
    return m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)


@pytest.mark.parametrize("sg", [2.0 ** -7 * 1.5, float(np.float32(1.37 * 2.0 ** -20)), float(np.float32(0.911 * 2.0 ** 33))])
def test_standalone_block_scale_every_boundary(F, sg):
    """Every E4M3 rounding boundary of the block scale: a block whose max |x| is the float nearest
    to 6 s_g times the midpoint between codes c - 1 and c, and the floats one unit below and above
    it, for c = 1..126 (ties fall to the even code when the product is exact)."""
    blocks = []
    for c in range(1, 127):
        t = 6.0 * 0.5 * (_e4m3_value(c - 1) + _e4m3_value(c)) * sg     # exact in FP64
        f = np.float32(t)
        for top in (np.nextafter(f, np.float32(0)), f, np.nextafter(f, np.float32(np.inf))):
            blk = np.full(16, top, np.float32) * np.float32(0.5) ** np.arange(16, dtype=np.float32)
            blk[1::2] *= -1
            blocks.append(blk)
    x = np.concatenate(blocks).astype(np.float32)
    xt = torch.from_numpy(x).cuda()
    n = x.size
    q = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(n // 16, dtype=torch.uint8, device="cuda")
    F.nvfp4_quantize_scaled(xt, q, sc, torch.tensor([sg], dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    codes, scales = oracle.nvfp4_quantize_scaled(x, sg)
    np.testing.assert_array_equal(sc.cpu().numpy(), scales)
    np.testing.assert_array_equal(q.cpu().numpy(), codes)
    assert len(set(scales.tolist())) >= 120


def test_two_pass_reports_amax(F):
    """Two-pass NVFP4 with opts.out_amax: the caller's word is the |O| max the quantiser uses, so it
    equals max |O| of the FP32 output and s_g = fp32(amax / 2688)."""
    w = inputs.Workload("t", 2, 4, 4, 160, 520, 64, 1.0, "nvfp4", 93)
    q, k, v, _ = w.make("cuda")
    a = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", num_splits=0, want_f32=True, want_amax=True)
    amax = float(np.abs(a["o"]).max())
    assert a["amax"] == amax
    assert a["tensor_scale"] == float(np.float32(np.float64(np.float32(amax)) / 2688.0))
    codes, scales, sg = oracle.nvfp4_quantize(a["o"].reshape(-1))
    np.testing.assert_array_equal(a["codes"], codes)
    np.testing.assert_array_equal(a["scales"], scales)
