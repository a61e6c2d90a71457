"""GPU parity of the decode (split-KV) path against the FP64 oracle, through the C ABI.

Small cases compare every output element; the full-size decode workloads compare sampled rows
(the oracle regenerates just the slices it needs) plus properties that hold at any size."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, oracle_rows, run_attention, split_boundary_units, stratified_rows, unit_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


def _full_case(F, B, Hq, Hkv, Sq, Skv, D, sigma=1.0, seed=11, seqlens=None, **kw):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "bf16", seed)
    q, k, v, _ = w.make("cuda")
    sl_t = None if seqlens is None else torch.tensor(seqlens, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, **kw)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale,
                                    seqlens_k=None if seqlens is None else np.array(seqlens, np.int32))
    return res, o_ref, l_ref


def test_single_head_fp32_out(F):
    """B1 H1 Sq1 Skv128 D64, N(0,1), scale 1/8, FP32 O + LSE (the single-head workload)."""
    w = inputs.workloads()[0]
    q, k, v, _ = w.make("cuda")
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    for ns in (1, 0):
        res = run_attention(F, q, k, v, w.scale, out_kind="f32", num_splits=ns)
        check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"splits={ns}")
        assert np.abs(res["o"] - o_ref).max() < 2e-3   # FP32 output: only P's BF16 rounding remains


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D", [
    (2, 4, 2, 1, 300, 128),     # 3 tiles, ragged tail of 44
    (1, 2, 2, 1, 1, 64),        # a single key
    (3, 2, 2, 4, 257, 64),      # Sq = 4 query rows per head, tail of 1
    (1, 16, 1, 1, 640, 128),    # G = 16: the whole MMA N
    (2, 8, 2, 2, 1000, 128),    # G = 8 (GQA 4 x Sq 2)
])
@pytest.mark.parametrize("mode", ["fwd", "whole", "split"])
def test_small_shapes(F, B, Hq, Hkv, Sq, Skv, D, mode):
    kw = {"fwd": {}, "whole": {"num_splits": 1}, "split": {"num_splits": 0}}[mode]
    res, o_ref, l_ref = _full_case(F, B, Hq, Hkv, Sq, Skv, D, **kw)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, mode)


def test_ragged_with_empty_and_nan_padding(F):
    """Ragged keys incl. 0, 1, tile edges; padding rows hold NaN and must never be read."""
    B, Hq, Hkv, Skv, D = 6, 8, 2, 700, 128
    sl = [0, 1, 128, 129, 700, 255]
    w = inputs.Workload("t", B, Hq, Hkv, 1, Skv, D, 1.0, "bf16", 21)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    kc, vc = k.cpu(), v.cpu()
    o_ref, l_ref = oracle.attention(q.cpu(), kc, vc, w.scale, seqlens_k=np.array(sl, np.int32))
    for ns in (0, 1):
        res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=ns)
        check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"splits={ns}")
        assert np.all(res["o"][: Hq] == 0.0) and np.all(np.isneginf(res["lse"][:Hq]))


def test_split_and_whole_agree(F):
    res1, o_ref, l_ref = _full_case(F, 4, 4, 4, 1, 3000, 128, num_splits=1, seed=5)
    res0, _, _ = _full_case(F, 4, 4, 4, 1, 3000, 128, num_splits=0, seed=5)
    check_o_lse(res0["o"], res0["lse"], o_ref, l_ref, "split")
    # number of splits is not part of the result: both within BF16 rounding of each other
    assert np.abs(res0["o"] - res1["o"]).max() <= 2 * 2 ** -8 * np.abs(o_ref).max() + 1e-6


def test_decode_full_size_every_row(F):
    """B8 H32 Sq1 Skv4096 D128 (split-KV, BF16 O + LSE): every one of the 256 query rows, one per
    (b, kv-head) unit, so every unit is checked: on 152 SMs 128 CTAs take two whole units each; on a
    device whose SM count gives no such divisor the units are split and every split boundary is."""
    w = inputs.workloads()[1]
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0)
    rows = np.arange(w.B * w.Hq * w.Sq, dtype=np.int64)
    o_ref, l_ref = oracle_rows(w, rows, tensors=(q, k, v))
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "decode full size, every row")
    assert np.abs(res["o"]).max() <= float(v.abs().max()) + 1e-3


def test_ragged_gqa_nvfp4_full_size(F):
    """B64 Hq32 Hkv8 Sq1 ragged Skv<=32768 D128 with NVFP4 output.  FP32 O against the oracle on
    one row of every (b, kv-head) unit plus every row of each unit that the stream-K split cuts
    across CTAs; NVFP4 codes/scales bit-exact against the oracle quantiser on the same FP32 O."""
    w = inputs.workloads()[4]
    q, k, v, sl = w.make("cuda", pad_fill=float("nan"))
    res = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=0, want_f32=True)
    lens = w.seqlens().astype(np.int64)
    tiles = [int((lens[u // w.Hkv] + 127) // 128) for u in range(w.B * w.Hkv)]
    cut = split_boundary_units(tiles, F.fmha_num_sms())
    assert len(cut) > 50, len(cut)
    rows = stratified_rows(w, all_units=True, edge_units=cut, tile=1, extra=16, seed=2)
    o_ref, l_ref = oracle_rows(w, rows, tensors=(q, k, v))
    check_o_lse(res["o"][rows], res["lse"][rows], o_ref, l_ref, "ragged nvfp4 (fp32 O)")
    codes, scales, sg = oracle.nvfp4_quantize(res["o"].reshape(-1))
    assert sg == res["tensor_scale"]
    np.testing.assert_array_equal(res["scales"], scales)
    np.testing.assert_array_equal(res["codes"], codes)
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n,kind", [(16, "ones"), (4096, "normal"), (262144, "normal"), (4096, "zeros"),
                                    (8192, "ties"), (1 << 20, "wide")])
def test_nvfp4_quantize_bit_exact(F, n, kind):
    g = torch.Generator().manual_seed(n)
    if kind == "ones":
        x = torch.ones(n)
    elif kind == "zeros":
        x = torch.zeros(n)
        x[::3] = -0.0
    elif kind == "ties":
        # amax = 42 makes s_g = 42/2688 = 2^-6 exact; a block whose max is 6 * 2^j then has the
        # scale 64 * 2^j (exact in E4M3) and den = 2^j, so these values sit exactly on midpoints
        base = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.1, -0.1, 4.0, 0.0, -6.0])
        first = torch.zeros(16)
        first[3] = 42.0
        x = torch.cat([first] + [base * 2.0 ** (i % 6 - 3) for i in range(1, n // 16)])
    elif kind == "wide":
        x = torch.randn(n, generator=g) * torch.exp2(torch.randint(-20, 10, (n,), generator=g).float())
    else:
        x = torch.randn(n, generator=g)
    xd = x.float().cuda()
    q = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
    sc = torch.zeros(F.nvfp4_scales_bytes(n), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # twice: the amax scratch must be re-zeroed by the call
        F.nvfp4_quantize(xd, q, sc)
        torch.cuda.synchronize()
        codes, scales, sg = oracle.nvfp4_quantize(x.numpy())
        scb = sc.cpu().numpy()
        off = (n // 16 + 15) // 16 * 16
        assert np.frombuffer(scb[off:off + 4].tobytes(), np.float32)[0] == np.float32(sg)
        np.testing.assert_array_equal(scb[: n // 16], scales)
        np.testing.assert_array_equal(q.cpu().numpy(), codes)


def test_bad_arguments_return_codes(F):
    q = torch.zeros(1, 1, 1, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    lib = F.load()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.fmha_fwd(P(q), P(q), P(q), P(out), None, 1, 3, 2, 1, 1, 64, 1.0, s) == F.FMHA_ERR_INVALID   # Hq % Hkv
    assert lib.fmha_fwd(P(q), P(q), P(q), P(out), None, 1, 1, 1, 1, 1, 96, 1.0, s) == F.FMHA_ERR_INVALID   # D
    opts = F.make_opts(F.FMHA_OUT_F32, num_splits=2)
    assert lib.fmha_fwd_ex(P(q), P(q), P(q), P(out), None, 1, 1, 1, 1, 1, 64, 1.0, s,
                           ctypes.byref(opts)) == F.FMHA_ERR_WORKSPACE
    assert F.fmha_check_status() == 0


@pytest.mark.parametrize("B,Hq,Hkv,Skv,D", [
    (1, 8, 1, 160000, 128),   # one unit over every CTA: up to one partial per SM, merged by the last arrival
    (1, 4, 1, 1000, 64),      # fewer key tiles than SMs: one CTA per tile (8 CTAs, 4 query columns)
    (3, 16, 2, 777, 128),     # several units, partial tail tiles
    (1, 1, 1, 5100, 64),      # one column, 40 tiles: 40 CTAs, one partial each, merged (more than four)
    (1, 16, 1, 5100, 128),    # 16 columns (epilogue warpgroup), 40 CTAs of one tile, 40 partials merged
])
def test_split_merge_in_kernel(F, B, Hq, Hkv, Skv, D):
    """Split-KV units are merged inside the decode kernel by the CTA that completes them."""
    w = inputs.Workload("t", B, Hq, Hkv, 1, Skv, D, 1.0, "bf16", 37)
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "in-kernel merge")


@pytest.mark.parametrize("B,Hq,Hkv,Skv,D", [
    (10, 15, 15, 300, 128),    # 150 units: one whole unit per CTA on 150 CTAs
    (20, 15, 15, 200, 64),     # 300 units: two whole units per CTA on 150 CTAs
    (2, 127, 127, 130, 128),   # 254 units: two per CTA on 127 CTAs (5/6 of 152), a one-key tail tile
    (16, 32, 8, 500, 128),     # 128 units of four query columns: the epilogue-warpgroup kernel
    (1, 157, 157, 400, 128),   # 157 units (prime, no divisor in range): the stream-K split stays
])
def test_whole_units_when_units_divide_evenly(F, B, Hq, Hkv, Skv, D):
    """With uniform lengths the split decode launches as many CTAs as divide the units evenly when that
    number lies between 5/6 of the SMs and all of them, and each CTA streams whole units (no partials,
    no merge).  The shapes are chosen for 152 SMs; on any device the result must match the oracle."""
    w = inputs.Workload("t", B, Hq, Hkv, 1, Skv, D, 1.0, "bf16", 38)
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "whole units")


def test_merge_counters_across_calls(F):
    """Arrival counters are tagged per call, not reset: repeated calls on one workspace (and a
    workspace first filled with arbitrary bytes) give identical results."""
    w = inputs.Workload("t", 4, 8, 2, 1, 5000, 128, 1.0, "bf16", 38)
    q, k, v, _ = w.make("cuda")
    B, Hq, Sq, D = q.shape
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0)
    wsb = F.fmha_workspace_size(B, Hq, w.Hkv, Sq, w.Skv, D, opts)
    ws = torch.randint(0, 256, (wsb,), dtype=torch.uint8, device="cuda")
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, ws)
    outs = []
    for _ in range(3):
        out = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
        F.fmha_fwd_ex(q, k, v, out, lse, w.scale, opts)
        outs.append(out.float().cpu().numpy())
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(outs[0].reshape(-1, D), None, o_ref, l_ref, "merge across calls")
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


@pytest.mark.parametrize("Hkv,Sq,causal", [(8, 4, True), (4, 1, False)])
def test_multi_column_split_merge_repeatable(F, Hkv, Sq, causal):
    """Several query columns per key/value head (16 = 4 heads x 4 causal tokens, and 8 heads x 1),
    split across CTAs and merged in the kernel: every column matches the oracle, and ten calls on one
    workspace give bit-identical O and LSE (the per-column sums, 1/L and the merged partials do not
    depend on which CTA arrives last)."""
    w = inputs.Workload("t", 2, 32, Hkv, Sq, 3000, 128, 1.0, "bf16", 52)
    q, k, v, _ = w.make("cuda")
    B, Hq, _, D = q.shape
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, None, None, None, None, causal)
    wsb = F.fmha_workspace_size(B, Hq, Hkv, Sq, w.Skv, D, opts)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, ws, None, None, None, causal)
    outs, lses = [], []
    for _ in range(10):
        out = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
        F.fmha_fwd_ex(q, k, v, out, lse, w.scale, opts)
        outs.append(out.float().cpu().numpy())
        lses.append(lse.cpu().numpy())
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=causal)
    check_o_lse(outs[0].reshape(-1, D), lses[0].reshape(-1), o_ref.reshape(-1, D), l_ref.reshape(-1),
                f"G={Hq // Hkv * Sq}")
    for o, l in zip(outs[1:], lses[1:]):
        np.testing.assert_array_equal(o, outs[0])
        np.testing.assert_array_equal(l, lses[0])
