"""GPU parity of the wide-head (D = 512) path against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, oracle_rows, run_attention, stratified_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv", [
    (2, 128, 1, 1, 300),     # 128 heads on one key/value head, 10 key tiles with a tail of 12
    (1, 8, 1, 1, 1000),      # 8 query rows: rows 8..127 of the MMA tile are padding
    (1, 64, 1, 3, 200),      # 192 rows per key/value head: two 128-row blocks
    (3, 16, 2, 1, 33),       # GQA 8, two key tiles, the second with one key
])
@pytest.mark.parametrize("mode", ["fwd", "bf16", "f32", "f32_whole"])
@pytest.mark.parametrize("variant", ["auto", "independent", "pair"])
def test_shapes(F, B, Hq, Hkv, Sq, Skv, mode, variant):
    """fwd: fmha_fwd without options (whole units per CTA pair, no workspace); bf16/f32: split over
    every SM pair with a workspace; f32_whole: whole units with FP32 output.  variant: the kernel
    (automatic, independent CTAs, or the CTA-pair MMA)."""
    if mode == "fwd" and variant != "auto":
        pytest.skip("fmha_fwd has no options")
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, 512, 0.5, "bf16", 51)
    q, k, v, _ = w.make("cuda")
    kw = {"fwd": {}, "bf16": {"num_splits": 0}, "f32": {"out_kind": "f32", "num_splits": 0},
          "f32_whole": {"out_kind": "f32", "num_splits": 1}}[mode]
    if variant != "auto":
        kw["wide_variant"] = {"independent": F.FMHA_WIDE_INDEPENDENT, "pair": F.FMHA_WIDE_PAIR}[variant]
    res = run_attention(F, q, k, v, w.scale, **kw)
    if mode in ("fwd", "f32_whole"):
        assert res.get("workspace_bytes", 0) == 0
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, mode)


def test_ragged_nan_padding_and_empty(F):
    B, Hq, Hkv, Skv = 4, 16, 2, 500
    sl = [0, 1, 33, 500]
    w = inputs.Workload("t", B, Hq, Hkv, 1, Skv, 512, 0.5, "bf16", 52)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=np.array(sl, np.int32))
    for ns in (0, 1):   # split with a workspace, and whole units (no workspace; the empty unit too)
        res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=ns)
        check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"ragged wide, num_splits={ns}")
        assert np.all(res["o"][:Hq] == 0.0) and np.all(np.isneginf(res["lse"][:Hq]))


@pytest.mark.parametrize("variant", ["pair", "independent"])
def test_nvfp4_output_bit_exact(F, variant):
    w = inputs.Workload("t", 2, 32, 1, 1, 700, 512, 0.5, "bf16", 53)
    q, k, v, _ = w.make("cuda")
    wv = {"independent": F.FMHA_WIDE_INDEPENDENT, "pair": F.FMHA_WIDE_PAIR}[variant]
    res = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", num_splits=0, want_f32=True, wide_variant=wv)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "wide nvfp4 fp32 O")
    codes, scales, sg = oracle.nvfp4_quantize(res["o"].reshape(-1))
    assert sg == res["tensor_scale"]
    np.testing.assert_array_equal(res["scales"], scales)
    np.testing.assert_array_equal(res["codes"], codes)


@pytest.mark.parametrize("mode", ["split", "split_pair", "fwd"])
def test_wide_full_size_stratified(F, mode):
    """B32 Hq128 Hkv1 Sq1 Skv16384 D512, N(0, 0.5), BF16 O + LSE: the first and last row of every
    unit (each unit is one 128-row tile, cut by the stream-K split into about two pieces) and random
    rows.  split: fmha_fwd_ex with a workspace (the default, independent CTAs); split_pair: the same
    on the CTA-pair MMA kernel; fwd: fmha_fwd (whole units, no workspace)."""
    w = inputs.workloads()[3]
    q, k, v, _ = w.make("cuda")
    kw = {"split": {"num_splits": 0}, "fwd": {},
          "split_pair": {"num_splits": 0, "wide_variant": F.FMHA_WIDE_PAIR}}[mode]
    res = run_attention(F, q, k, v, w.scale, **kw)
    rows = stratified_rows(w, all_units=True, edge_units=range(w.B * w.Hkv), tile=128, extra=32, seed=4)
    o_ref, l_ref = oracle_rows(w, rows, tensors=(q, k, v))
    check_o_lse(res["o"][rows], res["lse"][rows], o_ref, l_ref, f"wide full size ({mode})")
    assert np.all(np.isfinite(res["o"])) and np.all(np.isfinite(res["lse"]))
    del q, k, v
    torch.cuda.empty_cache()


@pytest.mark.parametrize("variant", ["pair", "independent"])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,splits", [
    (2, 16, 1, 3, 300, 0),      # 3 causal tokens per head, split over pairs
    (1, 64, 1, 2, 1000, 1),     # 2 tokens per head, whole units
    (3, 128, 1, 1, 129, 0),     # a tile with one key past 128
])
def test_variants_causal_and_tails(F, variant, B, Hq, Hkv, Sq, Skv, splits):
    """Both D = 512 kernels under the bottom-right causal mask and with partial last key tiles."""
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, 512, 0.5, "bf16", 54)
    q, k, v, _ = w.make("cuda")
    wv = {"independent": F.FMHA_WIDE_INDEPENDENT, "pair": F.FMHA_WIDE_PAIR}[variant]
    res = run_attention(F, q, k, v, w.scale, num_splits=splits, causal=True, wide_variant=wv)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=True)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"{variant} causal")


def test_pair_variant_with_ragged_keys_runs_independent(F):
    """Asking for the pair MMA with ragged keys is served by the independent CTAs (their ring clears
    the NaN padding), and the result is still correct."""
    B, Hq, Hkv, Skv = 3, 16, 1, 400
    sl = [1, 250, 400]
    w = inputs.Workload("t", B, Hq, Hkv, 1, Skv, 512, 0.5, "bf16", 55)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=0, wide_variant=F.FMHA_WIDE_PAIR)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=np.array(sl, np.int32))
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "pair requested, ragged")
