"""A seeded sweep of 600 random shapes across the dispatch: head dimension (64, 128, 512), grouping,
query rows per head, key length, bottom-right causal mask, ragged key lengths (including empty
sequences), output kind (BF16, FP32, NVFP4), split mode (no options, automatic split, whole units)
and the D = 512 kernel variant, plus 120 (and 20 single-pass) with up to 40,000 keys.  Each case
against the FP64 oracle; for NVFP4 the FP32 output against the oracle and the codes and scales
bit-exact against the oracle's quantiser on that output.  The shapes are drawn once from a fixed
seed, so the sweep is the same on every run."""
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


def _cases(n=600, seed=2024, skv_max=2500, cap=3e8):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128, 512], p=[0.4, 0.4, 0.2]))
        Hkv = int(rng.choice([1, 2, 4]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 8, 16]))
        Sq = int(rng.choice([1, 1, 2, 4, 16, 33, 130, 300]))
        Skv = int(rng.integers(1, skv_max))
        B = int(rng.integers(1, 4))
        causal = bool(rng.random() < 0.4)
        ragged = bool(rng.random() < 0.4)
        kind = str(rng.choice(["bf16", "f32", "nvfp4"], p=[0.45, 0.35, 0.2]))
        splits = [None, 0, 1][int(rng.integers(0, 3))]
        variant = int(rng.integers(0, 3))           # D = 512: automatic, independent, CTA pair
        case_seed = int(rng.integers(1, 1 << 30))
        if B * Hq * Sq * Skv * D > cap:             # keep the oracle within seconds
            continue
        if splits is None and (kind != "bf16" or ragged or causal):
            splits = 0                              # fmha_fwd takes no options
        cases.append((B, Hq, Hkv, Sq, Skv, D, causal, ragged, kind, splits, variant, case_seed))
    return cases


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_random_shape_against_oracle(F, case):
    B, Hq, Hkv, Sq, Skv, D, causal, ragged, kind, splits, variant, seed = case
    w = inputs.Workload("sweep", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", seed)
    q, k, v, _ = w.make("cuda")
    lens = None
    sl_t = None
    if ragged:
        lens = np.random.default_rng(seed).integers(0, Skv + 1, B).astype(np.int32)
        sl_t = torch.from_numpy(lens).cuda()
    kw = {}
    if D == 512:
        kw["wide_variant"] = [None, F.FMHA_WIDE_INDEPENDENT, F.FMHA_WIDE_PAIR][variant]
    res = run_attention(F, q, k, v, w.scale, out_kind=kind, seqlens=sl_t, num_splits=splits,
                        want_f32=(kind == "nvfp4"), causal=causal, **kw)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=lens, causal=causal)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"sweep {case}")
    if kind == "nvfp4":
        codes, scales, _ = oracle.nvfp4_quantize(res["o"].reshape(-1))
        np.testing.assert_array_equal(res["codes"], codes)
        np.testing.assert_array_equal(res["scales"][: scales.size], scales)


# longer key sets (up to 40,000 keys, ten times the work per shape): long split units, deep merges
BIG_CASES = _cases(n=120, seed=880001, skv_max=40000, cap=3e9)
BIG_SP_CASES = _cases(n=20, seed=880002, skv_max=40000, cap=3e9)


@pytest.mark.parametrize("case", BIG_CASES, ids=[f"b{i}" for i in range(len(BIG_CASES))])
def test_random_long_shape_against_oracle(F, case):
    test_random_shape_against_oracle(F, case)


SP_CASES = _cases(n=80, seed=9090)


@pytest.mark.parametrize("case", SP_CASES, ids=[f"s{i}" for i in range(len(SP_CASES))])
def test_random_shape_single_pass_nvfp4(F, case):
    """Single-pass NVFP4 (a given per-tensor scale s_g, encoded in the epilogues or the combine) on
    random shapes: s_g between 0.1 and 2 times the two-pass scale, so some blocks saturate and
    others do not.  Codes and scales bit-exact against the oracle's encoding with that s_g of the
    kernel's own FP32 O, and that O against the oracle."""
    B, Hq, Hkv, Sq, Skv, D, causal, ragged, _, splits, variant, seed = case
    w = inputs.Workload("sweep", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", seed)
    q, k, v, _ = w.make("cuda")
    lens = np.random.default_rng(seed).integers(0, Skv + 1, B).astype(np.int32) if ragged else None
    sl_t = None if lens is None else torch.from_numpy(lens).cuda()
    ns = 0 if splits is None else splits
    kw = {}
    if D == 512:
        kw["wide_variant"] = [None, F.FMHA_WIDE_INDEPENDENT, F.FMHA_WIDE_PAIR][variant]
    two = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl_t, num_splits=ns, causal=causal, **kw)
    factor = float(np.random.default_rng(seed + 1).uniform(0.1, 2.0))
    sg = float(np.float32(two["tensor_scale"] * factor))
    if not sg > 0.0:
        sg = 1.0 / 2688.0   # an all-zero output (every row empty): any usable scale
    a = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl_t, num_splits=ns, want_f32=True,
                      causal=causal, nvfp4_scale=sg, **kw)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=lens, causal=causal)
    check_o_lse(a["o"], a["lse"], o_ref, l_ref, f"single-pass sweep {case}")
    codes, scales = oracle.nvfp4_quantize_scaled(a["o"].reshape(-1), sg)
    np.testing.assert_array_equal(a["scales"], scales)
    np.testing.assert_array_equal(a["codes"], codes)


@pytest.mark.parametrize("case", BIG_SP_CASES, ids=[f"bs{i}" for i in range(len(BIG_SP_CASES))])
def test_random_long_shape_single_pass_nvfp4(F, case):
    test_random_shape_single_pass_nvfp4(F, case)
