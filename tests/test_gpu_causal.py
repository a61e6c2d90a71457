"""GPU parity of the bottom-right aligned causal mask (query s of Sq sees keys 0 .. s + n - Sq) on
every kernel path, against the FP64 oracle, through the C ABI."""
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


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,sigma", [
    (2, 8, 2, 4, 300, 128, 1.0),      # decode path: 4 heads x 4 new tokens = 16 columns
    (1, 2, 2, 8, 5, 64, 1.0),         # decode path, Sq > Skv: the first 3 queries see no key
    (1, 2, 2, 1000, 1000, 64, 1.0),   # row-tile path, square causal
    (1, 1, 1, 300, 700, 64, 1.0),     # row-tile path, Sq < Skv (bottom-right)
    (1, 2, 1, 700, 300, 64, 1.0),     # row-tile path, Sq > Skv: 400 queries see no key
    (1, 8, 2, 64, 500, 128, 1.0),     # row-tile path, GQA: head blocks of 64 rows interleave
    (1, 1, 1, 513, 513, 128, 1.0),    # D = 128 (shared S, query tiles with different key-tile counts), 1-row last tile
    (1, 2, 2, 700, 300, 128, 1.0),    # D = 128, Sq > Skv: whole query tiles see no key (no QK in the shared-S order)
    (2, 16, 1, 3, 100, 512, 0.5),     # wide-head path, 3 tokens per head
])
def test_causal(F, B, Hq, Hkv, Sq, Skv, D, sigma):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "bf16", 81)
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0, causal=True)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=True)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "causal")


def test_causal_ragged_nan_padding(F):
    B, H, Sq, Skv, D = 3, 2, 200, 600, 64
    sl = [150, 1, 600]
    w = inputs.Workload("t", B, H, H, Sq, Skv, D, 1.0, "bf16", 82)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=0, causal=True)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=np.array(sl, np.int32), causal=True)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "causal ragged")


def test_causal_prefill_full_size_stratified(F):
    """B4 H16 Sq=Skv=8192 D64 causal, BF16 O: one row of every unit, the first and last row of every
    128-row query tile of six seeded units (the diagonal tiles included), and random rows."""
    w = inputs.workloads()[2]
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0, causal=True)
    edge = np.random.default_rng(5).choice(w.B * w.Hkv, 6, replace=False)
    rows = stratified_rows(w, all_units=True, edge_units=edge, tile=128, extra=32, seed=5)
    o_ref, l_ref = oracle_rows(w, rows, causal=True, tensors=(q, k, v))
    check_o_lse(res["o"][rows], res["lse"][rows], o_ref, l_ref, "causal prefill full size")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,seq", [
    (1, 2, 2, 1000, 1000, 64, None),      # causal, fixed item order (no workspace counter)
    (1, 8, 2, 64, 500, 128, None),
    (3, 2, 2, 200, 600, 64, [150, 1, 600]),
])
def test_causal_fixed_order(F, B, Hq, Hkv, Sq, Skv, D, seq):
    """num_splits = 1: the row-tile kernel walks its items in the fixed strided order instead of
    claiming them from the workspace counter; results must not depend on the order."""
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 83)
    q, k, v, _ = w.make("cuda")
    sl_t = None if seq is None else torch.tensor(seq, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=1, causal=True)
    sl = None if seq is None else np.array(seq, np.int32)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=sl, causal=True)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "causal fixed order")


@pytest.mark.parametrize("D", [64, 128])
def test_ragged_prefill_balanced_order_many_units(F, D):
    """Ragged non-causal prefill with the workspace counter: 48 units of very different lengths,
    192 items for at most 152 CTAs, so CTAs claim several items of unequal size (at D = 128 the two
    query tiles of every item also take the shared S buffer in turns, across items)."""
    B, H, Sq, Skv = 6, 8, 800, 1500
    sl = [1500, 3, 700, 1, 1280, 129]
    w = inputs.Workload("t", B, H, H, Sq, Skv, D, 1.0, "bf16", 84)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=0)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=np.array(sl, np.int32))
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, f"ragged prefill, counter order, D={D}")


def test_causal_workspace_reuse_back_to_back(F):
    """The work-item counter is reset on the stream before each launch: two causal calls in a row
    on one workspace give the same (correct) result."""
    w = inputs.Workload("t", 2, 4, 4, 600, 600, 64, 1.0, "bf16", 85)
    q, k, v, _ = w.make("cuda")
    B, Hq, Sq, D = q.shape
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, None, None, None, None, True)
    wsb = F.fmha_workspace_size(B, Hq, w.Hkv, Sq, w.Skv, D, opts)
    assert wsb >= 4
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, ws, None, None, None, True)
    outs = []
    for _ in range(2):
        out = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
        F.fmha_fwd_ex(q, k, v, out, lse, w.scale, opts)
        outs.append((out.float().cpu().numpy().reshape(-1, D), lse.cpu().numpy().reshape(-1)))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=True)
    for o, l in outs:
        check_o_lse(o, l, o_ref, l_ref, "causal back to back")
    np.testing.assert_array_equal(outs[0][0], outs[1][0])


@pytest.mark.parametrize("num_splits", [0, 1])
def test_chunked_prefill_ragged_causal_d128(F, num_splits):
    """Chunked prefill over a ragged KV cache at D = 128: 300 new queries per sequence against
    ragged key counts, some shorter than the query chunk (their first queries see no key), NaN in the
    padding; counter order (workspace) and fixed order."""
    B, H, Sq, Skv, D = 4, 2, 300, 1000, 128
    sl = [1000, 120, 301, 777]
    w = inputs.Workload("t", B, H, H, Sq, Skv, D, 1.0, "bf16", 86)
    q, k, v, _ = w.make("cuda")
    for b, n in enumerate(sl):
        k[b, :, n:] = float("nan")
        v[b, :, n:] = float("nan")
    sl_t = torch.tensor(sl, dtype=torch.int32, device="cuda")
    res = run_attention(F, q, k, v, w.scale, seqlens=sl_t, num_splits=num_splits, causal=True)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=np.array(sl, np.int32), causal=True)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "chunked prefill")


def test_speculative_decode_full_size_every_row(F):
    """B8 Hq32 Hkv8 Sq4 Skv8192 D128, causal (16 query columns per key/value head): every one of the
    1024 rows against the oracle.  64 units for 152 or so CTAs: the stream-K split gives each CTA
    about 27 of the 4096 key tiles, so units are cut into two or three parts and many CTAs end one
    unit and start the next (their first epilogue runs on the epilogue warps while the next unit
    streams); the CTA that completes a unit merges it."""
    w = inputs.Workload("speculative decode", 8, 32, 8, 4, 8192, 128, 1.0, "bf16", 1006)
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0, causal=True)
    rows = np.arange(w.B * w.Hq * w.Sq, dtype=np.int64)
    o_ref, l_ref = oracle_rows(w, rows, causal=True, tensors=(q, k, v))
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "speculative decode full size")
