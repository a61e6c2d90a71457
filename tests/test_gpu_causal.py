"""GPU parity of the bottom-right aligned causal mask (query s of Sq sees keys 0 .. s + n - Sq) on
every kernel path, against the FP64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, oracle_rows, run_attention, sample_rows

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
    (1, 1, 1, 513, 513, 128, 1.0),    # D = 128 (P over S) with a 1-row last tile
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


def test_causal_prefill_full_size_sampled(F):
    """B4 H16 Sq=Skv=8192 D64 causal, BF16 O: 64 sampled rows against the oracle."""
    w = inputs.workloads()[2]
    q, k, v, _ = w.make("cuda")
    res = run_attention(F, q, k, v, w.scale, num_splits=0, causal=True)
    rows = sample_rows(w, 64, seed=5)
    o_ref, l_ref = oracle_rows(w, rows, causal=True)
    check_o_lse(res["o"][rows], res["lse"][rows], o_ref, l_ref, "causal prefill full size")
