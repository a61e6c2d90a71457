"""Failure detection on the GPU without faulting it: with the bounded-wait limit set to one cycle,
the first wait of each kernel that is not already satisfied expires.  The kernel must then stop
issuing copies and MMAs, drain what is in flight, free its Tensor Memory and return; the host
must see FMHA_ERR_TIMEOUT from fmha_check_status, and the context must stay usable (the same call
with the default limit is correct afterwards)."""
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


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,sigma,wv", [
    (2, 8, 8, 1, 2048, 128, 1.0, 0),   # decode path (split-KV)
    (1, 2, 2, 512, 1024, 64, 1.0, 0),  # row-tile path
    (1, 32, 1, 1, 512, 512, 0.5, 1),   # wide-head path, independent CTAs
    (1, 32, 1, 1, 512, 512, 0.5, 2),   # wide-head path, CTA pairs (cluster: both CTAs must drain and meet)
])
def test_forced_timeout_is_reported_and_context_survives(F, B, Hq, Hkv, Sq, Skv, D, sigma, wv):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "bf16", 61)
    q, k, v, _ = w.make("cuda")
    out = torch.empty(B, Hq, Sq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, wide_variant=wv)
    wsb = F.fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, opts)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    opts = F.make_opts(F.FMHA_OUT_BF16, None, 0, ws, wide_variant=wv)
    assert F.fmha_check_status() == F.FMHA_OK
    F.fmha_set_wait_limit(1)
    try:
        F.fmha_fwd_ex(q, k, v, out, lse, w.scale, opts)
        rc = F.fmha_check_status()
    finally:
        F.fmha_set_wait_limit(0)
    assert rc == F.FMHA_ERR_TIMEOUT
    assert F.fmha_check_status() == F.FMHA_OK          # the status word was cleared
    res = run_attention(F, q, k, v, w.scale, num_splits=0, wide_variant=wv if D == 512 else None)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "after timeout")
