"""GPU check of the closed form "softmax rows sum to 1" on every kernel path, through the C ABI.

With a constant value matrix V = c the exact output is O = c for every query that sees at least one
key, whatever the scores.  The GPU's O may differ from c only by the BF16 rounding of P before the
PV product (relative 2^-9 per weight) and of O itself: |O - c| <= |c| * 2^-7.  The oracle (which
gives c to FP64 rounding) supplies the LSE, compared with the usual tolerance."""
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


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,sigma,causal,splits", [
    (3, 8, 8, 1, 5000, 128, 2.0, False, 0),     # decode, split over every SM, merged in the kernel
    (3, 8, 8, 1, 5000, 128, 2.0, False, 1),     # decode, whole units
    (2, 32, 2, 1, 3000, 64, 2.0, False, 0),     # decode, 16 query columns per key/value head
    (2, 8, 2, 4, 2000, 128, 2.0, True, 0),      # multi-token decode, causal
    (1, 2, 2, 700, 900, 64, 2.0, False, None),  # row-tile D = 64, fmha_fwd
    (1, 2, 1, 600, 600, 64, 2.0, True, 0),      # row-tile D = 64, causal, counter order
    (1, 2, 2, 513, 700, 128, 2.0, False, None), # row-tile D = 128, shared S buffer
    (2, 128, 1, 1, 3000, 512, 0.5, False, 0),   # wide head, split over CTA pairs + combine
    (2, 128, 1, 1, 3000, 512, 0.5, False, None),  # wide head, fmha_fwd (whole units)
])
@pytest.mark.parametrize("c", [1.0, -2.5])
def test_constant_values_give_constant_output(F, B, Hq, Hkv, Sq, Skv, D, sigma, causal, splits, c):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "bf16", 91)
    q, k, _, _ = w.make("cuda")
    v = torch.full(k.shape, c, dtype=torch.bfloat16, device="cuda")
    kw = {} if splits is None else {"num_splits": splits}
    if causal:
        kw["causal"] = True
    res = run_attention(F, q, k, v, w.scale, **kw)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=causal)
    assert np.all(np.isfinite(l_ref))
    np.testing.assert_allclose(o_ref, c, rtol=Skv * 2.0 ** -52, atol=0)
    assert np.abs(res["o"] - c).max() <= abs(c) * 2.0 ** -7, np.abs(res["o"] - c).max()
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "constant V")
