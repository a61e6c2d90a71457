"""NVFP4 output through the workspace staging path (no out_f32 buffer from the caller), on each
kernel path: codes, block scales and tensor scale must be bit-identical to the run that also
returns its FP32 O, whose quantisation is checked against the oracle elsewhere."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,sigma,ragged", [
    (4, 8, 2, 1, 1500, 128, 1.0, True),     # decode path, ragged, split
    (2, 2, 2, 300, 700, 64, 1.0, False),    # row-tile path, fixed item order
    (3, 4, 2, 300, 700, 64, 1.0, True),     # row-tile path, ragged: counter order, staging after the counter
    (2, 16, 1, 1, 300, 512, 0.5, False),    # wide-head path
])
def test_staging_path_matches_fp32_path(F, B, Hq, Hkv, Sq, Skv, D, sigma, ragged):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, sigma, "nvfp4", 71, ragged=ragged)
    q, k, v, sl = w.make("cuda")
    a = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=0, want_f32=True)
    b = run_attention(F, q, k, v, w.scale, out_kind="nvfp4", seqlens=sl, num_splits=0, want_f32=False)
    np.testing.assert_array_equal(a["codes"], b["codes"])
    np.testing.assert_array_equal(a["scales"], b["scales"])
    assert a["tensor_scale"] == b["tensor_scale"]
    codes, scales, sg = oracle.nvfp4_quantize(a["o"].reshape(-1))
    np.testing.assert_array_equal(b["codes"], codes)
    np.testing.assert_array_equal(b["scales"], scales)
    assert sg == b["tensor_scale"]
