"""The allocation-free decode entry point, through the C ABI.

fmha_fwd_decode_noalloc serves callers that cannot give the library a workspace (plug-ins and
bindings that only see tensor pointers, loops that may not call cudaMalloc): its split-KV scratch
is a fixed array inside the library.  Two calls in a row, with different shapes, must match the
FP64 oracle and the workspace-based entry point (fmha_fwd_ex) within the parity tolerances, and a
problem too large for the fixed array must be refused with FMHA_ERR_WORKSPACE.

Named to be collected last, so a run that stops at the first failure has run every other test."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, oracle_rows, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


def _noalloc(F, q, k, v, scale, seqlens=None):
    B, Hq, Sq, D = q.shape
    out = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    F.fmha_fwd_decode_noalloc(q, k, v, out, lse, scale, seqlens)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    return out.float().cpu().numpy().reshape(-1, D), lse.cpu().numpy().reshape(-1)


def test_two_calls_match_workspace_entry_point_and_oracle(F):
    """Two calls in a row on the shared scratch, each checked element by element against the FP64
    oracle and against the workspace-based entry point, within the parity tolerances."""
    # call 1: the decode workload (B8 H32 Sq1 Skv4096 D128), every row
    w = inputs.workloads()[1]
    q, k, v, _ = w.make("cuda")
    o1, l1 = _noalloc(F, q, k, v, w.scale)
    o_ref, l_ref = oracle_rows(w, np.arange(w.B * w.Hq * w.Sq), tensors=(q, k, v))
    check_o_lse(o1, l1, o_ref, l_ref, "noalloc call 1 vs oracle")
    ref = run_attention(F, q, k, v, w.scale, num_splits=0)
    check_o_lse(o1, l1, ref["o"].astype(np.float64), ref["lse"].astype(np.float64), "noalloc call 1 vs fmha_fwd_ex")
    del q, k, v
    # call 2: another shape on the same scratch (GQA, Sq = 2, ragged keys including an empty set)
    w2 = inputs.Workload("t", 5, 8, 2, 2, 900, 64, 1.0, "bf16", 31)
    q, k, v, _ = w2.make("cuda")
    lens = [0, 1, 900, 129, 513]
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    o2, l2 = _noalloc(F, q, k, v, w2.scale, sl)
    o_ref2, l_ref2 = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w2.scale, seqlens_k=np.array(lens, np.int32))
    check_o_lse(o2, l2, o_ref2, l_ref2, "noalloc call 2 vs oracle")
    ref2 = run_attention(F, q, k, v, w2.scale, seqlens=sl, num_splits=0)
    check_o_lse(o2, l2, ref2["o"].astype(np.float64), ref2["lse"].astype(np.float64), "noalloc call 2 vs fmha_fwd_ex")
    assert np.all(o2[:16] == 0.0) and np.all(np.isneginf(l2[:16]))


def test_too_large_is_refused(F):
    # 64 x 128 key/value heads need far more split scratch than the fixed array holds
    B, H, D = 64, 128, 128
    q = torch.zeros(B, H, 1, D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, H, 1, D, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    lib = F.load()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.fmha_fwd_decode_noalloc(P(q), P(k), P(k), P(out), None, B, H, H, 1, 1, D, 1.0, None,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == F.FMHA_ERR_WORKSPACE
    assert b"static area holds" in lib.fmha_last_error()
    assert F.fmha_check_status() == 0


def _noalloc_cases(n=16, seed=616):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 4, 8, 16]))
        Sq = int(rng.choice([1, 2, 4]))
        if g * Sq > 16:
            continue
        cases.append((int(rng.integers(1, 9)), Hkv * g, Hkv, Sq, int(rng.integers(1, 5000)), D,
                      bool(rng.random() < 0.5), int(rng.integers(1, 1 << 30))))
    return cases


NOALLOC_CASES = _noalloc_cases()


@pytest.mark.parametrize("case", NOALLOC_CASES, ids=[f"n{i}" for i in range(len(NOALLOC_CASES))])
def test_noalloc_random_shapes(F, case):
    """A seeded sweep of decode shapes (up to 16 query rows per key/value head, ragged lengths with
    empty sequences) through the allocation-free entry point, against the oracle."""
    B, Hq, Hkv, Sq, Skv, D, ragged, seed = case
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", seed)
    q, k, v, _ = w.make("cuda")
    lens = np.random.default_rng(seed).integers(0, Skv + 1, B).astype(np.int32) if ragged else None
    sl = None if lens is None else torch.from_numpy(lens).cuda()
    o, l = _noalloc(F, q, k, v, w.scale, sl)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, seqlens_k=lens)
    check_o_lse(o, l, o_ref, l_ref, f"noalloc {case}")
