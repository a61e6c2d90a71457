"""The GPU parity checker (``attn_util.check_o_lse``) must tell a right result from a wrong one.

CPU only, with the FP64 oracle on both sides: the "wrong" output is the oracle's answer to a
slightly different problem, standing for a plausible kernel mistake (a dropped key or key tile, a
causal diagonal off by one, the wrong key/value head, split partials merged without their LSE weights),
on shapes the GPU parity tests use.  Each must fail the check, while the right answer rounded to
BF16 (what the kernels store) must pass it.  Dropping a single key of thousands changes O and LSE
by about 1/n, below the tolerance, so single-key mistakes are asserted on the small multi-tile
shapes (where the GPU tests compare every element) and whole-tile mistakes at full size."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse


def _bf16(o):
    return torch.from_numpy(o).to(torch.bfloat16).double().numpy()


def _rejected(o, lse, o_ref, lse_ref):
    try:
        check_o_lse(o, lse, o_ref, lse_ref, "planted")
    except AssertionError:
        return True
    return False


@pytest.fixture(scope="module")
def small():
    """A small multi-tile shape with a ragged tail: B2 Hq8 Hkv2 Sq5 Skv300 D64."""
    w = inputs.Workload("tol", 2, 8, 2, 5, 300, 64, 1.0, "bf16", 4242)
    q, k, v, _ = w.make("cpu")
    return w, q, k, v


def test_right_answer_in_bf16_passes(small):
    w, q, k, v = small
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, w.scale, causal=causal)
        check_o_lse(_bf16(o), lse.astype(np.float32), o, lse, "bf16-rounded oracle")


def test_dropped_last_key_is_rejected(small):
    w, q, k, v = small
    o, lse = oracle.attention(q, k, v, w.scale)
    o2, lse2 = oracle.attention(q, k, v, w.scale, seqlens_k=np.full(w.B, w.Skv - 1, np.int32))
    assert _rejected(_bf16(o2), lse2, o, lse)


def test_dropped_ragged_tail_is_rejected(small):
    """The 44 keys past the last whole 128-key tile (300 = 2 * 128 + 44)."""
    w, q, k, v = small
    o, lse = oracle.attention(q, k, v, w.scale)
    o2, lse2 = oracle.attention(q, k, v, w.scale, seqlens_k=np.full(w.B, 256, np.int32))
    assert _rejected(_bf16(o2), lse2, o, lse)


def test_causal_diagonal_off_by_one_is_rejected(small):
    """Each query seeing one key fewer than the bottom-right mask allows: the causal problem with
    the last key removed, for the same queries."""
    w, q, k, v = small
    o, lse = oracle.attention(q, k, v, w.scale, causal=True)
    o2, lse2 = oracle.attention(q, k[:, :, :-1].contiguous(), v[:, :, :-1].contiguous(), w.scale, causal=True)
    # the shorter problem aligns its mask to 299 keys: query i sees keys 0 .. i + 299 - Sq
    assert _rejected(_bf16(o2), lse2, o, lse)


def test_wrong_kv_head_is_rejected(small):
    """Query head hq served by key/value head hq % Hkv instead of hq // (Hq/Hkv)."""
    w, q, k, v = small
    o, lse = oracle.attention(q, k, v, w.scale)
    g = w.Hq // w.Hkv
    idx = [hq % w.Hkv for hq in range(w.Hq)]
    kr, vr = k[:, idx].contiguous(), v[:, idx].contiguous()   # one key/value head per query head
    o2, lse2 = oracle.attention(q, kr, vr, w.scale)
    assert g > 1
    assert _rejected(_bf16(o2), lse2, o, lse)


def test_partials_merged_with_equal_weights_are_rejected(small):
    """Two key-range partials merged with equal weights instead of their LSE weights (a split-KV
    merge that forgets the rescale): O = (O1 + O2) / 2, LSE = max(LSE1, LSE2) + ln 2."""
    w, q, k, v = small
    o, lse = oracle.attention(q, k, v, w.scale)
    h = 128
    o1, l1 = oracle.attention(q, k[:, :, :h].contiguous(), v[:, :, :h].contiguous(), w.scale)
    o2, l2 = oracle.attention(q, k[:, :, h:].contiguous(), v[:, :, h:].contiguous(), w.scale)
    assert _rejected(_bf16((o1 + o2) / 2.0), np.maximum(l1, l2) + np.log(2.0), o, lse)


def test_full_size_decode_dropped_tile_is_rejected():
    """Single-token decode B8 H32 Skv4096 D128, 64 sampled rows: the last 128-key tile dropped."""
    w = inputs.workloads()[1]
    q, k, v, _ = w.make("cpu")
    rows = np.random.default_rng(5).choice(w.B * w.Hq * w.Sq, 64, replace=False).astype(np.int64)
    o, lse = oracle.attention(q, k, v, w.scale, rows=rows)
    check_o_lse(_bf16(o), lse.astype(np.float32), o, lse, "bf16-rounded oracle")
    o2, lse2 = oracle.attention(q, k, v, w.scale, rows=rows, seqlens_k=np.full(w.B, w.Skv - 128, np.int32))
    assert _rejected(_bf16(o2), lse2, o, lse)
