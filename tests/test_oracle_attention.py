"""Pins for the FP64 attention oracle (CPU only).

Each test checks the oracle against something other than itself: a library routine the
definition reduces to (torch's FP64 scaled-dot-product attention and logsumexp), closed forms,
invariants, or an arbitrary-precision brute force on tiny shapes.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from attention_tensor_cores_gb300 import inputs


def _bf16(shape, seed, sigma=1.0):
    g = torch.Generator("cpu").manual_seed(seed)
    return (torch.randn(*shape, generator=g) * sigma).to(torch.bfloat16)


def _sdpa64(q, k, v, scale):
    return F.scaled_dot_product_attention(q.double(), k.double(), v.double(), scale=scale)


def _lse64(q, k, scale):
    return torch.logsumexp(scale * (q.double() @ k.double().transpose(-1, -2)), dim=-1)


@pytest.mark.parametrize("B,H,Sq,Skv,D", [(1, 1, 1, 1, 8), (2, 3, 5, 37, 16), (1, 2, 3, 130, 64),
                                          (1, 1, 2, 300, 128)])
def test_matches_library_sdpa(B, H, Sq, Skv, D):
    q, k, v = _bf16((B, H, Sq, D), 1), _bf16((B, H, Skv, D), 2), _bf16((B, H, Skv, D), 3)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.attention(q, k, v, scale)
    ref = _sdpa64(q, k, v, scale).reshape(-1, D).numpy()
    np.testing.assert_allclose(o, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, _lse64(q, k, scale).reshape(-1).numpy(), rtol=1e-13, atol=1e-13)


def test_gqa_equals_repeated_heads():
    """Consecutive query heads share one key/value head: hq -> hq // (Hq/Hkv)."""
    B, Hq, Hkv, Sq, Skv, D = 2, 8, 2, 3, 50, 32
    q, k, v = _bf16((B, Hq, Sq, D), 4), _bf16((B, Hkv, Skv, D), 5), _bf16((B, Hkv, Skv, D), 6)
    o, lse = oracle.attention(q, k, v, 0.25)
    kr, vr = k.repeat_interleave(Hq // Hkv, dim=1), v.repeat_interleave(Hq // Hkv, dim=1)
    np.testing.assert_allclose(o, _sdpa64(q, kr, vr, 0.25).reshape(-1, D).numpy(), atol=1e-12)
    np.testing.assert_allclose(lse, _lse64(q, kr, 0.25).reshape(-1).numpy(), atol=1e-12)


def test_ragged_equals_truncated_dense():
    B, H, Skv, D = 4, 2, 40, 16
    q, k, v = _bf16((B, H, 2, D), 7), _bf16((B, H, Skv, D), 8), _bf16((B, H, Skv, D), 9)
    sl = np.array([3, 1, 40, 17], dtype=np.int32)
    o, lse = oracle.attention(q, k, v, 0.3, seqlens_k=sl)
    o = o.reshape(B, H, 2, D)
    lse = lse.reshape(B, H, 2)
    for b in range(B):
        n = int(sl[b])
        ob, lb = oracle.attention(q[b:b + 1], k[b:b + 1, :, :n].contiguous(), v[b:b + 1, :, :n].contiguous(), 0.3)
        np.testing.assert_array_equal(o[b].reshape(-1, D), ob)
        np.testing.assert_array_equal(lse[b].reshape(-1), lb)
        np.testing.assert_allclose(ob, _sdpa64(q[b:b+1], k[b:b+1, :, :n], v[b:b+1, :, :n], 0.3).reshape(-1, D).numpy(), atol=1e-12)


def test_empty_key_set():
    q, k, v = _bf16((2, 1, 1, 8), 1), _bf16((2, 1, 4, 8), 2), _bf16((2, 1, 4, 8), 3)
    o, lse = oracle.attention(q, k, v, 1.0, seqlens_k=np.array([0, 4], dtype=np.int32))
    assert np.all(o[0] == 0.0) and lse[0] == -np.inf
    assert np.isfinite(lse[1])


def test_row_subset_equals_full():
    q, k, v = _bf16((2, 4, 3, 16), 10), _bf16((2, 2, 20, 16), 11), _bf16((2, 2, 20, 16), 12)
    o, lse = oracle.attention(q, k, v, 0.5)
    rows = np.array([23, 0, 7, 7, 12], dtype=np.int64)
    os_, ls = oracle.attention(q, k, v, 0.5, rows=rows)
    np.testing.assert_array_equal(os_, o[rows])
    np.testing.assert_array_equal(ls, lse[rows])


def test_single_key_returns_that_value_row():
    q, k, v = _bf16((1, 3, 2, 64), 13), _bf16((1, 3, 1, 64), 14), _bf16((1, 3, 1, 64), 15)
    o, lse = oracle.attention(q, k, v, 0.125)
    o = o.reshape(1, 3, 2, 64)
    for h in range(3):
        for i in range(2):
            np.testing.assert_array_equal(o[0, h, i], v[0, h, 0].double().numpy())
            s0 = 0.125 * float((q[0, h, i].double() * k[0, h, 0].double()).sum())
            assert abs(lse.reshape(3, 2)[h, i] - s0) <= 1e-14 * max(1.0, abs(s0))


def test_identical_keys_give_mean_of_values():
    n, D = 33, 16
    q, v = _bf16((1, 1, 1, D), 16), _bf16((1, 1, n, D), 17)
    k = _bf16((1, 1, 1, D), 18).expand(1, 1, n, D).contiguous()
    o, lse = oracle.attention(q, k, v, 0.7)
    np.testing.assert_allclose(o[0], v[0, 0].double().mean(0).numpy(), atol=1e-14)
    s = 0.7 * float((q[0, 0, 0].double() * k[0, 0, 0].double()).sum())
    assert abs(lse[0] - (s + math.log(n))) < 1e-13


def test_zero_query_gives_mean_and_log_n():
    n, D = 100, 32
    q = torch.zeros((1, 1, 1, D), dtype=torch.bfloat16)
    k, v = _bf16((1, 1, n, D), 19), _bf16((1, 1, n, D), 20)
    o, lse = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0], v[0, 0].double().mean(0).numpy(), atol=1e-14)
    assert abs(lse[0] - math.log(n)) < 1e-14


@pytest.mark.parametrize("sigma,causal,ragged", [(1.0, False, False), (4.0, False, False), (1.0, True, False),
                                                  (2.0, True, True)])
def test_softmax_rows_sum_to_one_constant_values(sigma, causal, ragged):
    """Softmax rows sum to 1, so a constant value matrix V = c gives O = c for every visible row,
    whatever the scores (large sigma: very skewed weights), the mask or the key lengths."""
    B, H, Sq, Skv, D = 2, 2, 5, 300, 16
    q, k = _bf16((B, H, Sq, D), 60, sigma), _bf16((B, H, Skv, D), 61, sigma)
    sl = np.array([300, 7], dtype=np.int32) if ragged else None
    for c in (1.0, -2.5):
        v = torch.full((B, H, Skv, D), c, dtype=torch.bfloat16)
        o, lse = oracle.attention(q, k, v, 0.3, seqlens_k=sl, causal=causal)
        vis = np.isfinite(lse)
        assert vis.all()   # every query of these shapes sees at least one key
        # FP64 summation of n terms: relative error at most about n * 2^-52
        np.testing.assert_allclose(o, c, rtol=Skv * 2.0 ** -52, atol=0)


def test_softmax_rows_sum_to_one_identity_values():
    """With V = I (value row j is the j-th unit vector), O is the softmax row itself: its entries
    must equal exp(s_j - max) / sum_j exp(s_j - max) computed directly, and each row sums to 1."""
    Skv = D = 48
    q, k = _bf16((1, 3, 4, D), 62, 2.0), _bf16((1, 3, Skv, D), 63, 2.0)
    v = torch.eye(Skv, dtype=torch.bfloat16).expand(1, 3, Skv, D).contiguous()
    scale = 0.25
    o, _ = oracle.attention(q, k, v, scale)
    s = scale * (q.double() @ k.double().transpose(-1, -2)).reshape(-1, Skv).numpy()
    e = np.exp(s - s.max(axis=1, keepdims=True))
    np.testing.assert_allclose(o, e / e.sum(axis=1, keepdims=True), rtol=0, atol=1e-15)
    np.testing.assert_allclose(o.sum(axis=1), 1.0, rtol=0, atol=Skv * 2.0 ** -52)


def test_joint_permutation_invariance():
    q, k, v = _bf16((1, 2, 4, 32), 21), _bf16((1, 2, 64, 32), 22), _bf16((1, 2, 64, 32), 23)
    perm = torch.randperm(64, generator=torch.Generator().manual_seed(0))
    o1, l1 = oracle.attention(q, k, v, 0.2)
    o2, l2 = oracle.attention(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), 0.2)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_dominant_key():
    D = 16
    q = torch.ones((1, 1, 1, D), dtype=torch.bfloat16)
    k = torch.zeros((1, 1, 8, D), dtype=torch.bfloat16)
    k[0, 0, 3] = 4.0  # s_3 = 64 * scale, all others 0
    v = _bf16((1, 1, 8, D), 24)
    o, lse = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0], v[0, 0, 3].double().numpy(), atol=1e-20 + 1e-25)
    assert abs(lse[0] - (64.0 + math.log1p(7 * math.exp(-64.0)))) < 1e-12


def test_brute_force_arbitrary_precision():
    """Tiny shapes against sum_j e^{s_j} v_j / sum_j e^{s_j} at 50 digits, no max subtraction."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    for seed, (Skv, D) in enumerate([(1, 1), (3, 2), (8, 8), (5, 7)]):
        q, k, v = _bf16((1, 1, 1, D), 100 + seed, 2.0), _bf16((1, 1, Skv, D), 200 + seed, 2.0), _bf16((1, 1, Skv, D), 300 + seed)
        scale = 0.37
        o, lse = oracle.attention(q, k, v, scale)
        qq = [mpmath.mpf(float(x)) for x in q[0, 0, 0].float()]
        es = []
        for j in range(Skv):
            kk = [mpmath.mpf(float(x)) for x in k[0, 0, j].float()]
            es.append(mpmath.exp(mpmath.mpf(scale) * mpmath.fsum(a * b for a, b in zip(qq, kk))))
        den = mpmath.fsum(es)
        for d in range(D):
            num = mpmath.fsum(es[j] * mpmath.mpf(float(v[0, 0, j, d])) for j in range(Skv))
            assert abs(float(num / den) - o[0, d]) <= 1e-14
        assert abs(float(mpmath.log(den)) - lse[0]) <= 1e-14


def test_brute_force_batched_grouped_layout():
    """The same 50-digit brute force over every row of a batched grouped-query problem, with no
    library routine involved: output row (b, hq, i) uses query head hq of batch b and key/value
    head hq // (Hq / Hkv) of the same batch, in contiguous (batch, head, sequence, dim) order."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    B, Hq, Hkv, Sq, Skv, D = 2, 4, 2, 2, 3, 2
    q, k, v = _bf16((B, Hq, Sq, D), 110, 2.0), _bf16((B, Hkv, Skv, D), 210, 2.0), _bf16((B, Hkv, Skv, D), 310)
    scale = 0.61
    o, lse = oracle.attention(q, k, v, scale)
    mp = lambda x: mpmath.mpf(float(x))
    row = 0
    for b in range(B):
        for hq in range(Hq):
            h = hq // (Hq // Hkv)
            for i in range(Sq):
                es = [mpmath.exp(mpmath.mpf(scale) * mpmath.fsum(mp(q[b, hq, i, d]) * mp(k[b, h, j, d]) for d in range(D)))
                      for j in range(Skv)]
                den = mpmath.fsum(es)
                for d in range(D):
                    num = mpmath.fsum(es[j] * mp(v[b, h, j, d]) for j in range(Skv))
                    assert abs(float(num / den) - o[row, d]) <= 1e-14, (b, hq, i, d)
                assert abs(float(mpmath.log(den)) - lse[row]) <= 1e-14, (b, hq, i)
                row += 1


def test_qk_raw_product():
    g = torch.Generator().manual_seed(5)
    q = torch.randint(-4, 5, (1, 16), generator=g).to(torch.bfloat16)
    k = torch.randint(-4, 5, (128, 16), generator=g).to(torch.bfloat16)
    s = oracle.qk(q, k)
    np.testing.assert_array_equal(s, (q.double() @ k.double().T).numpy())
    qn, kn = _bf16((3, 64), 30), _bf16((128, 64), 31)
    np.testing.assert_allclose(oracle.qk(qn, kn), (qn.double() @ kn.double().T).numpy(), atol=1e-12)


def test_oracle_sees_generator_slices():
    """The numpy slice generator and the torch generator give the same BF16 bits."""
    w = inputs.Workload("t", 2, 4, 2, 3, 40, 16, 0.5, "bf16", 77)
    q, k, v, _ = w.make()
    rows = [0, 5, 23]
    qr = w.q_rows_np(rows)
    np.testing.assert_array_equal(qr, q.reshape(-1, 16)[rows].view(torch.int16).numpy().view(np.uint16))
    kk, vv = w.kv_head_np(1, 1, 33)
    np.testing.assert_array_equal(kk, k[1, 1, :33].contiguous().view(torch.int16).numpy().view(np.uint16))
    np.testing.assert_array_equal(vv, v[1, 1, :33].contiguous().view(torch.int16).numpy().view(np.uint16))


def test_generator_distribution():
    t = inputs.normal_bf16_torch((1 << 18,), 1, 0, 1.0).double()
    assert abs(float(t.mean())) < 0.01 and abs(float(t.std()) - 1.0) < 0.01
    t = inputs.normal_bf16_torch((1 << 18,), 1, 0, 0.5).double()
    assert abs(float(t.std()) - 0.5) < 0.005


def _bottom_right_mask(Sq, n):
    i = torch.arange(Sq)[:, None]
    j = torch.arange(n)[None, :]
    return j <= i + (n - Sq)


@pytest.mark.parametrize("Sq,Skv", [(37, 37), (5, 300), (1, 64), (130, 129)])
def test_causal_matches_masked_sdpa(Sq, Skv):
    """Bottom-right aligned causal mask against torch FP64 SDPA with the explicit boolean mask
    (and is_causal=True when Sq == Skv, where both alignments coincide)."""
    B, Hq, Hkv, D = 2, 4, 2, 16
    q, k, v = _bf16((B, Hq, Sq, D), 31), _bf16((B, Hkv, Skv, D), 32), _bf16((B, Hkv, Skv, D), 33)
    o, lse = oracle.attention(q, k, v, 0.3, causal=True)
    kr, vr = k.repeat_interleave(Hq // Hkv, dim=1), v.repeat_interleave(Hq // Hkv, dim=1)
    mask = _bottom_right_mask(Sq, Skv)
    ref = F.scaled_dot_product_attention(q.double(), kr.double(), vr.double(), attn_mask=mask, scale=0.3)
    valid = mask.any(dim=1)                       # rows with at least one visible key
    o4, lse4 = o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)
    np.testing.assert_allclose(o4[:, :, valid.numpy()], ref[:, :, valid].numpy(), atol=1e-12)
    s = 0.3 * (q.double() @ kr.double().transpose(-1, -2))
    s = s.masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse4[:, :, valid.numpy()], torch.logsumexp(s, -1)[:, :, valid].numpy(), atol=1e-12)
    assert np.all(o4[:, :, ~valid.numpy()] == 0.0) and np.all(np.isneginf(lse4[:, :, ~valid.numpy()]))
    if Sq == Skv:
        ref2 = F.scaled_dot_product_attention(q.double(), kr.double(), vr.double(), is_causal=True, scale=0.3)
        np.testing.assert_allclose(o4, ref2.numpy(), atol=1e-12)


def test_causal_ragged_is_relative_to_each_length():
    B, H, Sq, Skv, D = 3, 2, 4, 50, 8
    q, k, v = _bf16((B, H, Sq, D), 34), _bf16((B, H, Skv, D), 35), _bf16((B, H, Skv, D), 36)
    sl = np.array([10, 2, 50], dtype=np.int32)
    o, lse = oracle.attention(q, k, v, 0.5, seqlens_k=sl, causal=True)
    o = o.reshape(B, H, Sq, D)
    for b in range(B):
        n = int(sl[b])
        mask = _bottom_right_mask(Sq, n)
        valid = mask.any(dim=1)
        ref = F.scaled_dot_product_attention(q[b:b+1].double(), k[b:b+1, :, :n].double(), v[b:b+1, :, :n].double(),
                                             attn_mask=mask, scale=0.5)
        np.testing.assert_allclose(o[b][:, valid.numpy()], ref[0][:, valid].numpy(), atol=1e-12)
        assert np.all(o[b][:, ~valid.numpy()] == 0.0)


def test_causal_single_query_is_dense():
    q, k, v = _bf16((1, 2, 1, 32), 37), _bf16((1, 2, 77, 32), 38), _bf16((1, 2, 77, 32), 39)
    a = oracle.attention(q, k, v, 0.2, causal=True)
    b = oracle.attention(q, k, v, 0.2)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
