"""GPU checks of the building blocks, through the C ABI: the raw Q K^T tensor-core product, the
Tensor Memory round trip, and the two PV operand layouts (MN-major V^T as A, and P in TMEM)."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


def _ints(shape, seed, lo=-4, hi=4):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


@pytest.mark.parametrize("Sq,Skv,D", [(1, 128, 16), (1, 128, 64), (128, 128, 64), (200, 300, 128),
                                      (3, 130, 512), (1, 7, 16)])
def test_qk_gemm_integer_inputs_bit_exact(F, Sq, Skv, D):
    """Integer inputs in [-4, 4] are exact in BF16 and every partial sum is exact in FP32, so the
    tensor-core result must equal the FP64 oracle bit for bit (no 4x factor, no lost terms)."""
    q, k = _ints((Sq, D), 1), _ints((Skv, D), 2)
    s = torch.full((Sq, Skv), float("nan"), dtype=torch.float32, device="cuda")
    F.fmha_qk_gemm(q.cuda(), k.cuda(), s)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    ref = oracle.qk(q, k)
    np.testing.assert_array_equal(s.cpu().double().numpy(), ref)


@pytest.mark.parametrize("D", [16, 64, 128])
def test_qk_gemm_normal_inputs_within_fp32_bound(F, D):
    g = torch.Generator().manual_seed(3)
    q = torch.randn(1, D, generator=g).to(torch.bfloat16)
    k = torch.randn(128, D, generator=g).to(torch.bfloat16)
    s = torch.empty(1, 128, dtype=torch.float32, device="cuda")
    F.fmha_qk_gemm(q.cuda(), k.cuda(), s)
    ref = oracle.qk(q, k)
    bound = D * 2.0 ** -23 * (q.double().abs() @ k.double().abs().T).numpy()
    assert np.all(np.abs(s.cpu().double().numpy() - ref) <= bound)


def test_tmem_round_trip(F):
    out = torch.zeros(128 * 64, dtype=torch.int32, device="cuda")
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    F.fmha_selftest(1, dummy, out)
    got = out.cpu().numpy().astype(np.int64).reshape(128, 64)
    lane = np.arange(128)[:, None]
    col = np.arange(64)[None, :]
    np.testing.assert_array_equal(got, lane * 1000 + col)


@pytest.mark.parametrize("D", [64, 128])
def test_pv_swap_ab_mn_major(F, D):
    """O^T[d][q] = sum_kv V[kv][d] P[q][kv]: V^T is the MN-major A operand, P^T the K-major B."""
    V = _ints((128, D), 4)
    P = _ints((16, 128), 5, -2, 2)
    inp = torch.cat([V.reshape(-1), P.reshape(-1)]).cuda()
    out = torch.full((128 * 16,), float("nan"), dtype=torch.float32, device="cuda")
    F.fmha_selftest(2, inp, out, D)
    got = out.cpu().double().numpy().reshape(128, 16)
    ref = (V.double().T @ P.double().T).numpy()      # [D][16]
    np.testing.assert_array_equal(got[:D], ref)
    if D == 64:   # the M rows above D repeat rows 0..63 (LBO = 0)
        np.testing.assert_array_equal(got[64:], ref)


@pytest.mark.parametrize("D", [64, 128, 256])
def test_pv_p_in_tensor_memory(F, D):
    """O = P V with P in Tensor Memory (A operand) and V MN-major in shared memory."""
    V = _ints((128, D), 6)
    P = _ints((128, 128), 7, -2, 2)
    inp = torch.cat([V.reshape(-1), P.reshape(-1)]).cuda()
    out = torch.full((128 * D,), float("nan"), dtype=torch.float32, device="cuda")
    F.fmha_selftest(3, inp, out, D)
    got = out.cpu().double().numpy().reshape(128, D)
    np.testing.assert_array_equal(got, (P.double() @ V.double()).numpy())


@pytest.mark.parametrize("flags", [0, 1, 2, 3, 4, 5, 6, 7])
def test_pair_mma_layout(F, flags):
    """The CTA-pair MMA (cta_group::2, M = 256) on integer inputs, bit-exact: the even CTA's Tensor
    Memory holds rows 0..127 of D and the odd CTA's rows 128..255 (each from its own rows of A), and
    B's columns come half from each CTA's shared memory, the first half from the even CTA.
    flags bit 0: A from Tensor Memory (TS form, B = V MN-major) instead of shared memory (SS form);
    bit 1: the completion reaches the odd CTA by a commit aimed at its barrier (else a relayed arrive);
    bit 2: the odd CTA's copy counts its bytes on the even CTA's barrier (else a relayed arrive)."""
    ts = flags & 1
    N, K = (256, 32) if ts else (128, 64)
    A = _ints((256, K), 10 + flags)
    B = _ints((K, N), 20 + flags) if ts else _ints((N, K), 20 + flags)
    inp = torch.cat([A.reshape(-1), B.reshape(-1)]).cuda()
    out = torch.full((2 * 128 * N + 2,), float("nan"), dtype=torch.float32, device="cuda")
    F.fmha_selftest(4, inp, out, flags)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    got = out.cpu().double().numpy()
    assert got[-2] == 0.0 and got[-1] == 0.0, "a wait gave up"
    D = got[: 2 * 128 * N].reshape(256, N)
    ref = (A.double() @ (B.double() if ts else B.double().T)).numpy()
    np.testing.assert_array_equal(D, ref)
