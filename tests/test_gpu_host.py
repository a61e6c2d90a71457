"""GPU parity of fmha_fwd_host (attention from host memory: copies in, attention, copies out, in
batch chunks whose copies overlap the previous chunk's attention) against the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


def _run_host(F, w, out_kind, causal=False, pinned=True, with_lse=True, dev_buf=None):
    q, k, v, _ = w.make("cpu")
    if pinned:
        q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    dt = torch.float32 if out_kind == F.FMHA_OUT_F32 else torch.bfloat16
    out = torch.full((w.B, w.Hq, w.Sq, w.D), float("nan"), dtype=dt)
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32) if with_lse else None
    if pinned:
        out = out.pin_memory()
        lse = lse.pin_memory() if lse is not None else None
    o = F.make_opts(out_kind, causal=causal)
    need = F.fmha_host_buffer_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, o)
    if dev_buf is None:
        dev_buf = torch.empty(need, dtype=torch.uint8, device="cuda")
    F.fmha_fwd_host(q, k, v, out, lse, w.scale, dev_buf, o)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    return q, k, v, out, lse, dev_buf


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,out", [
    (1, 8, 2, 1, 700, 128, "f32"),      # one chunk: everything on the caller's stream
    (3, 8, 2, 1, 700, 128, "bf16"),     # three chunks of one batch entry
    (5, 4, 4, 1, 300, 64, "f32"),       # chunks of 2, 2, 1
    (8, 16, 2, 2, 513, 128, "bf16"),    # four chunks of two; decode with 16 columns per unit
    (2, 2, 2, 300, 400, 64, "f32"),     # row-tile path, two chunks
    (2, 64, 1, 1, 300, 512, "bf16"),    # wide heads (D = 512), two chunks
])
def test_host_matches_oracle(F, B, Hq, Hkv, Sq, Skv, D, out):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 71)
    kind = F.FMHA_OUT_F32 if out == "f32" else F.FMHA_OUT_BF16
    q, k, v, o, lse, _ = _run_host(F, w, kind)
    o_ref, l_ref = oracle.attention(q, k, v, w.scale)
    check_o_lse(o.float().numpy().reshape(-1, w.D), lse.numpy().reshape(-1), o_ref, l_ref, f"host {out}")


def test_host_causal_pageable_no_lse_and_repeat(F):
    """Causal mask, pageable host memory, no LSE; a second call on the same device buffer (whose
    staging still holds the first call's tensors) gives the same bits."""
    w = inputs.Workload("t", 4, 8, 2, 4, 600, 128, 1.0, "bf16", 72)
    q, k, v, o1, _, buf = _run_host(F, w, F.FMHA_OUT_F32, causal=True, pinned=False, with_lse=False)
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, causal=True)
    check_o_lse(o1.numpy().reshape(-1, w.D), None, o_ref, l_ref, "host causal")
    _, _, _, o2, _, _ = _run_host(F, w, F.FMHA_OUT_F32, causal=True, pinned=False, with_lse=False, dev_buf=buf)
    assert torch.equal(o1, o2)


def test_host_matches_device_call(F):
    """The host entry point agrees with fmha_fwd_ex on device copies of the inputs (within
    rounding: its chunks split the keys over the SMs differently), and both with the oracle."""
    w = inputs.Workload("t", 6, 8, 2, 1, 900, 128, 1.0, "bf16", 73)
    q, k, v, o_host, lse_host, _ = _run_host(F, w, F.FMHA_OUT_BF16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(w.B, w.Hq, w.Sq, w.D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device="cuda")
    F.fmha_fwd_ex(qd, kd, vd, out, lse, w.scale, F.make_opts(F.FMHA_OUT_BF16, num_splits=1))
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention(q, k, v, w.scale)
    check_o_lse(out.float().cpu().numpy().reshape(-1, w.D), lse.cpu().numpy().reshape(-1), o_ref, l_ref, "device")
    check_o_lse(o_host.float().numpy().reshape(-1, w.D), lse_host.numpy().reshape(-1), o_ref, l_ref, "host")
    np.testing.assert_allclose(o_host.float().numpy(), out.float().cpu().numpy(), atol=2e-2)


def _host_cases(n=24, seed=515):
    rng = np.random.default_rng(seed)
    cases = []
    while len(cases) < n:
        D = int(rng.choice([64, 128, 512], p=[0.4, 0.4, 0.2]))
        Hkv = int(rng.choice([1, 2, 4]))
        Hq = Hkv * int(rng.choice([1, 2, 4, 8, 16]))
        Sq = int(rng.choice([1, 1, 2, 4, 33, 130]))
        Skv = int(rng.integers(1, 2000))
        B = int(rng.integers(1, 9))
        if B * Hq * Sq * Skv * D > 2e8:
            continue
        cases.append((B, Hq, Hkv, Sq, Skv, D, bool(rng.random() < 0.4), str(rng.choice(["bf16", "f32"])),
                      int(rng.integers(0, 2)), int(rng.integers(1, 1 << 30))))
    return cases


HOST_CASES = _host_cases()


@pytest.mark.parametrize("case", HOST_CASES, ids=[f"h{i}" for i in range(len(HOST_CASES))])
def test_host_random_shapes(F, case):
    """A seeded sweep of shapes through fmha_fwd_host (1 to 8 batch entries, so one to four chunks),
    against the oracle."""
    B, Hq, Hkv, Sq, Skv, D, causal, out, splits, seed = case
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", seed)
    q, k, v, _ = w.make("cpu")
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    kind = F.FMHA_OUT_F32 if out == "f32" else F.FMHA_OUT_BF16
    o = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.float32 if out == "f32" else torch.bfloat16).pin_memory()
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32).pin_memory()
    opts = F.make_opts(kind, num_splits=splits, causal=causal)
    buf = torch.empty(F.fmha_host_buffer_size(B, Hq, Hkv, Sq, Skv, D, opts), dtype=torch.uint8, device="cuda")
    F.fmha_fwd_host(q, k, v, o, lse, w.scale, buf, opts)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    o_ref, l_ref = oracle.attention(q, k, v, w.scale, causal=causal)
    check_o_lse(o.float().numpy().reshape(-1, D), lse.numpy().reshape(-1), o_ref, l_ref, f"host {case}")
