"""Back-to-back calls on one stream whose buffers depend on each other, with no synchronisation in
between.  The library launches its kernels with programmatic dependent launch: a call's kernel may be
placed on the SMs while the previous kernel still runs, and must not touch global memory before that
kernel has completed.  Each chain is

    1. A = attn(q0)        (into buffer bufA)
    2. B = attn(bufA)      reads what call 1 wrote (read after write)
    3. attn(q3) -> bufA    overwrites call 2's input (write after read)

and afterwards call 2's output is compared with the FP64 oracle on call 1's output, and bufA with a
separate call on q3 (the kernels are deterministic, so the bits must agree).  Each chain runs on the
legacy default stream and on a stream the caller created."""
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


CASES = {
    # name: (B, Hq, Hkv, Sq, Skv, D, causal, ragged, second call's output)
    "decode_split_1col": (4, 8, 8, 1, 2000, 128, False, False, "bf16"),         # in-kernel merge, six warps
    "decode_split_4col": (2, 16, 4, 1, 3000, 128, False, False, "bf16"),        # epilogue warpgroup
    "decode_ragged_combine": (4, 8, 2, 1, 1500, 128, False, True, "bf16"),      # prefix, decode, combine
    "decode_nvfp4_two_pass": (4, 8, 2, 1, 1500, 128, False, False, "nvfp4"),    # decode, quantiser
    "prefill_causal_counter": (1, 4, 2, 300, 500, 64, True, False, "bf16"),     # work-item counter
    "prefill_d128": (1, 2, 2, 400, 400, 128, False, False, "bf16"),
    "wide_split_combine": (2, 32, 1, 1, 900, 512, False, False, "bf16"),        # wide kernel, combine
}


class Call:
    """One fmha_fwd_ex configuration with its own workspace and output buffers."""

    def __init__(self, F, shape, seqlens, causal, kind):
        B, Hq, Hkv, Sq, Skv, D = shape
        self.F, self.shape, self.kind = F, shape, kind
        n = B * Hq * Sq * D
        self.lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
        if kind == "nvfp4":
            self.codes = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
            self.scales = torch.zeros(n // 16, dtype=torch.uint8, device="cuda")
            self.ts = torch.zeros(1, dtype=torch.float32, device="cuda")
            self.f32 = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
            okind = F.FMHA_OUT_NVFP4
        else:
            self.codes = self.scales = self.ts = self.f32 = None
            okind = F.FMHA_OUT_BF16
        o = F.make_opts(okind, seqlens, 0, None, self.scales, self.ts, self.f32, causal)
        wsb = F.fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, o)
        self.ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        self.opts = F.make_opts(okind, seqlens, 0, self.ws, self.scales, self.ts, self.f32, causal)

    def __call__(self, q, k, v, out, scale):
        self.F.fmha_fwd_ex(q, k, v, self.codes if self.kind == "nvfp4" else out, self.lse, scale, self.opts)


@pytest.mark.parametrize("stream", ["default", "created"])
@pytest.mark.parametrize("name", list(CASES))
def test_dependent_calls_back_to_back(F, name, stream):
    B, Hq, Hkv, Sq, Skv, D, causal, ragged, kind2 = CASES[name]
    w = inputs.Workload("chain", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 91, ragged=ragged)
    q0, k, v, sl = w.make("cuda")
    q3 = inputs.Workload("chain3", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 92, ragged=ragged).make("cuda")[0]
    shape = (B, Hq, Hkv, Sq, Skv, D)
    c1, c3 = Call(F, shape, sl, causal, "bf16"), Call(F, shape, sl, causal, "bf16")
    c2 = Call(F, shape, sl, causal, kind2)
    bufA = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    bufB = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    side = torch.cuda.Stream() if stream == "created" else torch.cuda.current_stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):   # the library launches on the current stream
        c1(q0, k, v, bufA, w.scale)
        c2(bufA, k, v, bufB, w.scale)
        c3(q3, k, v, bufA, w.scale)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    got_b = (c2.f32.cpu().numpy() if kind2 == "nvfp4" else bufB.float().cpu().numpy()).reshape(-1, D)
    got_lse2 = c2.lse.cpu().numpy().reshape(-1)
    got_a = bufA.clone()

    # call 1's output again, alone: the input call 2 saw
    a1 = torch.full_like(bufA, float("nan"))
    c1(q0, k, v, a1, w.scale)
    # call 3 alone: what bufA must hold
    a3 = torch.full_like(bufA, float("nan"))
    c3(q3, k, v, a3, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(got_a, a3), f"{name}: the overwriting call differs from the same call alone"

    lens = None if sl is None else sl.cpu().numpy()
    o_ref, l_ref = oracle.attention(a1.cpu(), k.cpu(), v.cpu(), w.scale, causal=causal, seqlens_k=lens)
    check_o_lse(got_b, got_lse2, o_ref, l_ref, f"chain {name}")
    if kind2 == "nvfp4":
        codes, scales, _ = oracle.nvfp4_quantize(got_b.reshape(-1))
        np.testing.assert_array_equal(c2.codes.cpu().numpy(), codes)
        np.testing.assert_array_equal(c2.scales.cpu().numpy()[: scales.size], scales)
