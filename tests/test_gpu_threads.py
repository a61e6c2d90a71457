"""Calls from several host threads at once, each on its own stream with its own inputs, workspace
and outputs (the header's thread-safety contract: per-thread error string and timing hook, shared
launch counter and status word).  ctypes releases the GIL during a call, so the library's host code
runs concurrently.  Every thread's result must equal, bit for bit, the same call made alone (the
kernels are deterministic), and one of them is also checked against the FP64 oracle."""
import threading

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


JOBS = [
    # (B, Hq, Hkv, Sq, Skv, D, causal, out kind)
    (4, 8, 8, 1, 2000, 128, False, "bf16"),     # split decode, merged in the kernel
    (2, 16, 4, 1, 3000, 128, False, "nvfp4"),   # epilogue warpgroup, two-pass NVFP4
    (1, 4, 2, 300, 500, 64, True, "f32"),       # causal row tiles, work-item counter
    (2, 32, 1, 1, 900, 512, False, "bf16"),     # wide head, split and combine
]


class Job:
    def __init__(self, F, spec, seed):
        B, Hq, Hkv, Sq, Skv, D, causal, kind = spec
        self.F, self.spec = F, spec
        self.w = inputs.Workload("thr", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", seed)
        self.q, self.k, self.v, _ = self.w.make("cuda")
        n = B * Hq * Sq * D
        self.lse = torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")
        self.scales = self.ts = None
        if kind == "nvfp4":
            self.out = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
            self.scales = torch.empty(n // 16, dtype=torch.uint8, device="cuda")
            self.ts = torch.empty(1, dtype=torch.float32, device="cuda")
            okind = F.FMHA_OUT_NVFP4
        else:
            dt = torch.float32 if kind == "f32" else torch.bfloat16
            self.out = torch.empty(B, Hq, Sq, D, dtype=dt, device="cuda")
            okind = F.FMHA_OUT_F32 if kind == "f32" else F.FMHA_OUT_BF16
        o = F.make_opts(okind, None, 0, None, self.scales, self.ts, None, causal)
        self.ws = torch.empty(max(F.fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, o), 256), dtype=torch.uint8,
                              device="cuda")
        self.opts = F.make_opts(okind, None, 0, self.ws, self.scales, self.ts, None, causal)
        self.stream = torch.cuda.Stream()
        self.error = None

    def call(self):
        self.F.fmha_fwd_ex(self.q, self.k, self.v, self.out, self.lse, self.w.scale, self.opts, stream=self.stream)

    def result(self):
        r = [self.out.clone(), self.lse.clone()]
        if self.scales is not None:
            r += [self.scales.clone(), self.ts.clone()]
        return r

    def run(self, n):
        try:
            for _ in range(n):
                self.call()
            self.stream.synchronize()
        except Exception as e:   # reported by the main thread
            self.error = e


def test_concurrent_threads_match_single_calls(F):
    jobs = [Job(F, spec, 300 + i) for i, spec in enumerate(JOBS)]
    torch.cuda.synchronize()
    alone = []
    for j in jobs:
        j.call()
        j.stream.synchronize()
        alone.append(j.result())
    for j in jobs:   # the concurrent calls must write every output again
        for t in (j.out, j.lse, j.scales, j.ts):
            if t is not None:
                t.zero_()
    torch.cuda.synchronize()
    launches0 = F.fmha_launch_count()
    threads = [threading.Thread(target=j.run, args=(20,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
        assert not t.is_alive(), "a thread did not finish"
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    for j in jobs:
        assert j.error is None, j.error
    assert F.fmha_launch_count() > launches0
    for j, ref in zip(jobs, alone):
        for got, want in zip(j.result(), ref):
            assert torch.equal(got, want), f"job {j.spec}: a concurrent call differs from the call made alone"
    # one of them against the oracle as well
    j = jobs[2]
    o_ref, l_ref = oracle.attention(j.q.cpu(), j.k.cpu(), j.v.cpu(), j.w.scale, causal=True)
    check_o_lse(j.out.cpu().numpy().reshape(-1, j.w.D), j.lse.cpu().numpy().reshape(-1), o_ref, l_ref, "threads")
