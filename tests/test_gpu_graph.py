"""CUDA graph capture and replay of the library's calls.  A replay reuses everything the capture
recorded, including the per-call tag of the split-KV merge's arrival counters, so the kernels must
leave nothing behind that the next replay would misread.  Each replay must give the same bits as a
direct call (the merge adds the partials in slot order whichever CTA does it)."""
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
    # name: (B, Hq, Hkv, Sq, Skv, D, out kind, causal)
    "decode_1col": (2, 8, 8, 1, 3000, 128, "bf16", False),      # in-kernel merge, six-warp kernel
    "decode_16col": (1, 16, 1, 1, 5100, 128, "bf16", False),    # in-kernel merge, epilogue warpgroup
    "prefill_causal": (2, 4, 2, 300, 700, 64, "f32", True),     # work-item counter in the workspace
    "wide": (2, 32, 1, 1, 900, 512, "bf16", False),             # split pairs and the combine kernel
    "decode_nvfp4": (4, 8, 2, 1, 1500, 128, "nvfp4", False),    # two-pass NVFP4: amax word, quantiser
}


def _setup(F, name):
    B, Hq, Hkv, Sq, Skv, D, kind, causal = CASES[name]
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 81)
    q, k, v, _ = w.make("cuda")
    n = B * Hq * Sq * D
    bufs = {"lse": torch.empty(B, Hq, Sq, dtype=torch.float32, device="cuda")}
    if kind == "nvfp4":
        bufs["out"] = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
        bufs["scales"] = torch.empty(n // 16, dtype=torch.uint8, device="cuda")
        bufs["ts"] = torch.empty(1, dtype=torch.float32, device="cuda")
        bufs["f32"] = torch.empty(n, dtype=torch.float32, device="cuda")
        okind = F.FMHA_OUT_NVFP4
    else:
        dt = torch.float32 if kind == "f32" else torch.bfloat16
        bufs["out"] = torch.empty(B, Hq, Sq, D, dtype=dt, device="cuda")
        okind = F.FMHA_OUT_F32 if kind == "f32" else F.FMHA_OUT_BF16
    o = F.make_opts(okind, None, 0, None, bufs.get("scales"), bufs.get("ts"), bufs.get("f32"), causal)
    wsb = F.fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, o)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    opts = F.make_opts(okind, None, 0, ws, bufs.get("scales"), bufs.get("ts"), bufs.get("f32"), causal)

    def call():
        F.fmha_fwd_ex(q, k, v, bufs["out"], bufs["lse"], w.scale, opts)

    # opts holds only the workspace's address: the tensor must outlive every call and replay (torch
    # frees its cached memory with cudaFree when a capture begins)
    call.workspace = ws
    return w, (q, k, v), bufs, call


def _snapshot(bufs):
    return {k: t.clone() for k, t in bufs.items()}


@pytest.mark.parametrize("name", list(CASES))
def test_graph_replay_matches_direct_call(F, name):
    w, (q, k, v), bufs, call = _setup(F, name)
    call()                                   # outside the capture: sets the kernels' attributes once
    torch.cuda.synchronize()
    direct = _snapshot(bufs)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    for _ in range(3):
        for t in bufs.values():
            t.fill_(0)
        g.replay()
        torch.cuda.synchronize()
        assert F.fmha_check_status() == 0
        for key in bufs:
            assert torch.equal(bufs[key], direct[key]), f"{name}: {key} differs from the direct call"
    kind, causal = CASES[name][6], CASES[name][7]
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=causal)
    if kind == "nvfp4":
        o = bufs["f32"].cpu().numpy().reshape(-1, w.D)
        codes, scales, sg = oracle.nvfp4_quantize(o.reshape(-1))
        np.testing.assert_array_equal(bufs["out"].cpu().numpy(), codes)
        np.testing.assert_array_equal(bufs["scales"].cpu().numpy()[: scales.size], scales)
    else:
        o = bufs["out"].float().cpu().numpy().reshape(-1, w.D)
    check_o_lse(o, bufs["lse"].cpu().numpy().reshape(-1), o_ref, l_ref, f"graph {name}")


def test_graph_replay_of_host_entry_point(F):
    """fmha_fwd_host in a CUDA graph: its copy stream joins the capture through events, the copies
    become memcpy nodes on the page-locked host buffers, and a replay gives the same bits."""
    w = inputs.Workload("t", 4, 8, 2, 1, 1500, 128, 1.0, "bf16", 82)
    q, k, v, _ = w.make("cpu")
    q, k, v = q.pin_memory(), k.pin_memory(), v.pin_memory()
    out = torch.zeros(w.B, w.Hq, w.Sq, w.D, dtype=torch.float32).pin_memory()
    lse = torch.zeros(w.B, w.Hq, w.Sq, dtype=torch.float32).pin_memory()
    opts = F.make_opts(F.FMHA_OUT_F32)
    buf = torch.empty(F.fmha_host_buffer_size(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, opts), dtype=torch.uint8,
                      device="cuda")
    F.fmha_fwd_host(q, k, v, out, lse, w.scale, buf, opts)
    torch.cuda.synchronize()
    direct_o, direct_l = out.clone(), lse.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        F.fmha_fwd_host(q, k, v, out, lse, w.scale, buf, opts)
    torch.cuda.synchronize()
    for _ in range(2):
        out.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, direct_o) and torch.equal(lse, direct_l)
    o_ref, l_ref = oracle.attention(q, k, v, w.scale)
    check_o_lse(out.numpy().reshape(-1, w.D), lse.numpy().reshape(-1), o_ref, l_ref, "graph host")
