"""Helpers for the GPU parity tests: run the library through the C ABI and compare with the
FP64 oracle (full tensors for small cases, sampled rows for the full-size workloads)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from attention_tensor_cores_gb300 import inputs

# Tolerances: O max |err| <= 2e-2 and mean |err| <= 2e-3; LSE |err| <= 1e-3 * max(1, |lse|).
O_MAX = 2e-2
O_MEAN = 2e-3
LSE_REL = 1e-3


def run_attention(F, q, k, v, scale, out_kind="bf16", seqlens=None, num_splits=None, want_f32=False, causal=False,
                  nvfp4_scale=None, want_amax=False, wide_variant=None):
    """Calls fmha_fwd (no options) or fmha_fwd_ex; returns dict of host numpy results.

    nvfp4_scale: a given per-tensor scale s_g (single-pass NVFP4); want_amax: also return max|O|
    through opts.out_amax; wide_variant: opts.wide_variant for D = 512 (None: automatic)."""
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    lse = torch.full((B, Hq, Sq), float("nan"), dtype=torch.float32, device="cuda")
    res = {}
    if out_kind == "bf16" and seqlens is None and num_splits is None and not causal and wide_variant is None:
        out = torch.full((B, Hq, Sq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        F.fmha_fwd(q, k, v, out, lse, scale)
        torch.cuda.synchronize()
        res["o"] = out.float().cpu().numpy().reshape(-1, D)
    else:
        kind = {"bf16": F.FMHA_OUT_BF16, "f32": F.FMHA_OUT_F32, "nvfp4": F.FMHA_OUT_NVFP4}[out_kind]
        n = B * Hq * Sq * D
        if out_kind == "nvfp4":
            out = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
            scales = torch.zeros(n // 16, dtype=torch.uint8, device="cuda")
            ts = torch.zeros(1, dtype=torch.float32, device="cuda")
            f32 = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda") if want_f32 else None
            sg_in = None if nvfp4_scale is None else torch.tensor([nvfp4_scale], dtype=torch.float32, device="cuda")
            amax = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda") if want_amax else None
        else:
            sg_in = amax = None
            dt = torch.bfloat16 if out_kind == "bf16" else torch.float32
            out = torch.full((B, Hq, Sq, D), float("nan"), dtype=dt, device="cuda")
            scales = ts = f32 = None
        ns = 0 if num_splits is None else num_splits
        wv = F.FMHA_WIDE_AUTO if wide_variant is None else wide_variant
        opts = F.make_opts(kind, seqlens, ns, None, scales, ts, f32, causal, sg_in, amax, wv)
        wsb = F.fmha_workspace_size(B, Hq, Hkv, Sq, Skv, D, opts)
        ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device="cuda") if wsb else None
        opts = F.make_opts(kind, seqlens, ns, ws, scales, ts, f32, causal, sg_in, amax, wv)
        res["workspace_bytes"] = wsb
        F.fmha_fwd_ex(q, k, v, out, lse, scale, opts)
        torch.cuda.synchronize()
        if out_kind == "nvfp4":
            res["codes"] = out.cpu().numpy()
            res["scales"] = scales.cpu().numpy()
            res["tensor_scale"] = float(ts.cpu()[0])
            if want_amax:
                res["amax"] = float(amax.cpu()[0])
            if want_f32:
                res["o"] = f32.cpu().numpy().reshape(-1, D)
        else:
            res["o"] = out.float().cpu().numpy().reshape(-1, D)
    res["lse"] = lse.cpu().numpy().reshape(-1)
    assert F.fmha_check_status() == 0, "device status word set (bounded wait expired)"
    return res


def check_o_lse(o, lse, o_ref, lse_ref, what=""):
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    err = np.abs(o.astype(np.float64) - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    assert err.max() <= O_MAX, f"{what}: max|dO| = {err.max():.3e}"
    assert err.mean() <= O_MEAN, f"{what}: mean|dO| = {err.mean():.3e}"
    if lse is not None:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin) and np.all(lse[~fin] == lse_ref[~fin]), f"{what}: LSE inf pattern"
        lerr = np.abs(lse[fin].astype(np.float64) - lse_ref[fin])
        assert np.all(lerr <= LSE_REL * np.maximum(1.0, np.abs(lse_ref[fin]))), f"{what}: max|dLSE| = {lerr.max():.3e}"
    return float(err.max()), float(err.mean())


def oracle_rows(w: inputs.Workload, rows, causal: bool = False, tensors=None):
    """FP64 oracle for flat query rows of workload `w`.

    tensors: the (q, k, v) torch tensors the GPU call used (any device): they are copied to the host
    and the oracle computes every requested row in one call.  Without them the oracle regenerates
    just the slices it needs from the seeded generator (slow for long key sets)."""
    sl = w.seqlens()
    rows = np.asarray(rows, dtype=np.int64)
    if tensors is not None:
        q, k, v = (t.cpu() for t in tensors)
        return oracle.attention(q, k, v, w.scale, seqlens_k=sl, rows=rows, causal=causal)
    g = w.Hq // w.Hkv
    o = np.zeros((len(rows), w.D))
    lse = np.zeros(len(rows))
    qs = w.q_rows_np(rows)
    cache = {}
    for i, r in enumerate(rows):
        b = r // (w.Hq * w.Sq)
        hq = (r // w.Sq) % w.Hq
        kvh = hq // g
        n = w.Skv if sl is None else int(sl[b])
        key = (b, kvh)
        if key not in cache:
            cache = {key: w.kv_head_np(b, kvh, n)}
        kk, vv = cache[key]
        if n == 0:
            o[i] = 0.0
            lse[i] = -math.inf
            continue
        s_idx = r % w.Sq
        if causal:   # bottom-right aligned: query s of Sq sees keys 0 .. s + n - Sq
            n_vis = max(0, min(n, s_idx + n - w.Sq + 1))
            if n_vis == 0:
                o[i] = 0.0
                lse[i] = -math.inf
                continue
        else:
            n_vis = n
        oi, li = oracle.attention(qs[i].reshape(1, 1, 1, w.D), kk[:n_vis].reshape(1, 1, n_vis, w.D),
                                  vv[:n_vis].reshape(1, 1, n_vis, w.D), w.scale)
        o[i] = oi[0]
        lse[i] = li[0]
    return o, lse


def unit_rows(w: inputs.Workload, u: int) -> tuple[int, int]:
    """Flat row range [first, end) of (b, kv-head) unit u = b * Hkv + kvh: the query rows of its
    Hq / Hkv heads, which are contiguous in the [B, Hq, Sq] order."""
    g = w.Hq // w.Hkv
    b, kvh = divmod(u, w.Hkv)
    first = (b * w.Hq + kvh * g) * w.Sq
    return first, first + g * w.Sq


def split_boundary_units(tiles_per_unit, parts: int) -> list[int]:
    """Units whose key tiles a stream-K split cuts: the tiles of all units laid end to end, part c
    of `parts` taking [c*T/parts, (c+1)*T/parts) (integer division), as the split decode and
    wide-head kernels partition them over CTAs or CTA pairs."""
    pre = np.concatenate([[0], np.cumsum(np.asarray(tiles_per_unit, dtype=np.int64))])
    T = int(pre[-1])
    cut = set()
    for c in range(1, parts):
        b = c * T // parts
        u = int(np.searchsorted(pre, b, side="right")) - 1
        if 0 <= u < len(tiles_per_unit) and pre[u] < b < pre[u + 1]:
            cut.add(u)
    return sorted(cut)


def stratified_rows(w: inputs.Workload, all_units: bool = True, edge_units=None, tile: int = 128,
                    extra: int = 16, seed: int = 0):
    """Flat query rows spread over the problem's structure rather than uniformly:
      * one seeded row of every (b, kv-head) unit (all_units);
      * for each unit in `edge_units`: the first and last row of every `tile`-row query tile and
        the unit's last row (every query tile boundary of those units);
      * `extra` seeded random rows."""
    rng = np.random.default_rng(seed)
    U = w.B * w.Hkv
    rows = set()
    if all_units:
        for u in range(U):
            a, e = unit_rows(w, u)
            rows.add(int(rng.integers(a, e)))
    for u in ([] if edge_units is None else edge_units):
        a, e = unit_rows(w, int(u))
        for t0 in range(a, e, tile):
            rows.add(t0)
            rows.add(min(t0 + tile, e) - 1)
    total = w.B * w.Hq * w.Sq
    rows |= set(rng.choice(total, size=min(extra, total), replace=False).tolist())
    rows |= {0, total - 1}
    return np.array(sorted(rows), dtype=np.int64)
