"""GPU edge and degenerate cases through the C ABI: empty problems; a zero query, where every
visible key has the same score, so O is the plain mean of the visible value rows and LSE = ln n
(a closed form that does not depend on the keys), on every kernel path including the causal mask;
shapes at the edges of the dispatch and the mask against the oracle; and an output of more than
2^31 elements."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_tensor_cores_gb300 import inputs
from attn_util import check_o_lse, run_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_tensor_cores_gb300 as F
    F.load()
    return F


@pytest.mark.parametrize("B,Sq,D", [(0, 1, 128), (2, 0, 64), (0, 300, 64), (0, 1, 512)])
def test_empty_problem_is_a_no_op(F, B, Sq, D):
    q = torch.zeros(max(B, 1), 4, max(Sq, 1), D, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(max(B, 1), 2, 16, D, dtype=torch.bfloat16, device="cuda")
    out = torch.full_like(q, float("nan"))
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    lib = F.load()
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    launches = F.fmha_launch_count()
    assert lib.fmha_fwd(P(q), P(k), P(k), P(out), P(lse), B, 4, 2, Sq, 16, D, 0.125, s) == F.FMHA_OK
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    assert F.fmha_launch_count() == launches      # nothing launched
    assert torch.isnan(out).all() and torch.isnan(lse).all()   # nothing written


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,causal,splits", [
    (2, 8, 2, 1, 3000, 128, False, 0),     # decode, split
    (2, 32, 8, 4, 500, 64, True, 0),       # multi-token decode, causal
    (1, 2, 2, 300, 700, 64, False, None),  # row tiles D = 64
    (1, 2, 1, 400, 400, 128, True, 0),     # row tiles D = 128, causal
    (2, 128, 1, 1, 700, 512, False, 0),    # wide head, split
    (1, 16, 1, 2, 300, 512, True, 1),      # wide head, whole units, causal
])
def test_zero_query_gives_mean_of_visible_values(F, B, Hq, Hkv, Sq, Skv, D, causal, splits):
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 95)
    _, k, v, _ = w.make("cuda")
    q = torch.zeros(B, Hq, Sq, D, dtype=torch.bfloat16, device="cuda")
    kw = {} if splits is None else {"num_splits": splits}
    if causal:
        kw["causal"] = True
    res = run_attention(F, q, k, v, w.scale, **kw)
    vv = v.double().cpu().numpy()
    g = Hq // Hkv
    o_ref = np.zeros((B * Hq * Sq, D))
    l_ref = np.zeros(B * Hq * Sq)
    for r in range(B * Hq * Sq):
        b, hq, i = r // (Hq * Sq), (r // Sq) % Hq, r % Sq
        n = min(Skv, i + Skv - Sq + 1) if causal else Skv   # bottom-right aligned
        o_ref[r] = vv[b, hq // g, :n].mean(axis=0)
        l_ref[r] = math.log(n)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "zero query")


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D,causal,splits", [
    (1, 17, 1, 1, 300, 64, False, 0),      # G = 17: the first shape on the row-tile path (17 of 128 rows)
    (1, 17, 1, 1, 300, 128, False, None),  # the same at D = 128, whole units
    (1, 2, 2, 200, 1, 64, False, 0),       # row tiles, a single key
    (1, 2, 2, 200, 1, 128, True, 0),       # row tiles, one key: only the last query sees it
    (2, 8, 2, 4, 2, 128, True, 0),         # decode (16 columns), causal with Sq > Skv: queries that see nothing
    (1, 16, 1, 1, 1, 512, False, 0),       # wide head, a single key
    (1, 32, 1, 4, 2, 512, True, 1),        # wide head, causal with Sq > Skv, whole units
])
def test_boundary_shapes_against_oracle(F, B, Hq, Hkv, Sq, Skv, D, causal, splits):
    """Shapes at the edges of the dispatch and of the mask: the decode / row-tile boundary, one key per
    head on every path, and causal queries with no visible key (O = 0, LSE = -inf)."""
    w = inputs.Workload("t", B, Hq, Hkv, Sq, Skv, D, 1.0, "bf16", 96)
    q, k, v, _ = w.make("cuda")
    kw = {} if splits is None else {"num_splits": splits}
    if causal:
        kw["causal"] = True
    res = run_attention(F, q, k, v, w.scale, **kw)
    o_ref, l_ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), w.scale, causal=causal)
    check_o_lse(res["o"], res["lse"], o_ref, l_ref, "boundary shape")
    if causal and Sq > Skv:
        assert np.isneginf(l_ref).any() and np.all(res["o"][np.isneginf(l_ref)] == 0.0)


def test_output_beyond_2_to_31_elements(F):
    """A prefill whose output holds more than 2^31 elements (Hq = Hkv = 72, Sq = 262144, one 128-key
    tile, D = 128: 2.4e9 elements), so every output offset past 2^31 must be formed in 64 bits.  Rows on
    both sides of the 2^31-element boundary and at the very end, against the oracle head by head."""
    H, Sq, Skv, D = 72, 262144, 128, 128
    g = torch.Generator(device="cuda").manual_seed(96)
    q = torch.randn(1, H, Sq, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(1, H, Skv, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(1, H, Skv, D, generator=g, device="cuda").to(torch.bfloat16)
    out = torch.empty(1, H, Sq, D, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, H, Sq, dtype=torch.float32, device="cuda")
    scale = 1.0 / math.sqrt(D)
    F.fmha_fwd(q, k, v, out, lse, scale)
    torch.cuda.synchronize()
    assert F.fmha_check_status() == 0
    n_rows = H * Sq
    boundary = (1 << 31) // D            # the first row whose elements start at offset 2^31
    rng = np.random.default_rng(7)
    rows = np.unique(np.concatenate([[0, boundary - 2, boundary - 1, boundary, boundary + 1, n_rows - 1],
                                     rng.integers(boundary, n_rows, 24)]))
    rows_t = torch.from_numpy(rows).cuda()
    o = out.view(-1, D)[rows_t].float().cpu().numpy()
    l = lse.view(-1)[rows_t].cpu().numpy()
    qs = q.view(-1, D)[rows_t].cpu()
    o_ref = np.zeros((len(rows), D))
    l_ref = np.zeros(len(rows))
    kc, vc = k.cpu(), v.cpu()
    for h in np.unique(rows // Sq):
        sel = np.where(rows // Sq == h)[0]
        oh, lh = oracle.attention(qs[torch.from_numpy(sel)].view(1, 1, len(sel), D), kc[:, h:h + 1], vc[:, h:h + 1], scale)
        o_ref[sel], l_ref[sel] = oh, lh
    check_o_lse(o, l, o_ref, l_ref, "output beyond 2^31 elements")
    del q, k, v, out, lse
    torch.cuda.empty_cache()
