"""The oracle's pins must reject a wrong oracle.

Each case plants one plausible mistake in a copy of the oracle's C source: a dropped term, a wrong
sign, index or constant, a transposed operand, a wrong rounding, saturation or packing rule.  It
builds that copy with the oracle's own compiler flags and runs the oracle pin tests against it in
a subprocess (``ORACLE_LIB`` makes the oracle load that build).  At least one pin must fail, and
that among the pins that use no library routine (golden tables, closed forms, invariants and
brute force; the comparisons with torch's attention, logsumexp and FP8 cast and with CUDA's host
conversions are left out), so the mistake is caught independently of any library.  The
unmodified copy, built and run the same way, must pass them all, so a failure comes from the
planted mistake and not from the harness.  Every planted mistake keeps each access in bounds, so
a pin, not a crash, has to catch it.  The builds go to ``tests/_mutants/`` (git-ignored)."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

pytest.importorskip("mpmath")   # the brute-force pins, some of which must catch the layout mistakes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")
WORK = os.path.join(ROOT, "tests", "_mutants")
SOURCES = ("attn_ref.c", "nvfp4_ref.c")
PINS = ["tests/test_oracle_attention.py", "tests/test_oracle_nvfp4.py", "tests/test_oracle_nvfp4_scaled.py"]
# the pins that compare with a library routine (torch SDPA / logsumexp, torch's FP8 cast, CUDA's
# host conversions): deselected, so that what remains is library-free
LIBRARY_PINS = ("matches_library_sdpa", "gqa_equals_repeated_heads", "ragged_equals_truncated_dense",
                "causal_matches_masked_sdpa", "causal_ragged_is_relative_to_each_length", "torch_cast",
                "cuda_host_cvt")

# name: (source file, text, replacement, which occurrence: None = the only one, "all", or an index)
MUTANTS = {
    # attention: softmax(scale * Q K^T) V and LSE
    "scale_dropped": ("attn_ref.c", "s[j] = scale * acc;", "s[j] = acc;", None),
    "exponent_sign_flipped": ("attn_ref.c", "s[j] = exp(s[j] - m);", "s[j] = exp(m - s[j]);", None),
    "normalisation_dropped": ("attn_ref.c", "orow[d] /= l;", "orow[d] /= 1.0;", None),
    "lse_max_dropped": ("attn_ref.c", "lse[t] = m + log(l);", "lse[t] = log(l);", None),
    "empty_lse_zero": ("attn_ref.c", "lse[t] = -INFINITY;", "lse[t] = 0.0;", None),
    "k_transposed": ("attn_ref.c", "bf16_bits_to_double(kbase[j * D + d])", "bf16_bits_to_double(kbase[d * n + j])", None),
    "v_rows_reversed": ("attn_ref.c", "const uint16_t* vrow = vbase + j * D;",
                        "const uint16_t* vrow = vbase + (n - 1 - j) * D;", None),
    "query_row_of_head": ("attn_ref.c", "const uint16_t* qrow = q + r * D;",
                          "const uint16_t* qrow = q + (r - i) * D;", None),
    "gqa_head_modulo": ("attn_ref.c", "const int64_t kvh = hq / group;", "const int64_t kvh = hq % Hkv;", None),
    "batch_head_transposed": ("attn_ref.c", "(b * Hkv + kvh)", "(kvh * B + b)", "all"),
    "seqlens_ignored": ("attn_ref.c", "int64_t n = seqlens_k ? seqlens_k[b] : Skv;", "int64_t n = Skv;", None),
    "causal_top_left": ("attn_ref.c", "const int64_t last = i + n - Sq;", "const int64_t last = i;", None),
    "causal_off_by_one": ("attn_ref.c", "n = last < 0 ? 0 : (last + 1 < n ? last + 1 : n);",
                          "n = last < 0 ? 0 : (last < n ? last : n);", None),
    "raw_qk_transposed": ("attn_ref.c", "bf16_bits_to_double(k[(int64_t)j * D + d])",
                          "bf16_bits_to_double(k[(int64_t)d * Skv + j])", None),
    "raw_qk_scaled": ("attn_ref.c", "s[(int64_t)i * Skv + j] = acc;", "s[(int64_t)i * Skv + j] = acc * 0.125;", None),
    # NVFP4: E4M3 block scales, E2M1 elements, per-tensor scale, packing
    "e4m3_subnormal_exponent": ("nvfp4_ref.c", "ldexp((double)m, -9)", "ldexp((double)m, -10)", None),
    "e4m3_bias": ("nvfp4_ref.c", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", None),
    "e4m3_saturates_to_nan": ("nvfp4_ref.c", "return 0x7E;", "return 0x7F;", None),
    "e4m3_ties_away": ("nvfp4_ref.c", "err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)",
                       "err <= best_err", 0),
    "e2m1_ties_away": ("nvfp4_ref.c", "err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)",
                       "err <= best_err", 1),
    "e2m1_table": ("nvfp4_ref.c", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}",
                   "{0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 4.0, 6.0}", None),
    "e2m1_sign_dropped": ("nvfp4_ref.c", "return (code & 8) ? -m : m;", "return m;", None),
    "e2m1_saturation_sign_dropped": ("nvfp4_ref.c", "return (uint8_t)(7 | (signbit(v) ? 8 : 0));",
                                     "return (uint8_t)7;", None),
    "block_scale_divisor": ("nvfp4_ref.c", "(6.0 * (double)s_g)", "(4.0 * (double)s_g)", None),
    "block_amax_half_block": ("nvfp4_ref.c", "for (int i = 0; i < 16; ++i) {\n            const float a = fabsf(xb[i]);",
                              "for (int i = 0; i < 8; ++i) {\n            const float a = fabsf(xb[i]);", None),
    "element_divisor_without_tensor_scale": ("nvfp4_ref.c", "oracle_e4m3_decode(sc) * (double)s_g",
                                             "oracle_e4m3_decode(sc)", None),
    "tensor_scale_divisor": ("nvfp4_ref.c", "(double)amax / 2688.0", "(double)amax / 448.0", None),
    "nibble_order_swapped": ("nvfp4_ref.c", "if ((e & 1) == 0)", "if ((e & 1) == 1)", None),
}


def _plant(src, text, repl, which):
    n = src.count(text)
    assert n >= 1, f"anchor not found: {text!r}"
    if which == "all":
        return src.replace(text, repl)
    if which is None:
        assert n == 1, f"anchor not unique ({n}): {text!r}"
        which = 0
    assert which < n
    pos = -1
    for _ in range(which + 1):
        pos = src.index(text, pos + 1)
    return src[:pos] + repl + src[pos + len(text):]


def _build(name, mutant):
    d = os.path.join(WORK, name)
    if os.path.isdir(d):
        shutil.rmtree(d)
    os.makedirs(d)
    shutil.copy(os.path.join(ORACLE_DIR, "oracle.h"), d)
    for s in SOURCES:
        with open(os.path.join(ORACLE_DIR, s)) as f:
            text = f.read()
        if mutant is not None and mutant[0] == s:
            text = _plant(text, *mutant[1:])
        with open(os.path.join(d, s), "w") as f:
            f.write(text)
    lib = os.path.join(d, "liboracle.so")
    subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-Wall", "-o", lib]
                   + [os.path.join(d, s) for s in SOURCES] + ["-lm"], check=True, capture_output=True)
    return lib


def _run_pins(name, mutant):
    lib = _build(name, mutant)
    env = dict(os.environ, ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                        "-k", " and ".join(f"not {n}" for n in LIBRARY_PINS)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.fixture(scope="module")
def outcomes():
    jobs = {"unmodified": None, **MUTANTS}
    with ThreadPoolExecutor(max_workers=max(1, min(8, (os.cpu_count() or 2) // 2))) as ex:
        futs = {k: ex.submit(_run_pins, k, m) for k, m in jobs.items()}
        res = {k: f.result() for k, f in futs.items()}
    shutil.rmtree(WORK, ignore_errors=True)
    return res


def test_unmodified_copy_passes_the_pins(outcomes):
    rc, tail = outcomes["unmodified"]
    assert rc == 0, tail
    assert "deselected" in tail, tail   # the library pins were left out, the rest ran


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_reject_planted_mistake(outcomes, name):
    rc, tail = outcomes[name]
    # 1 = tests ran and at least one failed; anything else (0 = all passed, 2+ = the run broke,
    # negative = a crash) does not show that a pin caught the mistake
    assert rc == 1, f"{name}: pins returned {rc}\n{tail}"
