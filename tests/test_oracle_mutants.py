"""The oracle's pins catch plausible mistakes in the oracle.

Each mutant below plants one mistake of the kind a restatement of the pages
could contain: a dropped term, a wrong sign, an off-by-one, a wrong index, or
a transposed operand.  The mistake goes into a copy of ``oracle/`` in a
temporary directory; the original is never touched.  Then
``tests/test_oracle_pins.py`` runs in a subprocess whose ``import oracle``
resolves to that copy.  The pins pass on an unmutated copy built the same
way, and some pin must fail on every mutant.  A mutant that survives names a
mistake the pins cannot see.  CPU only: gcc and the fp64 oracle.
"""
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = os.path.join("tests", "test_oracle_pins.py")
C, PY = "attn_oracle.c", "__init__.py"

# (name, file, [(text, replacement), ...], the mistake it stands for)
MUTANTS = [
    # --- attention: the causal mask and its alignment
    ("causal_excludes_diagonal", C, [("                last = ctx + i;\n", "                last = ctx + i - 1;\n")],
     "the query does not see its own key"),
    ("causal_flag_ignored", C, [("if (causal && ctx + i < last)", "if (ctx + i < last)")],
     "non-causal calls (the cascade prefix) masked as causal"),
    ("top_left_alignment", C, [("const int64_t ctx = kv_len - q_len;", "const int64_t ctx = 0;")],
     "the causal mask aligned top-left instead of bottom-right"),
    ("request_bounds_inclusive", C, [("t < cu_seqlens_q[r + 1]))", "t <= cu_seqlens_q[r + 1]))")],
     "a request's first token is credited to the request before it"),
    # --- attention: heads and the paged address
    ("gqa_head_modulo", C, [("const int g = h / G;", "const int g = h % Hkv;")],
     "query heads interleaved over KV heads instead of grouped"),
    ("logical_block_for_keys", C, [("const int64_t k_off = (((int64_t)phys * bs",
                                    "const int64_t k_off = (((int64_t)(j / bs) * bs")],
     "keys read from the logical block index, not the block table's entry"),
    ("cache_layout_head_major", C, [("const int64_t k_off = (((int64_t)phys * bs + j % bs) * Hkv + g) * D;",
                                     "const int64_t k_off = (((int64_t)phys * Hkv + g) * bs + j % bs) * D;"),
                                    ("const int64_t v_off = (((int64_t)phys * bs + j % bs) * Hkv + g) * D;",
                                     "const int64_t v_off = (((int64_t)phys * Hkv + g) * bs + j % bs) * D;")],
     "the cache read as [block, head, row, d] instead of [block, row, head, d]"),
    ("values_from_key_cache", C, [("load_elem(v_cache, v_off + d, kv_dtype)", "load_elem(k_cache, v_off + d, kv_dtype)")],
     "P multiplied by K instead of V"),
    # --- attention: the softmax
    ("softmax_scale_dropped", C, [("s[j] = softmax_scale * dot;", "s[j] = dot;")],
     "the logits not scaled"),
    ("max_not_subtracted", C, [("const double e = exp(s[j] - M);", "const double e = exp(s[j]);")],
     "exponentials taken without the running max"),
    ("lse_without_max", C, [("lse[oi * Hq + h] = M + log(L);", "lse[oi * Hq + h] = log(L);")],
     "the max dropped from the log-sum-exp"),
    ("output_not_normalised", C, [("for (int d = 0; d < D; ++d) o[d] /= L;", "")],
     "the output not divided by the softmax sum"),
    # --- attention: variants
    ("window_left_off_by_one", C, [("first = ctx + i - window_left;", "first = ctx + i - window_left + 1;")],
     "the sliding window one key short on the left"),
    ("window_right_off_by_one", C, [("last = ctx + i + window_right;", "last = ctx + i + window_right - 1;")],
     "the sliding window one key short on the right"),
    ("window_right_ignored", C, [("if (window_right >= 0 && ctx + i + window_right < last)",
                                  "if (0 && ctx + i + window_right < last)")],
     "the right window bound ignored"),
    ("softcap_unscaled", C, [("softcap * tanh(s[j] / softcap)", "softcap * tanh(s[j])")],
     "the soft cap applied to s instead of s / c"),
    ("softcap_before_scale", C, [("s[j] = softmax_scale * dot;\n                if (softcap > 0.0)\n                    s[j] = softcap * tanh(s[j] / softcap);",
                                  "s[j] = dot;\n                if (softcap > 0.0)\n                    s[j] = softcap * tanh(s[j] / softcap);\n                s[j] *= softmax_scale;")],
     "the soft cap applied to q . k before the scale"),
    ("sink_dropped", C, [("double L = z == -INFINITY ? 0.0 : exp(z - M);", "double L = 0.0;")],
     "the sink logit left out of the normalisation"),
    ("q_scale_dropped", C, [("qv[d] = load_elem(q, q_off + d, q_dtype) * q_scale;",
                             "qv[d] = load_elem(q, q_off + d, q_dtype);")],
     "an e4m3 query's scale ignored"),
    ("k_scale_dropped", C, [("(load_elem(k_cache, k_off + d, kv_dtype) * k_scale)",
                             "(load_elem(k_cache, k_off + d, kv_dtype))")],
     "the K cache's scale ignored"),
    ("v_scale_dropped", C, [("(load_elem(v_cache, v_off + d, kv_dtype) * v_scale)",
                             "(load_elem(v_cache, v_off + d, kv_dtype))")],
     "the V cache's scale ignored"),
    # --- the log-sum-exp merge
    ("merge_weights_swapped", C, [("w1 * o1[i * D + d] + w2 * o2[i * D + d]", "w2 * o1[i * D + d] + w1 * o2[i * D + d]")],
     "each state weighted by the other's share"),
    ("merge_lse_without_max", C, [("const double l = mx + log(exp(a - mx) + exp(b - mx));",
                                   "const double l = log(exp(a - mx) + exp(b - mx));")],
     "the max dropped from the merged log-sum-exp"),
    ("merge_weights_unnormalised", C, [("const double w1 = exp(a - l), w2 = exp(b - l);",
                                        "const double w1 = exp(a - mx), w2 = exp(b - mx);")],
     "the merge weights taken relative to the max, not to the merged lse"),
    ("merge_empty_states_unhandled", C, [("if (a == -INFINITY && b == -INFINITY) {", "if (0) {")],
     "two empty states merged by the general formula"),
    # --- e4m3 decoding and encoding
    ("e4m3_bias_8", C, [("v = ldexp((double)(8 + m), e - 10);", "v = ldexp((double)(8 + m), e - 11);")],
     "exponent bias 8 instead of 7"),
    ("e4m3_subnormal_scale", C, [("v = ldexp((double)m, -9);", "v = ldexp((double)m, -10);")],
     "subnormals on the wrong grid"),
    ("e4m3_ties_away", C, [("double mant = nearbyint((2.0 * f - 1.0) * 8.0);", "double mant = round((2.0 * f - 1.0) * 8.0);")],
     "ties rounded away from zero instead of to even"),
    ("e4m3_saturates_to_nan", C, [("if (a >= 448.0)\n        return (uint8_t)(sign | 0x7E);",
                                   "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7F);")],
     "out-of-range values mapped to NaN instead of +-448"),
    ("e4m3_subnormal_ties_away", C, [("double m = nearbyint(a * 512.0);", "double m = round(a * 512.0);")],
     "ties in the subnormal range rounded away from zero"),
    ("e4m3_sign_lost", C, [("uint8_t sign = signbit(x) ? 0x80 : 0x00;", "uint8_t sign = 0x00;")],
     "negative values encoded as positive"),
    ("fp16_exponent_bias", C, [("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);")],
     "fp16 decoded with bias 14"),
    # --- the slot_mapping write
    ("kv_write_scale_multiplies", C, [("oracle_e4m3_from_float(kx / k_scale)", "oracle_e4m3_from_float(kx * k_scale)")],
     "the cache stores x * scale instead of x / scale"),
    ("kv_write_values_use_key_scale", C, [("oracle_e4m3_from_float(vx / v_scale)", "oracle_e4m3_from_float(vx / k_scale)")],
     "the e4m3 V cache quantised with the key scale"),
    ("kv_write_skips_slot_zero", C, [("        if (slot < 0)\n            continue;", "        if (slot <= 0)\n            continue;")],
     "slot 0 treated as padding"),
    ("kv_write_v_gets_keys", C, [("memcpy((char *)v_cache + dst * cb, (const char *)value + src * sb",
                                  "memcpy((char *)v_cache + dst * cb, (const char *)key + src * sb")],
     "the V cache written with keys"),
    ("kv_write_row_zero", C, [("const int64_t blk = slot / bs, row = slot % bs;", "const int64_t blk = slot / bs, row = 0;")],
     "every token of a block written to its first row"),
    # --- the dense brute-force formulation
    ("dense_causal_strict", PY, [("mask &= loc_k[None, :] <= pos\n", "mask &= loc_k[None, :] < pos\n")],
     "the dense mask hides the diagonal"),
    ("dense_gqa_modulo", PY, [("        g = h // G\n", "        g = h % Hkv\n")],
     "the dense formulation interleaves the heads"),
    ("dense_context_dropped", PY, [("ctx_q[cq[r]:cq[r + 1]] = (ck[r + 1] - ck[r]) - (cq[r + 1] - cq[r])",
                                    "ctx_q[cq[r]:cq[r + 1]] = 0")],
     "the dense formulation aligns the mask top-left"),
]

_BOOT = r"""
import sys
sys.path.insert(0, sys.argv[1])
import oracle, oracle.build
assert oracle.__file__.startswith(sys.argv[1]), oracle.__file__
try:
    oracle.build.build_oracle(force=True)
except Exception as e:
    print("BUILD FAILED", e)
    sys.exit(90)
import pytest
sys.exit(pytest.main([sys.argv[2], "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"]))
"""


def _copy_oracle(dst, edits=()):
    """A copy of the oracle package in dst/oracle with the edits applied."""
    pkg = os.path.join(dst, "oracle")
    os.makedirs(pkg)
    for name in (C, "build.py", PY):
        with open(os.path.join(ORACLE, name), encoding="utf-8") as f:
            src = f.read()
        for fname, old, new in edits:
            if fname == name:
                assert src.count(old) == 1, "mutation text not found once in %s: %r" % (name, old)
                src = src.replace(old, new)
        with open(os.path.join(pkg, name), "w", encoding="utf-8") as f:
            f.write(src)


def _run(dst):
    env = dict(os.environ, OMP_NUM_THREADS="1", PYTHONDONTWRITEBYTECODE="1")
    p = subprocess.run([sys.executable, "-c", _BOOT, dst, PINS], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=600)
    caught = re.findall(r"^(?:FAILED|ERROR) \S+::(\S+)", p.stdout, re.M)
    return p.returncode, caught[0] if caught else None, p.stdout[-2000:] + p.stderr[-2000:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    if shutil.which(os.environ.get("CC", "gcc")) is None:
        pytest.skip("no C compiler")
    base = tmp_path_factory.mktemp("oracle_mutants")
    jobs = {"control": []}
    for name, fname, subs, _ in MUTANTS:
        jobs[name] = [(fname, old, new) for old, new in subs]
    dirs = {}
    for name, edits in jobs.items():
        dirs[name] = str(base / name)
        _copy_oracle(dirs[name], edits)
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        futs = {name: ex.submit(_run, d) for name, d in dirs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmutated_copy_passes_every_pin(outcomes):
    rc, caught, log = outcomes["control"]
    assert rc == 0, log


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_some_pin_catches_the_mutant(outcomes, name):
    rc, caught, log = outcomes[name]
    assert rc != 90, "the mutant did not compile:\n" + log
    assert rc == 1 and caught, "no pin caught mutant %s:\n%s" % (name, log)
