"""Planted mistakes in the oracle: every one must make a pin fail.

The oracle's pins are only worth something if a plausible slip in the oracle
trips one of them. Each entry below rewrites one spot of a copy of
``oracle/oracle.c`` -- a reversed loop, a dropped term, an index off by one,
a rounding rule changed -- and the pin suites (``test_oracle_pins.py`` and
``test_oracle_gemm_pins.py``) run against that copy in its own temporary
directory. Everything happens on the CPU; the CUDA library is not involved,
and the real oracle is never modified.

If the oracle's source changes so that an anchor below no longer matches,
this test fails: update the anchor together with the change.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# name: (text in oracle.c, its planted replacement)
MUTATIONS = {
    # plan: deficits filled in descending rank order
    "pour_rank_desc": ("for (r = 0; r < R; ++r) {\n      int64_t need",
                       "for (r = R - 1; r >= 0; --r) {\n      int64_t need"),
    # plan: the keep budget never shrinks
    "keep_no_budget_dec": ("budget -= k_e;", ";"),
    # plan: exclusive instead of inclusive cu_seqlens
    "cu_exclusive": ("run += c[(int64_t)r * G + j];\n      cu[(int64_t)r * G + j] = (int32_t)run;",
                     "cu[(int64_t)r * G + j] = (int32_t)run;\n      run += c[(int64_t)r * G + j];"),
    # plan: home rank by modulo instead of contiguous blocks
    "home_mod": ("load[e / per] += counts[e];", "load[e % R] += counts[e];"),
    # plan: the inference fallback ignored
    "fallback_ignored": ("if (b >= B && fallback) {", "if (0) {"),
    # plan: a fallback piece counted in the last slot row instead of its home row
    "fallback_row_slot": ("      c[(int64_t)pieces[j].r * G + pieces[j].e] = pieces[j].hi - pieces[j].lo;\n"
                          "      continue;",
                          "      c[(int64_t)pieces[j].r * G + E + B - 1] += pieces[j].hi - pieces[j].lo;\n"
                          "      continue;"),
    # combine: separate multiply and add instead of fma
    "combine_mul_add": ("acc = fmaf(w[t * K + k], orc_bf16_to_f32(y[row * H + h]), acc);",
                        "acc = acc + (float)((double)w[t * K + k] * orc_bf16_to_f32(y[row * H + h]));"),
    # combine: k summed in reverse order
    "combine_k_reverse": ("int64_t row = dst_pos[t * K + k];\n        acc",
                          "int64_t row = dst_pos[t * K + (K - 1 - k)];\n        acc"),
    # bf16 rounding: ties away from zero instead of to even
    "rne_ties_up": ("(low == 0x8000u && (keep_hi & 1u))", "(low == 0x8000u)"),
    # reduce_grad: slots added in reverse (rank, slot) order
    "reduce_order_rev": ("for (s = 0; s < R * B; ++s) {\n      const float* srow;",
                         "for (s = R * B - 1; s >= 0; --s) {\n      const float* srow;"),
    # prefetch: slot 0 copies the next expert's weights
    "prefetch_off_by_one": ("memcpy(slot + (int64_t)s * nbytes, home + (int64_t)slot_expert[s] * nbytes",
                            "memcpy(slot + (int64_t)s * nbytes, home + (int64_t)(slot_expert[s] + (s == 0))"
                            " * nbytes"),
    # prefetch: an out-of-range slot map accepted
    "prefetch_no_check": ("if (slot_expert[s] < -1 || slot_expert[s] >= E) return ORC_BAD_ROUTING;\n"
                          "  for (s = 0; s < R * B; ++s)\n    if (slot_expert[s] >= 0)",
                          "for (s = 0; s < R * B; ++s)\n    if (slot_expert[s] >= 0 && slot_expert[s] < E)"),
    # dispatch backward: k summed in reverse order
    "dbwd_k_reverse": ("for (k = 0; k < K; ++k) acc = acc + orc_bf16_to_f32(dbuf[(int64_t)dst_pos[t * K + k] * H + h]);",
                       "for (k = K - 1; k >= 0; --k) acc = acc + orc_bf16_to_f32(dbuf[(int64_t)dst_pos[t * K + k] * H + h]);"),
    # combine backward: w * dout rounded once to bf16 from double, not via fp32
    "cbwd_single_round": ("const float p = wk * d;\n        dy[row * H + h] = orc_f32_to_bf16(p);",
                          "const double pe = (double)wk * d; int ex; double m = frexp(fabs(pe), &ex); "
                          "double q = ldexp(nearbyint(ldexp(m, 8)), ex - 8); const float p = (float)(pe < 0 ? -q : q);\n"
                          "        dy[row * H + h] = orc_f32_to_bf16(p);"),
    # combine backward: dw dotted with the wrong buffer row
    "cbwd_dw_wrong_row": ("acc += (double)d * (double)orc_bf16_to_f32(y[row * H + h]);",
                          "acc += (double)d * (double)orc_bf16_to_f32(y[(row ^ 1) * H + h]);"),
    # grouped GEMM: slot rows use the next slot's weights
    "gemm_slot_off_by_one": ("w_slot + ((int64_t)r * B + (j - E)) * H * Hp",
                             "w_slot + ((int64_t)r * B + (j - E + 1) % B) * H * Hp"),
    # grouped GEMM: slot rows served by home weights
    "gemm_slot_uses_home": ("W = j < E ? w_home + (int64_t)j * H * Hp :",
                            "W = j < E + B ? w_home + (int64_t)(j % E) * H * Hp :"),
    # grouped GEMM: a row on a group boundary assigned to the earlier group
    "gemm_group_lt": ("while (cu[(int64_t)r * G + j] <= i) ++j;", "while (cu[(int64_t)r * G + j] < i) ++j;"),
    # grouped GEMM: weights read transposed
    "gemm_transposed_w": ("const uint16_t* wrow = W + h * Hp;\n      for (n = 0; n < Hp; ++n) out[n] += xv * "
                          "(double)orc_bf16_to_f32(wrow[n]);",
                          "for (n = 0; n < Hp; ++n) out[n] += xv * (double)orc_bf16_to_f32(W[(n * H + h) % (H * Hp)]);"),
    # grouped GEMM: the last term of the sum dropped
    "gemm_drop_last_h": ("for (h = 0; h < H; ++h) {\n      const double xv", "for (h = 0; h < H - 1; ++h) {\n      const double xv"),
}

PIN_SUITES = ["tests/test_oracle_pins.py", "tests/test_oracle_gemm_pins.py"]


def _copy_tree(dst):
    skip = shutil.ignore_patterns("*.so", "*.so.tmp*", "__pycache__", "_build", "csrc", "golden_out")
    for part in ("oracle", "tests", "load_balancing_topk_gb300"):
        shutil.copytree(os.path.join(ROOT, part), os.path.join(dst, part), ignore=skip)


def _pins_fail_on(name, src, base):
    old, new = MUTATIONS[name]
    d = os.path.join(base, name)
    _copy_tree(d)
    with open(os.path.join(d, "oracle", "oracle.c"), "w") as f:
        f.write(src.replace(old, new, 1))
    r = subprocess.run([sys.executable, "-m", "pytest", *PIN_SUITES, "-x", "-q", "-p", "no:cacheprovider"],
                       cwd=d, capture_output=True, text=True, timeout=600)
    return name, r.returncode != 0


def test_every_planted_mistake_is_caught(tmp_path):
    with open(os.path.join(ROOT, "oracle", "oracle.c")) as f:
        src = f.read()
    missing = [n for n, (old, _) in MUTATIONS.items() if src.count(old) != 1]
    assert not missing, f"anchors no longer match oracle.c: {missing}"
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda n: _pins_fail_on(n, src, str(tmp_path)), MUTATIONS))
    uncaught = [n for n, caught in results if not caught]
    assert not uncaught, f"planted mistakes no pin caught: {uncaught}"
