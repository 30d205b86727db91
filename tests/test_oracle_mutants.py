"""Planted mistakes: a copy of the oracle's C source with one plausible bug
(the page's own bug table -- no slot filter, no truncation, repeat instead
of repeat_interleave, scale after the softmax -- plus index, operand and
rounding slips) must fail at least one pin.  This shows the pins constrain
every part of the oracle.  CPU only; each mutant runs in a child process so
that one which reads out of bounds cannot take the test run down."""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "no_slot_filter": [("if (slot < 0) continue;", "if (slot < 0) slot += num_blocks * block_size;")],
    "block_offset_transposed": [("const int64_t dst = (blk * block_size + off) * row_elems;",
                                 "const int64_t dst = (off * num_blocks + blk) * row_elems;")],
    "no_truncation": [("for (int64_t t = 0; t < n; ++t) {\n        const int64_t phys",
                       "for (int64_t t = 0; t < nb * bs; ++t) {\n        const int64_t phys"),
                      ("for (int64_t t = 0; t < n; ++t) {\n          const int64_t phys",
                       "for (int64_t t = 0; t < nb * bs; ++t) {\n          const int64_t phys"),
                      ("(double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1))",
                       "(double *)malloc(sizeof(double) * (size_t)(nb * bs + 1))"),
                      ("for (int64_t t = 0; t < n; ++t) {\n        s[t] = exp",
                       "for (int64_t t = 0; t < nb * bs; ++t) {\n        s[t] = exp")],
    "gqa_repeat_not_interleave": [("const int64_t kvh = h / group;", "const int64_t kvh = h % KVH;")],
    "scale_after_softmax": [("s[t] = scale * dot;", "s[t] = dot;"),
                            ("store_elem(out, qoff + d, dtype, acc / denom);",
                             "store_elem(out, qoff + d, dtype, scale * acc / denom);")],
    "scale_dropped": [("s[t] = scale * dot;", "s[t] = dot;")],
    "table_index_wrong": [("const int64_t phys = tbl[t / bs];\n        const int64_t row",
                           "const int64_t phys = tbl[(t / bs) % (nb > 1 ? nb - 1 : 1)];\n        const int64_t row")],
    "row_in_block_wrong": [("const int64_t row = ((phys * bs + t % bs) * KVH + kvh) * D;\n        double dot",
                            "const int64_t row = ((phys * bs + (bs - 1 - t % bs)) * KVH + kvh) * D;\n        double dot")],
    "k_from_v_cache": [("load_elem(k_cache, row + d, dtype)", "load_elem(v_cache, row + d, dtype)")],
    "no_max_subtraction": [("s[t] = exp(s[t] - m);", "s[t] = exp(s[t]);")],
    "exp_sign_flipped": [("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);")],
    "not_normalised": [("store_elem(out, qoff + d, dtype, acc / denom);",
                        "store_elem(out, qoff + d, dtype, acc / (double)n);")],
    "round_by_truncation": [("double r = nearbyint(ldexp(x, -q));", "double r = trunc(ldexp(x, -q));")],
    "subnormals_not_fixed_quantum": [("if (q < emin - p + 1) q = emin - p + 1;", "")],
    "prefill_top_left_causal": [("const int64_t p = n - qlen + i;", "const int64_t p = i;")],
    "prefill_excludes_self": [("const int64_t lim = p + 1;", "const int64_t lim = p > 0 ? p : 1;")],
    "prefill_no_causal_mask": [("const int64_t lim = p + 1;", "const int64_t lim = n;")],
    "prefill_ignores_row_offsets": [("const int64_t q_row = cu_seqlens_q[b] + i;",
                                     "const int64_t q_row = i;")],
    "prefill_gqa_repeat": [("const int64_t g = h / heads_per_kv;", "const int64_t g = h % KVH;")],
    "prefill_scale_dropped": [("w[t] = qk * scale;", "w[t] = qk;")],
    "empty_context_not_zero": [("for (int64_t d = 0; d < D; ++d) store_elem(out, qoff + d, dtype, 0.0);",
                                "for (int64_t d = 0; d < D; ++d) store_elem(out, qoff + d, dtype, 1.0);")],
}

CHILD = r"""
import sys, traceback
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle
from oracle_pins import ALL_PINS
lib = oracle.load({so!r})
failed = []
for pin in ALL_PINS:
    try:
        pin(lib)
    except Exception:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
"""


def _run_mutant(name, edits, tmp):
    with open(oracle._SRC) as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: mutation site not found once: {old!r}"
        src = src.replace(old, new)
    d = os.path.join(tmp, name)
    os.makedirs(d)
    c_path = os.path.join(d, "mutant.c")
    with open(c_path, "w") as f:
        f.write(src)
    so = oracle.build(src=c_path, out=os.path.join(d, "libmutant.so"))
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"), so=so)
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    line = [l for l in proc.stdout.splitlines() if l.startswith("FAILED:")]
    if proc.returncode != 0 or not line:
        return name, f"crashed (rc={proc.returncode})"
    return name, line[0][len("FAILED:"):]


def test_every_planted_mistake_fails_a_pin():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = dict(ex.map(lambda kv: _run_mutant(kv[0], kv[1], tmp), MUTANTS.items()))
    survivors = [n for n, failed in results.items() if failed == "" or failed.startswith("crashed")]
    assert not survivors, f"mutants no pin caught: {survivors}; all: {results}"


def test_unmutated_copy_passes_every_pin():
    with tempfile.TemporaryDirectory() as tmp:
        name, failed = _run_mutant("identity", [], tmp)
    assert failed == "", failed
