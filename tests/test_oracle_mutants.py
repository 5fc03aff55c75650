"""Plant plausible slips in copies of the oracle and check that its pins catch every one.

Each mutant is the oracle's C source with one textual change (a dropped term, a wrong sign,
a transposed index, an off-by-one, a wrong rounding), compiled into a temporary library.  The
full pin battery runs against it in a child process (a slip that reads out of bounds may crash
the child; that also counts as caught).  A mutant that passes every pin means the pins have a
blind spot.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    "padded_rows_floor_plus_one": ("m[p] = (rows[p] + R - 1) / R;", "m[p] = rows[p] / R + 1;"),
    "dropped_rank_term": ("for (int32_t r = 1; r < R; ++r)\n                        acc = acc +",
                          "for (int32_t r = 2; r < R; ++r)\n                        acc = acc +"),
    "wrong_sign": ("acc = acc + oracle_bf16_to_f32", "acc = acc - oracle_bf16_to_f32"),
    "transposed_input_index": ("int64_t i = row * row_len[p] + k;", "int64_t i = k * rows[p] + row;"),
    "transposed_output_index": ("shards[d][L.o[p] + j * row_len[p] + k] = acc;",
                                "shards[d][L.o[p] + j + k * L.m[p]] = acc;"),
    "padding_not_plus_zero": ("acc = 0.0f;", "acc = -0.0f;"),
    "offset_after_increment": ("o[p] = offset;\n        offset += s[p];", "offset += s[p];\n        o[p] = offset;"),
    "unsharded_counts_padding": ("unsharded += rows[p] * row_len[p];", "unsharded += m[p] * R * row_len[p];"),
    "valid_rows_unclamped": ("if (v > m_p)\n        v = m_p;", ""),
    "widening_shift": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    "ag_reads_global_row": ("params[p][row * row_len[p] + k] = shards[r][L.o[p] + j * row_len[p] + k];",
                            "params[p][row * row_len[p] + k] = shards[r][L.o[p] + row * row_len[p] + k];"),
    "ag_rank_row_base": ("int64_t row = (int64_t)r * L.m[p] + j;\n            if (row >= rows[p])\n                continue;\n            for (int64_t k = 0; k < row_len[p]; ++k)\n                params",
                         "int64_t row = (int64_t)r * L.s[p] + j;\n            if (row >= rows[p])\n                continue;\n            for (int64_t k = 0; k < row_len[p]; ++k)\n                params"),
    "fold_from_plus_zero": ("acc = oracle_bf16_to_f32(grads[0 * (int64_t)P + p][i]);\n                    for (int32_t r = 1;",
                            "acc = 0.0f;\n                    for (int32_t r = 0;"),
    "part_skips_last_param": ("for (int32_t p = p_begin; p < p_end; ++p) {", "for (int32_t p = p_begin; p + 1 < p_end; ++p) {"),
    "exact_sum_fp32_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "exact_sum_dropped_rank_term": ("for (int32_t r = 0; r < R; ++r)\n                            acc +=",
                                    "for (int32_t r = 1; r < R; ++r)\n                            acc +="),
}

_RUNNER = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import oracle, oracle_pins
oracle.use_library({lib!r})
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin()
    except AssertionError:
        failed.append(pin.__name__)
print("FAILED:" + ",".join(failed))
sys.exit(1 if failed else 0)
"""


def _build_mutant(tmp, name, old, new):
    with open(os.path.join(ROOT, "oracle", "tide_oracle.c")) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation site of {name} not found in the oracle source"
    src = src.replace(old, new, 1)
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    with open(c, "w") as f:
        f.write(src)
    subprocess.check_call(["gcc", *oracle.CFLAGS, c, "-o", so])
    return so


def test_every_mutant_is_caught(oracle_lib):
    with tempfile.TemporaryDirectory() as tmp:
        procs = {}
        for name, (old, new) in MUTANTS.items():
            so = _build_mutant(tmp, name, old, new)
            code = _RUNNER.format(root=ROOT, tests=HERE, lib=so)
            procs[name] = subprocess.Popen([sys.executable, "-c", code], stdout=subprocess.PIPE,
                                           stderr=subprocess.STDOUT, text=True)
        survivors = []
        for name, pr in procs.items():
            out, _ = pr.communicate(timeout=600)
            if pr.returncode == 0:
                survivors.append(name)
        assert not survivors, f"mutants not caught by any pin: {survivors}"


def test_unmutated_copy_passes(oracle_lib):
    """The runner itself reports success on an unchanged copy (guards against a runner that
    always fails)."""
    with tempfile.TemporaryDirectory() as tmp:
        so = _build_mutant(tmp, "identity", "#include <stdint.h>", "#include <stdint.h>")
        code = _RUNNER.format(root=ROOT, tests=HERE, lib=so)
        pr = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
        assert pr.returncode == 0, pr.stdout + pr.stderr
