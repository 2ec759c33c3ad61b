"""Plant plausible mistakes in a copy of the oracle and check that the pins catch each.

Each mutant is compiled from a patched copy of ``oracle/a2av_oracle.c`` into a
temporary directory and checked by ``python -m tests._pins <lib>`` in a
subprocess, so that a mutant that corrupts memory or crashes cannot take the
test session with it: a crash counts as caught.  The mistakes planted are the
kinds the definition leaves room for -- a transposed operand, an inclusive
instead of exclusive scan, a dropped term, a reversed order, an off-by-one in
a bound, a swapped output row.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "in_offset_transposed": ("off += S[(int64_t)r * W + q];", "off += S[(int64_t)q * W + r];"),
    "out_offset_inclusive": ("for (int q = 0; q < r; ++q) off += S[(int64_t)q * W + p];",
                             "for (int q = 0; q <= r; ++q) off += S[(int64_t)q * W + p];"),
    "sources_reversed": ("for (int q = 0; q < r; ++q) off += S[(int64_t)q * W + p];",
                         "for (int q = r + 1; q < W; ++q) off += S[(int64_t)q * W + p];"),
    "count_transposed": ("const int64_t n = in_splits[(int64_t)r * W + p];",
                         "const int64_t n = in_splits[(int64_t)p * W + r];"),
    "offset_row_is_source_offset": ("out_so_p[W + r] = dst_row;", "out_so_p[W + r] = src_row;"),
    "so_rows_swapped": ("out_so_p[r] = n;\n      out_so_p[W + r] = dst_row;",
                        "out_so_p[W + r] = n;\n      out_so_p[r] = dst_row;"),
    "row_index_dropped": ("in[r] + (src_row + i) * row_bytes", "in[r] + (src_row) * row_bytes"),
    "self_chunk_dropped": ("if (out_p == NULL) continue;", "if (out_p == NULL || r == p) continue;"),
    "in_capacity_off_by_one": ("rows > in_capacity_rows) return", "rows > in_capacity_rows + 1) return"),
    "out_capacity_off_by_one": ("rows > out_capacity_rows) return", "rows > out_capacity_rows + 1) return"),
    "negative_accepted": ("in_splits[e] < 0 ||", "in_splits[e] < -1 ||"),
    "limit_drops_W": ("kMaxBytes / ((int64_t)W * row_bytes)", "kMaxBytes / (row_bytes)"),
    "null_input_unchecked": ("if (in != NULL && in[r] == NULL && rows > 0)",
                             "if (in != NULL && in[r] == NULL && rows > kMaxBytes)"),
    "combine_reads_offsets_row": ("St[(int64_t)p * W + r] = dispatch_so[(int64_t)p * 2 * W + r];",
                                  "St[(int64_t)p * W + r] = dispatch_so[(int64_t)p * 2 * W + W + r];"),
    "combine_not_transposed": ("St[(int64_t)p * W + r] = dispatch_so[(int64_t)p * 2 * W + r];",
                               "St[(int64_t)r * W + p] = dispatch_so[(int64_t)p * 2 * W + r];"),
    "dispatch_unstable": ("      for (int64_t i = 0; i < m; ++i)\n        if (key[r][i] == k) {",
                          "      for (int64_t i = m - 1; i >= 0; --i)\n        if (key[r][i] == k) {"),
    "dispatch_dest_mod": ("S[(int64_t)r * W + key[r][i] / K] += 1;",
                          "S[(int64_t)r * W + key[r][i] % W] += 1;"),
    "dispatch_ignores_src": ("rows[r] + (int64_t)src_row[r][i] * row_bytes",
                             "rows[r] + (int64_t)(i % n_rows[r]) * row_bytes"),
    "dispatch_pos_off_by_one": ("place[r][i] = next++;", "place[r][i] = ++next - 0;"),
    "dispatch_key_bound": ("key[r][i] >= nkeys ||", "key[r][i] > nkeys ||"),
    "combine_items_no_group_start": (
        "out_offset(W, S, p, r) + (sorted_pos[r][i] - in_offset(W, S, r, p));",
        "out_offset(W, S, p, r) + (sorted_pos[r][i]);"),
    "combine_items_chunk_of_peer": (
        "out_offset(W, S, p, r) + (sorted_pos[r][i] - in_offset(W, S, r, p));",
        "out_offset(W, S, r, p) + (sorted_pos[r][i] - in_offset(W, S, r, p));"),
    "combine_items_group_bound": ("sorted_pos[r][i] >= lo + S[(int64_t)r * W + p])",
                                  "sorted_pos[r][i] > lo + S[(int64_t)r * W + p])"),
    "row_source_wrong_chunk": ("*i = in_offset(W, in_splits, q, p) + (k - start);",
                               "*i = in_offset(W, in_splits, p, q) + (k - start);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = tmp_path / "a2av_oracle.c"
    path.write_text(src.replace(old, new))
    lib = oracle.build(str(path), str(tmp_path / "liba2av_oracle_mutant.so"))
    # Some mutants index out of bounds: the pin process may crash or, rarely,
    # run away instead of failing an assertion (the unmutated pins take about
    # a second).  Either way the mutant did not pass the pins.
    try:
        res = subprocess.run([sys.executable, "-m", "tests._pins", lib], cwd=ROOT,
                             capture_output=True, text=True, timeout=60)
    except subprocess.TimeoutExpired:
        return
    assert res.returncode != 0, f"mutant {name} passed every pin:\n{res.stdout}{res.stderr}"


def test_unmutated_copy_passes(tmp_path):
    path = tmp_path / "a2av_oracle.c"
    path.write_text(open(oracle.SOURCE).read())
    lib = oracle.build(str(path), str(tmp_path / "liba2av_oracle_copy.so"))
    res = subprocess.run([sys.executable, "-m", "tests._pins", lib], cwd=ROOT,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
