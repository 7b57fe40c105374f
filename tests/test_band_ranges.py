"""Host check of the tile-skipping arithmetic (no GPU needed).

The kernels skip whole tiles with query_range / key_range and mask single
elements with the intervals of visible_queries / visible_keys, all restating
key_visible (csrc/fa_internal.cuh).  Skipping is only correct if
the ranges hold every visible (query, key) pair; it is only efficient if they
are tight.  This test compiles a small host program against that header with
nvcc and checks both, exhaustively, for every tile of small problems with and
without causal masking and sliding windows (the kernels' tiles are 128 rows;
here tiles of 1 to 7 rows cover the same edge cases in less time).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "flashattention_backward_preprocess_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "fa_internal.cuh"
using namespace fa;
int main() {
    long checked = 0;
    for (int S_q = 1; S_q <= 13; ++S_q)
    for (int S_k = 1; S_k <= 13; ++S_k)
    for (int causal = 0; causal < 2; ++causal)
    for (int window = 0; window <= 15; ++window)
    for (int T = 1; T <= 7; ++T) {
        Shape s{};
        s.S_q = S_q; s.S_k = S_k; s.causal = causal; s.window = window;
        const int off = S_k - S_q;
        // key tiles [j0, j1): query_range must be exactly the rows seeing one of its keys
        for (int j0 = 0; j0 < S_k; j0 += T) {
            const int j1 = j0 + T < S_k ? j0 + T : S_k;
            int lo, hi;
            query_range(s, j0, j1, lo, hi);
            for (int i = 0; i < S_q; ++i) {
                bool sees = false;
                for (int j = j0; j < j1; ++j) sees |= key_visible(i + off, j, causal, window);
                const bool in = i >= lo && i < hi;
                if (sees != in) {
                    printf("query_range S_q=%d S_k=%d causal=%d w=%d tile=[%d,%d) row %d: sees=%d in=%d [%d,%d)\n",
                           S_q, S_k, causal, window, j0, j1, i, sees, in, lo, hi);
                    return 1;
                }
                ++checked;
            }
        }
        // query tiles [i0, i1): key_range must be exactly the keys one of its rows sees
        for (int i0 = 0; i0 < S_q; i0 += T) {
            const int i1 = i0 + T < S_q ? i0 + T : S_q;
            int lo, hi;
            key_range(s, i0, i1, lo, hi);
            for (int j = 0; j < S_k; ++j) {
                bool seen = false;
                for (int i = i0; i < i1; ++i) seen |= key_visible(i + off, j, causal, window);
                const bool in = j >= lo && j < hi;
                if (seen != in) {
                    printf("key_range S_q=%d S_k=%d causal=%d w=%d tile=[%d,%d) key %d: seen=%d in=%d [%d,%d)\n",
                           S_q, S_k, causal, window, i0, i1, j, seen, in, lo, hi);
                    return 1;
                }
                ++checked;
            }
        }
    }
    // per-element intervals: visible_queries (one key, a run of queries) and
    // visible_keys (one query, a run of keys) against key_visible
    for (int causal = 0; causal < 2; ++causal)
    for (int window = 0; window <= 12; ++window)
    for (int d = -40; d <= 40; ++d) {
        int lo, hi;
        visible_queries(d, causal, window, lo, hi);
        for (int q = -60; q <= 60; ++q) {
            const bool vis = key_visible(1000 + q, 1000 + d, causal, window);
            if (vis != (q >= lo && q < hi)) {
                printf("visible_queries causal=%d w=%d dj=%d q=%d: %d vs [%d,%d)\n", causal, window, d, q, vis, lo, hi);
                return 1;
            }
            ++checked;
        }
        visible_keys(d, causal, window, lo, hi);
        for (int c = -60; c <= 60; ++c) {
            const bool vis = key_visible(1000 + d, 1000 + c, causal, window);
            if (vis != (c >= lo && c < hi)) {
                printf("visible_keys causal=%d w=%d dp=%d c=%d: %d vs [%d,%d)\n", causal, window, d, c, vis, lo, hi);
                return 1;
            }
            ++checked;
        }
    }
    printf("ok %ld\n", checked);
    return 0;
}
"""


def _nvcc():
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


def test_tile_ranges_are_exact(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    src = tmp_path / "ranges.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "ranges"
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok ")
