"""The boundary as a C caller sees it (CPU, no GPU needed).

include/dmuon.h must be plain C: it compiles as C99 with every warning an
error, and a C program linked against the built library plans the
Llama-3-8B-shaped layer set (one layer), reads the plan back and gets the
documented error for a bad argument -- all host-only calls.  The Python
tests reach the same library through ctypes; this checks the header itself.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
PKG = os.path.join(ROOT, "matrix_orthogonalising_optimizer_gb300")

C_SOURCE = r"""
#include "dmuon.h"
#include <stdio.h>

int main(void) {
    /* one layer: q, k, v, o, gate, up, down */
    const dmuon_shape_t shapes[7] = {
        {4096, 4096, DMUON_BF16, 0},  {1024, 4096, DMUON_BF16, 0}, {1024, 4096, DMUON_BF16, 0},
        {4096, 4096, DMUON_BF16, 0},  {14336, 4096, DMUON_BF16, 0}, {14336, 4096, DMUON_BF16, 0},
        {4096, 14336, DMUON_BF16, 0}};
    dmuon_options_t opt = {0};
    dmuon_handle_t h = dmuon_plan_ex(shapes, 7, &opt);
    int64_t b, nb, total = 0;
    if (!h) {
        printf("plan failed: %s\n", dmuon_last_error());
        return 1;
    }
    nb = dmuon_plan_num_buckets(h);
    for (b = 0; b < nb; ++b) {
        dmuon_bucket_info_t info;
        if (dmuon_plan_bucket(h, b, &info) != DMUON_OK) return 2;
        printf("bucket %lld m %lld n %lld count %lld route %d\n", (long long)b, (long long)info.m,
               (long long)info.n, (long long)info.count, (int)info.route);
        total += info.count;
    }
    printf("matrices %lld waves %lld workspace %llu\n", (long long)total, (long long)dmuon_plan_num_waves(h),
           (unsigned long long)dmuon_workspace_bytes(h));
    /* a bad argument: the documented status, and a message */
    printf("bad bucket %d %s\n", dmuon_plan_bucket(h, nb, NULL), dmuon_status_string(DMUON_ERR_INVALID_ARG));
    dmuon_destroy(h);
    dmuon_destroy(NULL);
    return 0;
}
"""


def _cc():
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    return cc


def test_header_compiles_as_c99(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "dmuon.h"\nint dmuon_header_only;\n')
    subprocess.run([_cc(), "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", INCLUDE, "-c", str(src),
                    "-o", str(tmp_path / "h.o")], check=True)


def test_c_program_plans_through_the_library(tmp_path):
    lib = os.path.join(PKG, "libdmuon.so")
    if not os.path.exists(lib):
        pytest.skip("library not built")
    src = tmp_path / "plan.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "plan"
    subprocess.run([_cc(), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe), "-L", PKG,
                    "-ldmuon", "-Wl,-rpath," + PKG], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True, timeout=60).stdout
    lines = out.splitlines()
    buckets = [ln.split() for ln in lines if ln.startswith("bucket ")]
    # (m, n) buckets of one layer: 1024x4096 (k, v), 4096x4096 (q, o), 4096x14336 (gate, up
    # transposed, and down)
    got = sorted((int(b[3]), int(b[5]), int(b[7])) for b in buckets)
    assert got == [(1024, 4096, 2), (4096, 4096, 2), (4096, 14336, 3)]
    summary = next(ln for ln in lines if ln.startswith("matrices "))
    assert summary.split()[1] == "7" and int(summary.split()[5]) > 0
    bad = next(ln for ln in lines if ln.startswith("bad bucket "))
    assert bad.split()[2] == str(-1)
