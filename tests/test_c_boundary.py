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


STEP_SOURCE = r"""
#include "dmuon.h"
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

static int fail(const char* what) {
    fprintf(stderr, "%s: %s\n", what, dmuon_last_error());
    return 1;
}

/* argv: input file, output file, lr, beta, wd.  Input: int64 count, then per
   matrix int64 rows, cols and the bf16 W, grad, momentum; output: W', M'. */
int main(int argc, char** argv) {
    FILE *in, *out;
    int64_t n, i;
    int k;
    dmuon_shape_t* shapes;
    void **dev[3], *ws;
    size_t ws_bytes;
    dmuon_handle_t h;
    float lr, beta, wd;
    if (argc != 6) return 2;
    lr = strtof(argv[3], NULL);
    beta = strtof(argv[4], NULL);
    wd = strtof(argv[5], NULL);
    in = fopen(argv[1], "rb");
    if (!in || fread(&n, 8, 1, in) != 1) return 3;
    shapes = (dmuon_shape_t*)calloc((size_t)n, sizeof *shapes);
    for (k = 0; k < 3; ++k) dev[k] = (void**)calloc((size_t)n, sizeof(void*));
    for (i = 0; i < n; ++i) {
        int64_t rc[2];
        size_t bytes;
        if (fread(rc, 8, 2, in) != 2) return 3;
        shapes[i].rows = rc[0];
        shapes[i].cols = rc[1];
        shapes[i].dtype = DMUON_BF16;
        bytes = (size_t)(rc[0] * rc[1] * 2);
        for (k = 0; k < 3; ++k) {
            void* buf = malloc(bytes);
            if (fread(buf, 1, bytes, in) != bytes) return 3;
            if (cudaMalloc(&dev[k][i], bytes) != cudaSuccess) return 4;
            if (cudaMemcpy(dev[k][i], buf, bytes, cudaMemcpyHostToDevice) != cudaSuccess) return 4;
            free(buf);
        }
    }
    fclose(in);
    h = dmuon_plan(shapes, n);
    if (!h) return fail("plan");
    ws_bytes = dmuon_workspace_bytes(h);
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess) return 4;
    if (dmuon_bind_workspace(h, ws, ws_bytes) != DMUON_OK) return fail("bind");
    if (dmuon_step(h, dev[0], (const void* const*)dev[1], dev[2], lr, beta, wd, 5, NULL) != DMUON_OK)
        return fail("step");
    if (dmuon_device_status(h, NULL) != DMUON_OK) return fail("device status");
    out = fopen(argv[2], "wb");
    for (i = 0; i < n; ++i) {
        size_t bytes = (size_t)(shapes[i].rows * shapes[i].cols * 2);
        void* buf = malloc(bytes);
        for (k = 0; k < 3; k += 2) {
            if (cudaMemcpy(buf, dev[k][i], bytes, cudaMemcpyDeviceToHost) != cudaSuccess) return 4;
            fwrite(buf, 1, bytes, out);
        }
        free(buf);
    }
    fclose(out);
    dmuon_destroy(h);
    cudaFree(ws);
    for (i = 0; i < n; ++i)
        for (k = 0; k < 3; ++k) cudaFree(dev[k][i]);
    return 0;
}
"""


@pytest.mark.gpu
def test_c_program_steps_on_the_gpu(tmp_path):
    """A C program runs a whole step through the ABI (cudaMalloc'd buffers, default
    stream): its W' and M' equal the Python binding's bit for bit, and O matches the
    oracle."""
    import numpy as np
    import torch

    import __graft_entry__
    import workloads
    from tests.helpers import TOL, f32, oracle_O, rel_fro, run_step
    import oracle

    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    shapes = [(320, 704), (704, 320), (300, 300), (48, 200)]
    cfg = workloads.Config("t", "test", "bf16", 41, tuple(shapes), "normal", grad_scale=1e-3, mom_std=1e-3)
    inputs = [workloads.make_matrix(cfg, i, "cpu") for i in range(len(shapes))]
    inputs = [(torch.zeros_like(w), g, m) for w, g, m in inputs]  # W = 0: W' = -lr*s*O
    beta = f32(0.95)

    def raw(t):
        return t.contiguous().view(torch.int16).numpy().tobytes()

    src = tmp_path / "step.c"
    src.write_text(STEP_SOURCE)
    exe = tmp_path / "step"
    subprocess.run([_cc(), "-std=c99", "-Wall", "-Werror", "-I", INCLUDE, "-I", os.path.join(cuda, "include"),
                    str(src), "-o", str(exe), "-L", PKG, "-ldmuon", "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    "-Wl,-rpath," + PKG, "-Wl,-rpath," + os.path.join(cuda, "lib64")], check=True)
    fin, fout = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(fin, "wb") as f:
        f.write(np.int64(len(shapes)).tobytes())
        for (r, c), (w, g, m) in zip(shapes, inputs):
            f.write(np.array([r, c], dtype=np.int64).tobytes())
            f.write(raw(w) + raw(g) + raw(m))
    subprocess.run([str(exe), str(fin), str(fout), "1.0", repr(beta), "0.0"], check=True, timeout=300)
    blob = np.fromfile(fout, dtype=np.int16)
    c_w, c_m, off = [], [], 0
    for r, c in shapes:
        for dst in (c_w, c_m):
            dst.append(torch.from_numpy(blob[off:off + r * c].copy()).view(torch.bfloat16).reshape(r, c))
            off += r * c
    py_w, py_m, _ = run_step(shapes, inputs, "bf16", lr=1.0, beta=beta, wd=0.0)
    for a, b in zip(c_w, py_w):
        assert torch.equal(a, b)
    for a, b in zip(c_m, py_m):
        assert torch.equal(a, b)
    want = oracle_O(inputs, beta=beta)
    for (r, c), wn, o in zip(shapes, c_w, want):
        got = -wn.double().numpy() / oracle.shape_scale(r, c)
        assert rel_fro(got, o) <= TOL["bf16"], (r, c)
