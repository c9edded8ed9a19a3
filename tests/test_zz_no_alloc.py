"""dmuon_step_noalloc: the Muon step for one small matrix with no device allocation.

Callers that cannot allocate device memory (their GPU memory is held by
another allocator, or they run under a fixed budget) cannot give dmuon_step
its workspace; this entry point keeps its scratch in a static device array
instead.  Here it is called through the C ABI three times in a row, on shapes with
different short sides and on both dtypes, and compared with dmuon_step in its fp32 validation mode
(the same arithmetic) on the same inputs: the momentum must match exactly and
the orthogonalised update O within the fp32 tolerance of 1e-4.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from matrix_orthogonalising_optimizer_gb300 import Muon, _lib

pytestmark = pytest.mark.gpu

BETA, LR, WD = float(np.float32(0.95)), float(np.float32(0.02)), float(np.float32(0.01))


def _inputs(rows, cols, dtype, seed):
    cfg = workloads.Config("t", "no-alloc test", dtype, seed, ((rows, cols),), "normal", grad_scale=1e-3,
                           mom_std=1e-3)
    return workloads.make_matrix(cfg, 0, "cpu")


def _noalloc(lib, w, g, m, dtype, lr, wd):
    rows, cols = w.shape
    st = lib.dmuon_step_noalloc(ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(g.data_ptr()),
                                ctypes.c_void_p(m.data_ptr()), rows, cols, 0 if dtype == "bf16" else 1, lr, BETA,
                                wd, 5, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.dmuon_last_error()


def _workspace_step(w, g, m, dtype, lr, wd):
    rows, cols = w.shape
    muon = Muon([(rows, cols, 0 if dtype == "bf16" else 1)], precision="fp32").bind()
    muon.step([w], [g], [m], lr, BETA, wd, 5)


def test_noalloc_matches_workspace_step_three_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = _lib.load(build_if_missing=True)
    # three calls in a row whose short side changes (128, 40, 96), so each
    # call's scratch layout differs from the one before; a tall bf16 matrix
    # takes the transposed load and store path
    for rows, cols, dtype, seed in [(128, 2048, "bf16", 41), (700, 40, "bf16", 42), (96, 700, "fp32", 43)]:
        w, g, m = _inputs(rows, cols, dtype, seed)
        s = oracle.shape_scale(rows, cols)
        outs = {}
        for name, fn in (("noalloc", _noalloc), ("workspace", lambda *a: _workspace_step(*a))):
            # W = 0, lr = 1, wd = 0 exposes O as W' = -s*O
            wz, gd, md = torch.zeros_like(w).cuda(), g.cuda(), m.cuda()
            if name == "noalloc":
                fn(lib, wz, gd, md, dtype, 1.0, 0.0)
            else:
                fn(wz, gd, md, dtype, 1.0, 0.0)
            torch.cuda.synchronize()
            outs[name] = (-wz.double().cpu().numpy() / s, md.cpu())
        o_new, m_new = outs["noalloc"]
        o_ref, m_ref = outs["workspace"]
        assert torch.equal(m_new, m_ref)
        assert np.linalg.norm(o_new - o_ref) / np.linalg.norm(o_ref) <= 1e-4
        want = oracle.muon_step(np.zeros((rows, cols)), g.double().numpy(), m.double().numpy(), lr=1.0, beta=BETA,
                                wd=0.0)["O"]
        tol = 1e-4 if dtype == "fp32" else 4e-3  # bf16 storage rounds the recovered O
        assert np.linalg.norm(o_new - want) / np.linalg.norm(want) <= tol
        # the real update, real parameters
        w_new, w_ref = w.cuda(), w.cuda()
        _noalloc(lib, w_new, g.cuda(), m.cuda(), dtype, LR, WD)
        _workspace_step(w_ref, g.cuda(), m.cuda(), dtype, LR, WD)
        torch.cuda.synchronize()
        d = (w_new.double() - w_ref.double()).abs().cpu().numpy()
        delta = (w_ref.double().cpu().numpy() - (1 - LR * WD) * w.double().numpy())
        ulp = np.ldexp(1.0, np.frexp(np.abs(w_ref.double().cpu().numpy()))[1] - (8 if dtype == "bf16" else 24))
        assert np.all(d <= ulp + 1e-4 * np.abs(delta).max())


def test_noalloc_rejects_shapes_beyond_the_scratch():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    lib = _lib.load(build_if_missing=True)
    buf = torch.zeros(1 << 19, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    # the last two overflow int64 if multiplied before the sides are bounded
    for rows, cols in [(129, 300), (300, 129), (64, 5000), (128, 1 << 57), (1 << 40, 1 << 40)]:
        st = lib.dmuon_step_noalloc(p, p, p, rows, cols, 1, LR, BETA, WD, 5, None)
        assert st == _lib.ERR_INVALID_ARG
        assert b"262144" in lib.dmuon_last_error()
