"""Shared helpers of the GPU parity tests (run the C ABI, compare with the oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from matrix_orthogonalising_optimizer_gb300 import Muon

TOL = {"bf16": 3e-2, "fp32": 1e-4}


def f32(x):
    return float(np.float32(x))


def storage(dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def rel_fro(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def ulp_diff(a: torch.Tensor, b: torch.Tensor) -> np.ndarray:
    """|a - b| in units in the last place, for bf16 or fp32 tensors of one dtype."""
    if a.dtype == torch.bfloat16:
        ia = a.view(torch.int16).to(torch.int64)
        ib = b.view(torch.int16).to(torch.int64)
        lo = -(1 << 15)
    else:
        ia = a.view(torch.int32).to(torch.int64)
        ib = b.view(torch.int32).to(torch.int64)
        lo = -(1 << 31)
    oa = torch.where(ia < 0, lo - ia, ia)
    ob = torch.where(ib < 0, lo - ib, ib)
    return (oa - ob).abs().numpy()


def ulp_of(x, dtype):
    """Spacing of the storage dtype at |x| (bf16: 8 significant bits, fp32: 24)."""
    _, e = np.frexp(np.asarray(x, dtype=np.float64))
    bits = 8 if dtype == "bf16" else 24
    return np.ldexp(1.0, np.maximum(e, -125) - bits)


def run_step(shapes, inputs, dtype, *, lr, beta, wd, ns_steps=5, zero_w=False, muon=None, **plan_kw):
    """One GPU step on copies of ``inputs`` [(W, grad, mom)] (CPU tensors).

    Returns (W', M') on the CPU and the plan.  With ``zero_w`` the parameters
    start at 0, so W' = -lr*s*O exposes the orthogonalised update O.
    """
    dt = 0 if dtype == "bf16" else 1
    if muon is None:
        muon = Muon([(r, c, dt) for r, c in shapes], **plan_kw).bind()
    ws = [torch.zeros_like(w).cuda() if zero_w else w.cuda() for w, _, _ in inputs]
    gs = [g.cuda() for _, g, _ in inputs]
    ms = [m.cuda().clone() for _, _, m in inputs]
    muon.step(ws, gs, ms, lr, beta, wd, ns_steps)
    torch.cuda.synchronize()
    assert muon.device_status() == 0
    return [w.cpu() for w in ws], [m.cpu() for m in ms], muon


def gpu_O(shapes, inputs, dtype, *, beta, ns_steps=5, scale_rule="aspect", **plan_kw):
    """O recovered through the ABI: W = 0, lr = 1, wd = 0 gives W' = -s*O."""
    w, _, muon = run_step(shapes, inputs, dtype, lr=1.0, beta=beta, wd=0.0, ns_steps=ns_steps, zero_w=True,
                          scale_rule=scale_rule, **plan_kw)
    out = []
    for (r, c), wi in zip(shapes, w):
        s = oracle.shape_scale(r, c, scale_rule)
        out.append(-wi.double().numpy() / s)
    return out, muon


def oracle_O(inputs, *, beta, ns_steps=5, nesterov=True, coeffs=oracle.NS_COEFFS):
    res = []
    for w, g, m in inputs:
        res.append(oracle.muon_step(np.zeros(tuple(w.shape)), g.double().numpy(), m.double().numpy(), lr=1.0,
                                    beta=beta, wd=0.0, ns_steps=ns_steps, nesterov=nesterov, coeffs=coeffs,
                                    dtype="fp32")["O"])
    return res


def check_update_against_oracle(w_gpu, w_in, want, o_orc, *, lr, wd, scale, dtype, tau):
    """W' from the GPU against the oracle's W' (not against the GPU's own O).

    The two differ by (a) one rounding of each to the storage dtype, (b) the
    kernel's fp32 arithmetic (decay = fl(1 - lr wd), fl(decay W), fl(lr s):
    at most 2^-23 |W| + 2^-23 lr s |O|), and (c) lr s (O_gpu - O_oracle), which
    the O parity bounds in Frobenius norm by lr s tau ||O||_F.  So:

    * Frobenius bar: what is left of |W'_gpu - W'_oracle| after (a) and (b)
      is at most lr s tau ||O_oracle||_F;
    * ulp bar where the O tolerance cannot move W' by a whole ulp: on the
      elements whose storage ulp is at least 4 lr s tau max(|O_ij|, rms(O)),
      >= 99.9 % are within 1 ulp and all within 2.  An element's share of the
      O error grows with its own |O_ij|: with heavy-tailed gradients (1 % of
      entries x100) a few outputs are 25x the rms and carry errors of a few
      percent of themselves, i.e. several ulps of W'.  Elements near W' = 0
      have a tiny ulp that the allowed O error spans many times.  An ulp bar
      over all elements would test the O error again, not the update.

    w_gpu, w_in: torch tensors (storage dtype); want, o_orc: float64 arrays.
    Returns (excess ratio, subset fraction, fraction within 1 ulp in the subset).
    """
    got = w_gpu.double().numpy()
    w64 = w_in.double().numpy()
    ulp = ulp_of(want, dtype)
    arith = 2.0 ** -23 * (np.abs(w64) + lr * scale * np.abs(o_orc))
    excess = np.maximum(np.abs(got - want) - ulp - arith, 0.0)
    allowed = lr * scale * tau * np.linalg.norm(o_orc)
    ratio = float(np.linalg.norm(excess) / allowed)
    assert ratio <= 1.0, f"W' excess {ratio:.3f} of what the O tolerance allows"
    rms = np.sqrt(np.mean(o_orc * o_orc))
    sub = ulp >= 4.0 * lr * scale * tau * np.maximum(np.abs(o_orc), rms)
    frac1, worst = 1.0, 0
    if sub.sum() >= 1000:
        d = ulp_diff(w_gpu, torch.from_numpy(want).to(w_gpu.dtype))[sub]
        frac1, worst = float((d <= 1).mean()), int(d.max())
        assert frac1 >= 0.999 and worst <= 2, (frac1, worst)
    print(f"W' vs oracle {tuple(w_gpu.shape)} {dtype}: excess {ratio:.3f} of allowed; ulp-bar subset "
          f"{sub.mean():.3f}, within 1 ulp there {frac1:.5f}, worst {worst}")
    return ratio, float(sub.mean()), frac1
