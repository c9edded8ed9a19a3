"""AdamW comparison step: oracle pins (CPU), host-side errors (CPU) and GPU parity.

The fp64 oracle (``oracle/adamw.py``) is pinned by closed forms that do not
restate it: on the first step from zero state Adam's bias-corrected ratio
m/sqrt(v) is g/|g|, so the update is lr*g/(|g|+eps); with beta1 = beta2 = 0
every step is that first step; a zero gradient from zero state leaves only
the decay; and the update is invariant to scaling g, m by k and v by k^2 when
eps is negligible.
"""
import ctypes

import numpy as np
import pytest
import torch

from matrix_orthogonalising_optimizer_gb300 import _lib, adamw_step
from oracle import adamw as oadam
from oracle import round_to_storage

from tests.helpers import ulp_diff, ulp_of

F32 = lambda x: float(np.float32(x))  # noqa: E731  hyper-parameters as the kernel receives them


def _rand(n, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(n) * scale


# ---------------------------------------------------------------- oracle pins

def test_first_step_from_zero_state_is_sign_like():
    w, g = _rand(257, 1), _rand(257, 2, 1e-3)
    lr, wd, eps = 1e-3, 0.1, 1e-8
    (_, _, _), (w1, m1, v1) = oadam.adamw_step(w, g, np.zeros(257), np.zeros(257), lr=lr, beta1=0.9, beta2=0.999,
                                               eps=eps, wd=wd, step=1)
    np.testing.assert_allclose(w1, (1 - lr * wd) * w - lr * g / (np.abs(g) + eps), rtol=1e-13, atol=0)
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-15, atol=0)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12, atol=0)


def test_zero_betas_make_every_step_the_first():
    w, g, m, v = _rand(64, 3), _rand(64, 4), _rand(64, 5), np.abs(_rand(64, 6))
    lr, wd, eps = 2e-3, 0.01, 1e-8
    _, (w1, _, _) = oadam.adamw_step(w, g, m, v, lr=lr, beta1=0.0, beta2=0.0, eps=eps, wd=wd, step=5)
    np.testing.assert_allclose(w1, (1 - lr * wd) * w - lr * g / (np.abs(g) + eps), rtol=1e-13, atol=0)


def test_zero_grad_from_zero_state_only_decays():
    w = _rand(100, 7)
    _, (w1, m1, v1) = oadam.adamw_step(w, np.zeros(100), np.zeros(100), np.zeros(100), lr=0.01, beta1=0.9,
                                       beta2=0.999, eps=1e-8, wd=0.1, step=1)
    np.testing.assert_array_equal(w1, (1 - 0.01 * 0.1) * w)
    assert not m1.any() and not v1.any()


def test_scale_invariance():
    w, g, m, v = _rand(50, 8), _rand(50, 9), _rand(50, 10), np.abs(_rand(50, 11))
    kw = dict(lr=1e-3, beta1=0.9, beta2=0.99, eps=1e-30, wd=0.0, step=4)
    _, (a, _, _) = oadam.adamw_step(w, g, m, v, **kw)
    _, (b, _, _) = oadam.adamw_step(w, 1e3 * g, 1e3 * m, 1e6 * v, **kw)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=0)


# ---------------------------------------------------------------- host-side errors (no GPU touched)

def test_host_errors(lib):
    def call(ptr=16, numel=8, dtype=_lib.BF16, step=1, beta1=0.9, eps=1e-8, count=1):
        P = ctypes.c_void_p * 1
        n = (ctypes.c_int64 * 1)(numel)
        d = (ctypes.c_int32 * 1)(dtype)
        return lib.dmuon_adamw_step(P(ptr), P(ptr), P(ptr), P(ptr), n, d, count, 1e-3, beta1, 0.999, eps, 0.0,
                                    step, None)

    assert call(ptr=8) == _lib.ERR_ALIGN
    assert call(ptr=0) == _lib.ERR_ALIGN
    assert call(dtype=5) == _lib.ERR_UNSUPPORTED_DTYPE
    assert call(numel=-1) == _lib.ERR_INVALID_ARG
    assert call(step=0) == _lib.ERR_INVALID_ARG
    assert call(beta1=1.0) == _lib.ERR_INVALID_ARG
    assert call(eps=0.0) == _lib.ERR_INVALID_ARG
    assert call(count=-1) == _lib.ERR_INVALID_ARG
    assert lib.dmuon_adamw_step(None, None, None, None, None, None, 0, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None) \
        == _lib.OK


# ---------------------------------------------------------------- GPU parity

def _check(dtype, sizes, step, zero_state, seed, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.01):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    rng = np.random.default_rng(seed)
    host = []
    for i, n in enumerate(sizes):
        w = round_to_storage(rng.standard_normal(n) * 0.02, dtype)
        g = round_to_storage(rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -1), dtype)
        if zero_state:
            m = np.zeros(n)
            v = np.zeros(n)
        else:
            m = round_to_storage(rng.standard_normal(n) * 1e-3, dtype)
            v = round_to_storage(np.abs(rng.standard_normal(n)) * 1e-6, dtype)
        host.append((w, g, m, v))
    dev = [[torch.tensor(x, dtype=torch.float64).to(tdt).cuda() for x in t] for t in host]
    adamw_step([d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev], [d[3] for d in dev],
               lr, beta1, beta2, eps, wd, step)
    torch.cuda.synchronize()
    assert _lib.load().dmuon_adamw_status() == _lib.OK
    # ulps against one rounding of the fp64 result, pooled over all tensors.
    # m and v: the kernel's fp32 arithmetic rounds (1-beta)*g and g^2 before
    # its fma, so fp32 storage may sit 1-2 ulps off; bf16 storage rounds that
    # fp32 value once more and only ties differ.  W: the fp32 arithmetic errs
    # by a few fp32 ulps of |decay*W| and of the update; where the two nearly
    # cancel, that is many ulps of the small W', so W' is bounded per element
    # by its ulps plus that absolute error, and most elements must be exact.
    us_state, us_w, excess = [], [], []
    for (w, g, m, v), d in zip(host, dev):
        if w.size == 0:
            continue
        (wr, mr, vr), (w1, _, v1) = oadam.adamw_step(w, g, m, v, lr=F32(lr), beta1=F32(beta1), beta2=F32(beta2),
                                                      eps=F32(eps), wd=F32(wd), step=step, dtype=dtype)
        b1, b2 = F32(beta1), F32(beta2)
        for got, want, mag in ((d[2], mr, np.abs(b1 * m) + np.abs((1 - b1) * g)),
                               (d[3], vr, np.abs(b2 * v) + np.abs((1 - b2) * g * g))):
            us_state.append(ulp_diff(got.cpu(), torch.tensor(want).to(tdt)))
            # m' = beta1*m + (1-beta1)*g can cancel: bound it by its terms
            allowed = 2 * ulp_of(want, dtype) + 4 * 2.0 ** -24 * mag
            excess.append(np.abs(got.double().cpu().numpy() - want) - allowed)
        us_w.append(ulp_diff(d[0].cpu(), torch.tensor(wr).to(tdt)))
        decayed = (1.0 - F32(lr) * F32(wd)) * w
        # the update carries m's absolute error (its terms' size) through m/denom
        denom = np.sqrt(v1) / np.sqrt(1 - b2 ** step) + F32(eps)
        m_terms = F32(lr) / (1 - b1 ** step) * (np.abs(b1 * m) + np.abs((1 - b1) * g)) / denom
        allowed = 2 * ulp_of(wr, dtype) + 8 * 2.0 ** -24 * (np.abs(decayed) + np.abs(decayed - w1) + m_terms)
        excess.append(np.abs(d[0].double().cpu().numpy() - wr) - allowed)
    us, uw = np.concatenate(us_state), np.concatenate(us_w)
    assert np.concatenate(excess).max() <= 0.0
    if dtype == "bf16":
        assert (us == 0).mean() >= 0.99, np.bincount(us)[:8]
        assert (uw <= 1).mean() >= 0.999, np.bincount(uw)[:8]
    else:
        # fp32: m' often cancels (beta1*m against (1-beta1)*g) and W' often
        # sits far below |W| and |update|, so the fp32 operands' rounding is
        # several ulps of the result; the per-element absolute bound above is
        # the check, and most elements still agree exactly
        assert (us == 0).mean() >= 0.8 and (uw == 0).mean() >= 0.6, (np.bincount(us)[:4], np.bincount(uw)[:4])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("step,zero_state", [(1, True), (7, False)])
def test_adamw_parity(dtype, step, zero_state):
    sizes = [0, 1, 7, 8, 4095, 4096, 4097, 768 * 3072, 12345, 3 * 4096 + 5]
    _check(dtype, sizes, step, zero_state, seed=step)


@pytest.mark.gpu
def test_adamw_many_tensors_span_launches():
    # 600 tensors: three launches of the 256-tensor table
    rng = np.random.default_rng(5)
    sizes = [int(x) for x in rng.integers(0, 3000, 600)]
    _check("bf16", sizes, 3, False, seed=11)
