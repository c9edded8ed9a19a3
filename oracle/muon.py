"""fp64 oracle of one Muon optimizer step over a set of weight matrices.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product never
imports this module.

What is computed, per matrix W (rows x cols) with gradient and momentum of the
same shape (DMuon technical summary on gist.science, pt/fr, section 1
"Declaracao do Problema": Newton-Schulz iterations applied to the
momentum-aggregated gradients of the weight matrices, which push the update's
singular values toward a uniform spectrum; section 2.2: the iteration works on
X X^T):

1. momentum:   M' = beta*M + grad,  U = grad + beta*M'   (Nesterov form)
2. orientation: X = U if rows <= cols else U^T, so X is m x n with m <= n
   (section 2.2 takes the short side m < n)
3. normalise:  X0 = X / (||X||_F + eps)
4. Newton-Schulz, T steps of   A = X X^T;  B = b*A + c*A@A;  X <- a*X + B@X
5. O = X_T in the original orientation
6. update:     W' = (1 - lr*wd)*W - lr*s*O,  s = sqrt(max(1, rows/cols))
7. W' and M' are rounded once, to nearest-even, to the storage dtype.

The pages fix none of: the momentum formula, eps, the NS coefficients and step
count, the update's decay form and shape scale.  The readings taken are the
commonly published Muon ones: Nesterov momentum, eps = 1e-7, the quintic
(a, b, c) = (3.4445, -4.7750, 2.0315), T = 5, decoupled weight decay and the
aspect scale sqrt(max(1, rows/cols)).  Each is a parameter here.

``ns_gram`` restates step 4 in the m x m Gram space of section 2.2
(G = X X^T; every iterate is a polynomial in G, so X_k = Q_k X0 with
P_k = a I + b R_k + c R_k^2, Q_{k+1} = P_k Q_k, R_{k+1} = P_k R_k P_k).  It
is exact in exact arithmetic and serves to pin the Gram-space identity.

Parity pins live in tests/test_oracle.py: the closed form U f^T(S) V^T
through an independent Jacobi SVD, the singular-value band of the quintic,
Gram == direct, orthonormal input, zero and rank-1 inputs, scale invariance,
transpose equivariance, the rounding rule and the planner brute force.
"""
from __future__ import annotations

import numpy as np

NS_COEFFS = (3.4445, -4.7750, 2.0315)
EPS = 1e-7

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_to_bf16(x):
    """Round float64 values to the nearest bfloat16 value, ties to even.

    bfloat16 keeps 8 significant bits and the float32 exponent range, so the
    quantum of a normal value v with 2**(e-1) <= |v| < 2**e is 2**(e-8); below
    the smallest normal 2**-126 the quantum stays 2**-133.  One rounding, from
    the exact fp64 value (no detour through float32).
    """
    x = np.asarray(x, dtype=np.float64)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    _, e = np.frexp(xf)
    q = np.maximum(e, -125) - 8
    y = np.ldexp(np.rint(np.ldexp(xf, -q)), q)
    y = np.where(np.abs(y) > _BF16_MAX, np.copysign(np.inf, y), y)
    return np.where(finite, y, x)


def round_to_fp32(x):
    """Round float64 values to the nearest float32 value, ties to even."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_to_storage(x, dtype: str):
    if dtype == "bf16":
        return round_to_bf16(x)
    if dtype == "fp32":
        return round_to_fp32(x)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def nesterov_momentum(grad, mom, beta: float, nesterov: bool = True):
    """Momentum accumulation: M' = beta*M + grad; Nesterov look-ahead U = grad + beta*M'.

    With ``nesterov=False`` the update direction is M' itself.
    """
    grad = np.asarray(grad, dtype=np.float64)
    mom = np.asarray(mom, dtype=np.float64)
    mom_new = beta * mom + grad
    u = grad + beta * mom_new if nesterov else mom_new
    return mom_new, u


def orient(u):
    """Return (X, transposed): X = U for rows <= cols, else U^T, so X is m x n, m <= n."""
    u = np.asarray(u, dtype=np.float64)
    if u.shape[0] > u.shape[1]:
        return u.T, True
    return u, False


def frobenius_normalise(x, eps: float = EPS):
    """X0 = X / (||X||_F + eps): brings every singular value to at most 1."""
    x = np.asarray(x, dtype=np.float64)
    return x / (np.sqrt(np.sum(x * x)) + eps)


def ns_direct(x0, steps: int, coeffs=NS_COEFFS):
    """Direct Newton-Schulz in the m x n space: T steps of X <- a X + (b A + c A^2) X, A = X X^T."""
    a, b, c = coeffs
    x = np.asarray(x0, dtype=np.float64)
    for _ in range(steps):
        gram = x @ x.T
        poly = b * gram + c * (gram @ gram)
        x = a * x + poly @ x
    return x


def ns_gram(x0, steps: int, coeffs=NS_COEFFS):
    """Gram-space Newton-Schulz: carry R_k = X_k X_k^T and Q_k (X_k = Q_k X0) in m x m.

    R_0 = X0 X0^T, Q_0 = I; per step P = a I + b R + c R^2, Q <- P Q,
    R <- P R P; result Q_T X0.
    """
    a, b, c = coeffs
    x0 = np.asarray(x0, dtype=np.float64)
    m = x0.shape[0]
    eye = np.eye(m)
    r = x0 @ x0.T
    q = eye.copy()
    for _ in range(steps):
        p = a * eye + b * r + c * (r @ r)
        q = p @ q
        r = p @ r @ p
    return q @ x0


def shape_scale(rows: int, cols: int, rule: str = "aspect") -> float:
    """Update scale s: 'aspect' = sqrt(max(1, rows/cols)); 'rms' = 0.2*sqrt(max(rows, cols))."""
    if rule == "aspect":
        return float(np.sqrt(max(1.0, rows / cols)))
    if rule == "rms":
        return float(0.2 * np.sqrt(max(rows, cols)))
    raise ValueError(f"unknown scale rule {rule!r}")


def muon_update(w, o, lr: float, wd: float, scale: float):
    """Decoupled weight decay then the scaled orthogonalised step: (1 - lr*wd) W - lr*s*O."""
    w = np.asarray(w, dtype=np.float64)
    return (1.0 - lr * wd) * w - lr * scale * np.asarray(o, dtype=np.float64)


def muon_step(w, grad, mom, *, lr: float, beta: float, wd: float, ns_steps: int = 5,
              dtype: str = "bf16", coeffs=NS_COEFFS, eps: float = EPS,
              nesterov: bool = True, scale_rule: str = "aspect", method: str = "direct"):
    """One Muon step on one matrix, in fp64.

    Inputs hold values exactly representable in ``dtype``.  Returns a dict with
    ``W`` and ``M`` (rounded once to ``dtype``, as float64 arrays) and ``O``,
    the fp64 orthogonalised update in the original orientation.
    """
    w = np.asarray(w, dtype=np.float64)
    rows, cols = w.shape
    mom_new, u = nesterov_momentum(grad, mom, beta, nesterov)
    x, transposed = orient(u)
    x0 = frobenius_normalise(x, eps)
    if method == "direct":
        xt = ns_direct(x0, ns_steps, coeffs)
    elif method == "gram":
        xt = ns_gram(x0, ns_steps, coeffs)
    else:
        raise ValueError(f"unknown NS method {method!r}")
    o = xt.T if transposed else xt
    w_new = muon_update(w, o, lr, wd, shape_scale(rows, cols, scale_rule))
    return {"W": round_to_storage(w_new, dtype), "M": round_to_storage(mom_new, dtype), "O": o}


def muon_step_many(mats, **kw):
    """Apply ``muon_step`` to a list of (W, grad, mom) triples, each on its own."""
    return [muon_step(w, g, m, **kw) for (w, g, m) in mats]
