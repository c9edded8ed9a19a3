"""AdamW step in fp64: the element-wise optimizer the DMuon pages compare against.

TEST INFRASTRUCTURE ONLY: the product never imports this module.

The pages report DMuon's step time relative to AdamW (gist.science technical
summary, section 4, "+2 %") but do not restate AdamW; this is the published
AdamW (Loshchilov & Hutter, decoupled weight decay) with Adam's bias
correction, the form the C ABI header states for ``dmuon_adamw_step``:

    m = beta1*m + (1-beta1)*g
    v = beta2*v + (1-beta2)*g^2
    W = (1 - lr*wd)*W - lr/(1-beta1^t) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)

Everything in float64 from the stored values, then one rounding to the
storage dtype.
"""
from __future__ import annotations

import numpy as np

from .muon import round_to_storage


def adamw_step(w, g, m, v, *, lr: float, beta1: float, beta2: float, eps: float, wd: float, step: int,
               dtype: str = "bf16"):
    """(W', m', v') rounded to ``dtype``, and the unrounded float64 values."""
    w = np.asarray(w, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m = np.asarray(m, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    m1 = beta1 * m + (1.0 - beta1) * g
    v1 = beta2 * v + (1.0 - beta2) * g * g
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    w1 = (1.0 - lr * wd) * w - (lr / bc1) * m1 / (np.sqrt(v1) / np.sqrt(bc2) + eps)
    exact = (w1, m1, v1)
    return tuple(round_to_storage(x, dtype) for x in exact), exact
