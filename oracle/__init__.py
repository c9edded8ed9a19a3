"""Plain fp64 CPU oracle for the batched Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (the CUDA library and its Python binding) never
imports, calls or links anything here, and nothing here imports the product.

Subject: "DMuon: Efficient Distributed Muon Training with Near-Adam Overhead"
(arXiv 2606.27153), as summarised on gist.science (pt and fr technical
summaries, sections 1-5) and in the English abstract on shd-paper.top.
"""
from .muon import (  # noqa: F401
    NS_COEFFS, EPS, round_to_bf16, round_to_fp32, round_to_storage,
    nesterov_momentum, orient, frobenius_normalise, ns_direct, ns_gram,
    shape_scale, muon_update, muon_step, muon_step_many,
)
from .plan import plan_buckets  # noqa: F401
