"""Owner assignment: brute-force optimum and the longest-processing-time rule.

TEST INFRASTRUCTURE ONLY: the product never imports this module.

DMuon technical summary (gist.science), section 2.3 "compute-aware load
balancing": each matrix gets one owner rank; the assignment minimises the
predicted makespan, the largest per-rank sum of predicted costs (a
mixed-integer program), with a greedy heuristic as the fallback for large
instances.

* ``makespan`` is the definition: every rank's costs summed in increasing
  matrix index, then the maximum.
* ``brute_force`` is the optimum by enumeration of every assignment of
  ``count`` matrices to ``ranks`` ranks (``ranks ** count`` of them: tiny
  instances only).
* ``lpt`` restates the greedy rule the C ABI header gives for
  ``DMUON_ASSIGN_GREEDY`` (longest processing time first: decreasing cost,
  ties by lower index; each to the least-loaded rank, ties by lower rank),
  with its load sums taken in the same order.
"""
from __future__ import annotations

import itertools


def makespan(costs, ranks, owner) -> float:
    load = [0.0] * ranks
    for i, c in enumerate(costs):
        load[owner[i]] += float(c)
    return max(load) if costs else 0.0


def brute_force(costs, ranks):
    """(optimal makespan, one optimal assignment) by enumeration."""
    best, best_owner = None, None
    for owner in itertools.product(range(ranks), repeat=len(costs)):
        ms = makespan(costs, ranks, owner)
        if best is None or ms < best:
            best, best_owner = ms, list(owner)
    if best is None:
        return 0.0, []
    return best, best_owner


def lpt(costs, ranks):
    """(assignment, makespan) of the longest-processing-time-first rule."""
    order = sorted(range(len(costs)), key=lambda i: (-float(costs[i]), i))
    load = [0.0] * ranks
    owner = [0] * len(costs)
    for i in order:
        r = min(range(ranks), key=lambda q: (load[q], q))
        owner[i] = r
        load[r] += float(costs[i])
    return owner, makespan(costs, ranks, owner)
