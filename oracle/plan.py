"""Brute-force restatement of the shape-bucketing planner's rules.

TEST INFRASTRUCTURE ONLY: the product never imports this module.

Batching of like shapes is the DMuon summary's section 2.2 ("Agrupamento
(Batching)": matrices of similar shape run the Gram NS recurrence together so
small ones do not leave the GPU idle).  The rules restated here are those the
C ABI header ``include/dmuon.h`` states for ``dmuon_plan``:

* canonical shape: m = min(rows, cols), n = max(rows, cols); tall matrices
  (rows > cols) are packed transposed;
* input order inside a bucket;
* route per matrix: its own rule if the shape gives one, else the plan's;
  FP32 precision -> Gram unless the rule is DIRECT; AUTO -> Gram when
  n >= 3m or m <= small_m, else direct;
* tile rule per matrix: its own if the shape gives one, else the plan's
  (AUTO meaning PACKED); SINGLE where packing does not apply (m > 128, FP32);
* buckets keyed (dtype, m, n, route, tile), ascending;
* m x m engine: FP32 precision -> fp32 FFMA; BF16 precision -> split-bf16
  tensor cores for Gram buckets with m <= small_m, plain bf16 tensor cores
  otherwise;
* per-matrix workspace bytes: the sum of the per-matrix buffers below, each
  rounded up to 256 bytes;
* waves: buckets packed greedily in bucket order under the budget, a bucket
  split across waves where it does not fit (budget 0: one wave).

Everything is plain Python integers; the result must equal the library's
plan bit for bit.
"""
from __future__ import annotations

BF16, FP32 = 0, 1
PREC_BF16, PREC_FP32 = 0, 1
ROUTE_AUTO, ROUTE_GRAM, ROUTE_DIRECT = 0, 1, 2
BUCKET_GRAM, BUCKET_DIRECT = 1, 2
ENGINE_TC_BF16, ENGINE_SIMT_FP32, ENGINE_TC_SPLIT = 0, 1, 2
TILE_AUTO, TILE_PACKED, TILE_SINGLE = 0, 1, 2


def _up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def per_matrix_bytes(m: int, n: int, precision: int, route: int, engine: int) -> int:
    ex = 2 if precision == PREC_BF16 else 4
    ldn, ldm = _up(n, 8), _up(m, 8)
    bufs = [m * ldn * ex]                       # packed u
    if route == BUCKET_GRAM:
        if engine == ENGINE_TC_BF16:
            bufs += [m * ldm * 2] * 5                      # R, P, Q0, Q1, RP (bf16)
        elif engine == ENGINE_TC_SPLIT:
            # Rf; R, P, Q0, Q1, RP as bf16 rows [hi | lo], each part m rounded up to 64
            bufs += [m * ldm * 4] + [m * 2 * _up(m, 64) * 2] * 5
        else:
            bufs += [m * ldm * 4] * 5                      # R, P, Q0, Q1, RP (fp32 mode)
    else:
        if precision == PREC_BF16:
            bufs += [m * ldn * 2, m * ldm * 2, m * ldm * 2]              # X1; A, B (bf16)
        else:
            bufs += [m * ldn * 4, m * ldm * 4, m * ldm * 4]              # X1; A, B
    bufs += [4 * 8 * ((m + 63) // 64) * ((n + 63) // 64)]  # sum-of-squares partials: 8 per 64 x 64 tile
    return sum(_up(b, 256) for b in bufs)


def plan_buckets(shapes, precision: int = PREC_BF16, route: int = ROUTE_AUTO,
                 small_m: int = 0, budget: int = 0, tile: int = TILE_AUTO):
    """shapes: list of (rows, cols, dtype[, route[, tile]]).  Returns (buckets, waves).

    buckets: list of dicts with dtype, m, n, members (input indices), route,
    engine, tile, per_matrix_bytes.  waves: list of lists of (bucket, start, count).
    """
    plan_tile = TILE_PACKED if tile == TILE_AUTO else tile

    def resolve_tile(own, m):
        if precision == PREC_FP32 or m > 128:
            return TILE_SINGLE
        return own if own != TILE_AUTO else plan_tile

    if small_m == 0:
        small_m = 256
    def resolve(rule, m, n):
        if precision == PREC_FP32:
            return BUCKET_DIRECT if rule == ROUTE_DIRECT else BUCKET_GRAM
        if rule == ROUTE_GRAM:
            return BUCKET_GRAM
        if rule == ROUTE_DIRECT:
            return BUCKET_DIRECT
        return BUCKET_GRAM if (n >= 3 * m or (small_m > 0 and m <= small_m)) else BUCKET_DIRECT

    keyed = {}
    for idx, shp in enumerate(shapes):
        rows, cols, dtype = shp[:3]
        own = shp[3] if len(shp) > 3 else ROUTE_AUTO
        own_tile = shp[4] if len(shp) > 4 else TILE_AUTO
        m, n = min(rows, cols), max(rows, cols)
        key = (dtype, m, n, resolve(own if own != ROUTE_AUTO else route, m, n), resolve_tile(own_tile, m))
        keyed.setdefault(key, []).append(idx)
    buckets = []
    for key in sorted(keyed):
        dtype, m, n, r, t = key
        if precision == PREC_FP32:
            eng = ENGINE_SIMT_FP32
        elif r == BUCKET_GRAM and small_m > 0 and m <= small_m:
            eng = ENGINE_TC_SPLIT
        else:
            eng = ENGINE_TC_BF16
        buckets.append({"dtype": dtype, "m": m, "n": n, "members": keyed[key], "route": r,
                        "engine": eng, "tile": t, "per_matrix_bytes": per_matrix_bytes(m, n, precision, r, eng)})
    waves = []
    if budget == 0:
        waves.append([(b, 0, len(bk["members"])) for b, bk in enumerate(buckets)])
        return buckets, waves
    cur, used = [], 0
    for b, bk in enumerate(buckets):
        pmb = bk["per_matrix_bytes"]
        if pmb > budget:
            raise ValueError("budget smaller than one matrix")
        start, left = 0, len(bk["members"])
        while left > 0:
            fit = (budget - used) // pmb
            if fit == 0:
                waves.append(cur)
                cur, used = [], 0
                continue
            take = min(fit, left)
            cur.append((b, start, take))
            used += take * pmb
            start += take
            left -= take
    if cur:
        waves.append(cur)
    return buckets, waves
