"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (relative Frobenius error of the orthogonalised update O): 3e-2 in
bf16 mode (tensor cores, bf16 operands, fp32 accumulation), 1e-4 in the fp32
validation mode.  Momentum: every element within 1 ulp of the oracle's single
rounding (the kernel rounds fl32(beta*M + grad) once more).  Parameters: every
element within one ulp plus the recovery rounding of O_gpu of
RN((1 - lr*wd) W - lr*s*O_gpu), O_gpu recovered through the ABI from the same
inputs, and 99 % within one ulp (bf16) or four ulps (fp32).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.helpers import TOL, f32, gpu_O, oracle_O, rel_fro, run_step, storage, ulp_diff, ulp_of

pytestmark = pytest.mark.gpu

BETA, LR, WD = f32(0.95), f32(0.02), f32(0.01)


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")


def make_inputs(shapes, dtype, seed, grad_scale=1e-3, mom_std=1e-3):
    cfg = workloads.Config("t", "test", dtype, seed, tuple(shapes), "normal", grad_scale=grad_scale,
                           mom_std=mom_std)
    return [workloads.make_matrix(cfg, i, "cpu") for i in range(len(shapes))]


def check_O(shapes, inputs, dtype, tol=None, ns_steps=5, **kw):
    got, muon = gpu_O(shapes, inputs, dtype, beta=BETA, ns_steps=ns_steps, **kw)
    want = oracle_O(inputs, beta=BETA, ns_steps=ns_steps)
    errs = [rel_fro(g, w) for g, w in zip(got, want)]
    if tol is None:
        tol = TOL["fp32"] if kw.get("precision", "bf16") == "fp32" else TOL["bf16"]
    worst = int(np.argmax(errs))
    assert errs[worst] <= tol, f"{shapes[worst]}: rel err {errs[worst]:.3e} > {tol}"
    return errs, muon


# ------------------------------------------------------------------ small and ragged

RAGGED = [(8, 16), (16, 8), (65, 130), (130, 65), (33, 33), (1, 37), (37, 1), (3, 500), (300, 300),
          (320, 704), (704, 320), (257, 600), (520, 1100), (1100, 520), (400, 520)]


def test_ragged_shapes_bf16():
    inputs = make_inputs(RAGGED, "bf16", 11)
    check_O(RAGGED, inputs, "bf16")


def test_ragged_shapes_fp32_validation():
    inputs = make_inputs(RAGGED, "fp32", 12)
    check_O(RAGGED, inputs, "fp32", precision="fp32")


def test_bf16_storage_fp32_validation_mode():
    # O is only visible through bf16 parameters here, so compare the stored
    # bits: fp32 arithmetic (error ~1e-6) rounds to the same bf16 as the oracle
    # up to one ulp where the exact value sits near a rounding boundary.
    shapes = [(96, 200), (200, 96), (150, 150), (320, 330)]
    inputs = make_inputs(shapes, "bf16", 13)
    w, _, _ = run_step(shapes, inputs, "bf16", lr=1.0, beta=BETA, wd=0.0, zero_w=True, precision="fp32")
    want = oracle_O(inputs, beta=BETA)
    for (r, c), wi, o in zip(shapes, w, want):
        s = oracle.shape_scale(r, c)
        ref = oracle.round_to_bf16(-s * o)
        # one bf16 ulp, plus the fp32 path's own error (1e-4 of the rms of s*O)
        # for elements near zero, whose ulp is far below that
        slack = 1e-4 * s * np.sqrt(np.mean(o * o))
        assert np.all(np.abs(wi.double().numpy() - ref) <= ulp_of(ref, "bf16") + slack), (r, c)
        d = ulp_diff(wi, torch.from_numpy(ref).to(torch.bfloat16))
        assert (d == 0).mean() > 0.97 and (d <= 1).mean() > 0.995, (r, c)


@pytest.mark.parametrize("route", ["gram", "direct"])
def test_forced_routes_rectangular(route):
    shapes = [(320, 704), (704, 320), (288, 1024), (64, 300)]
    inputs = make_inputs(shapes, "bf16", 14)
    check_O(shapes, inputs, "bf16", route=route, small_m=-1)


@pytest.mark.parametrize("ns_steps", [1, 2, 3, 4, 6])
def test_ns_step_counts(ns_steps):
    shapes = [(320, 704), (300, 320), (48, 200), (200, 48)]
    inputs = make_inputs(shapes, "bf16", 15)
    check_O(shapes, inputs, "bf16", ns_steps=ns_steps)


def test_momentum_and_update_ulps():
    shapes = [(320, 704), (704, 320), (300, 300), (48, 200), (65, 130)]
    for dtype in ("bf16", "fp32"):
        inputs = make_inputs(shapes, dtype, 16)
        prec = "bf16" if dtype == "bf16" else "fp32"
        w_new, m_new, _ = run_step(shapes, inputs, dtype, lr=LR, beta=BETA, wd=WD, precision=prec)
        o_gpu, _ = gpu_O(shapes, inputs, dtype, beta=BETA, precision=prec)
        st = storage(dtype)
        for i, (w, g, m) in enumerate(inputs):
            r, c = shapes[i]
            want_m = oracle.round_to_storage(BETA * m.double().numpy() + g.double().numpy(), dtype)
            assert ulp_diff(m_new[i], torch.from_numpy(want_m).to(st)).max() <= 1
            s = oracle.shape_scale(r, c)
            # The update applied to the kernel's own O.  o_gpu went through one
            # rounding to the storage dtype (relative 2^-9 for bf16, 2^-24 for
            # fp32), so each element may differ from the kernel's internal fp32
            # value by that much times lr*s*|O|, plus the final rounding.
            w64 = w.double().numpy()
            exact = (1 - LR * WD) * w64 - LR * s * o_gpu[i]
            want_w = oracle.round_to_storage(exact, dtype)
            got = w_new[i].double().numpy()
            # fp32 arithmetic in the kernel (decay*W and lr*s rounded, one fma)
            # costs up to about one ulp of max(|W|, |W'|); the recovered O adds
            # its own rounding (2^-9 bf16, 2^-24 fp32) times lr*s*|O|
            unit = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -23
            big = np.maximum(np.abs(want_w), np.abs(w64))
            bound = ulp_of(want_w, dtype) + ulp_of(big, "fp32") * 2 + 2 * unit * LR * s * np.abs(o_gpu[i])
            assert np.all(np.abs(got - want_w) <= bound), (shapes[i], dtype)
            # The fraction rule restates that bound for the typical element,
            # where |W'| is close to |W| (no cancellation).  The final fma
            # rounding and RN(exact) give one ulp.  fl(1 - lr wd) and fl(decay W)
            # add up to 2^-23 |W|: in bf16 that is 2^-15 of an ulp, in fp32 up
            # to two ulps of W'.  The recovered O adds about one fp32 ulp.  So:
            # bf16 one ulp, fp32 four; the per-element bound above covers the
            # elements near W' = 0.
            d = ulp_diff(w_new[i], torch.from_numpy(want_w).to(st))
            assert (d <= (1 if dtype == "bf16" else 4)).mean() >= 0.99, (shapes[i], dtype)


def test_momentum_many_one_tile_matrices():
    # About 1 800 one-tile matrices (half of them tall, so transposed) around a
    # few larger ragged ones: each block of the momentum kernel then jumps over
    # hundreds of matrices from one of its tiles to the next.
    shapes = [(8, 16)] * 900 + [(130, 65)] * 3 + [(16, 8)] * 900 + [(300, 300), (65, 130)]
    inputs = make_inputs(shapes, "bf16", 21)
    _, m_new, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    for i, (w, g, m) in enumerate(inputs):
        want_m = oracle.round_to_storage(BETA * m.double().numpy() + g.double().numpy(), "bf16")
        assert ulp_diff(m_new[i], torch.from_numpy(want_m).to(torch.bfloat16)).max() <= 1, (i, shapes[i])
    # the norms (per-warp partials of every tile) reach O
    picks = [0, 450, 899, 900, 902, 903, 1500, 1802, 1803, 1804]
    got, _ = gpu_O(shapes, inputs, "bf16", beta=BETA)
    want = oracle_O([inputs[i] for i in picks], beta=BETA)
    errs = [rel_fro(got[i], w) for i, w in zip(picks, want)]
    assert max(errs) <= TOL["bf16"], max(errs)


def test_momentum_tall_transposes_ragged_and_interleaved():
    # Tall matrices are transposed through shared memory, a quad of threads
    # per packed row: rows whose 64-row segment ends inside a tile (1000 and
    # 130 rows) are stored element-wise at their end, and rows of odd length
    # (65, 41 columns) are not on 16 bytes.  About 4 000 tiles over the
    # persistent blocks, each of which meets several kinds; the step is
    # repeated to catch a race on the shared tile.
    shapes = ([(1000, 136)] * 20 + [(1000, 130)] * 20 + [(130, 64)] * 60 + [(130, 65)] * 60
              + [(72, 40)] * 40 + [(75, 41)] * 40)
    inputs = make_inputs(shapes, "bf16", 23)
    w1, m_new, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    w2, _, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    for i, (w, g, m) in enumerate(inputs):
        want_m = oracle.round_to_storage(BETA * m.double().numpy() + g.double().numpy(), "bf16")
        assert ulp_diff(m_new[i], torch.from_numpy(want_m).to(torch.bfloat16)).max() <= 1, (i, shapes[i])
        assert torch.equal(w1[i], w2[i]), (i, shapes[i])
    picks = [0, 19, 20, 39, 40, 99, 100, 159, 160, 199, 200, 239]
    got, _ = gpu_O(shapes, inputs, "bf16", beta=BETA)
    want = oracle_O([inputs[i] for i in picks], beta=BETA)
    errs = [rel_fro(got[i], w) for i, w in zip(picks, want)]
    assert max(errs) <= TOL["bf16"], max(errs)


@pytest.mark.gpu
def test_flat_momentum_pass():
    # A wave whose wide bf16 matrices of at least 2^20 elements hold 2^26 or
    # more elements streams them through the flat (bulk-copy) momentum pass;
    # a 1000 x 1056 matrix ends in a partial chunk.  Alone, the same matrices
    # take the tile pass.  M' is the same element-wise formula either way
    # (bitwise equal, within one ulp of the oracle); O meets the bf16 bar.
    shapes = [(1024, 4096)] * 16 + [(1000, 1056)] * 2 + [(4096, 1024), (100, 300)]
    inputs = make_inputs(shapes, "bf16", 41)
    w_all, m_all, _ = run_step(shapes, inputs, "bf16", lr=1.0, beta=BETA, wd=0.0, zero_w=True)
    picks = [0, 16, 17, 18, 19]
    for i in picks:
        w_one, m_one, _ = run_step([shapes[i]], [inputs[i]], "bf16", lr=1.0, beta=BETA, wd=0.0, zero_w=True)
        assert torch.equal(m_one[0], m_all[i])
        w, g, m = inputs[i]
        want_m = oracle.round_to_storage(BETA * m.double().numpy() + g.double().numpy(), "bf16")
        assert ulp_diff(m_all[i], torch.from_numpy(want_m).to(torch.bfloat16)).max() <= 1
    want = oracle_O([inputs[i] for i in picks], beta=BETA)
    for i, o in zip(picks, want):
        r, c = shapes[i]
        got = -w_all[i].double().numpy() / oracle.shape_scale(r, c)
        assert rel_fro(got, o) <= TOL["bf16"], shapes[i]


def test_zero_gradient_gives_pure_decay():
    shapes = [(320, 704), (48, 200), (300, 300)]
    inputs = [(w, torch.zeros_like(g), torch.zeros_like(m)) for w, g, m in make_inputs(shapes, "bf16", 17)]
    w_new, m_new, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    for i, (w, _, _) in enumerate(inputs):
        want = oracle.round_to_bf16((1 - LR * WD) * w.double().numpy())
        assert ulp_diff(w_new[i], torch.from_numpy(want).to(torch.bfloat16)).max() <= 1
        assert torch.all(m_new[i] == 0)


def test_nesterov_off_and_rms_scale():
    shapes = [(320, 704), (704, 320), (48, 200)]
    inputs = make_inputs(shapes, "bf16", 18)
    got, _ = gpu_O(shapes, inputs, "bf16", beta=BETA, nesterov=False, scale_rule="rms")
    want = oracle_O(inputs, beta=BETA, nesterov=False)
    for g, w in zip(got, want):
        assert rel_fro(g, w) <= 3e-2


def test_deterministic_and_batching_invariant():
    shapes = [(320, 704)] * 3 + [(48, 200)] * 3 + [(300, 300)] * 2
    inputs = make_inputs(shapes, "bf16", 19)
    a, _, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    b, _, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    # each matrix alone gives the same bits as inside its bucket
    for i in (1, 4, 7):
        alone, _, _ = run_step([shapes[i]], [inputs[i]], "bf16", lr=LR, beta=BETA, wd=WD)
        assert torch.equal(alone[0], a[i])


def test_symmetric_operands_bitwise():
    # The R / A that the products read (bf16 on tensor cores; split into
    # [hi | lo] bf16 parts for small m) is stored as lower triangle plus
    # mirror: bitwise symmetric.  The fp32 copy kept for the next polynomial's
    # aux term holds the same lower triangle before rounding.  An fp32 mode
    # plan checks the FFMA engine's fp32 operand the same way.
    shapes = [(320, 704)] * 2 + [(300, 960)] + [(520, 1100)] + [(100, 400)] * 2
    inputs = make_inputs(shapes, "bf16", 20)
    _, _, muon = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    ws = muon.workspace
    buckets = muon.buckets()
    assert {b["route"] for b in buckets} == {1, 2} and {b["engine"] for b in buckets} == {0, 2}
    _check_symmetric_operands(muon, ws, buckets)
    _, _, m32 = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD, precision="fp32")
    assert {b["engine"] for b in m32.buckets()} == {1}
    _check_symmetric_operands(m32, m32.workspace, m32.buckets())
    # split operands over several 256-row pair tiles (small_m raised): hi and
    # lo parts mirrored across tiles; O to the oracle
    big = [(520, 1600), (1600, 520), (300, 1000)]
    big_in = make_inputs(big, "bf16", 24)
    _, _, ms = run_step(big, big_in, "bf16", lr=LR, beta=BETA, wd=WD, small_m=1024)
    assert {b["engine"] for b in ms.buckets()} == {2}
    _check_symmetric_operands(ms, ms.workspace, ms.buckets())
    check_O(big, big_in, "bf16", small_m=1024)


def _check_symmetric_operands(muon, ws, buckets):
    def matrices(p, which, m, nb, col0=0):
        off, ld, bs, dt = muon.debug_buffer(0, p, which)
        tdt, esz = (torch.bfloat16, 2) if dt == "bf16" else (torch.float32, 4)
        raw = ws[off: off + nb * bs * esz].view(tdt).cpu().view(nb, bs)
        return [raw[j, : m * ld].view(m, ld)[:, col0:col0 + m] for j in range(nb)], dt, ld

    for p, (bi, start, nb) in enumerate(muon.waves()[0]):
        m = buckets[bi]["m"]
        ops, dt, ld = matrices(p, 2, m, nb)
        split = buckets[bi]["engine"] == 2
        plain_tc = buckets[bi]["engine"] == 0  # bf16 operand only, no fp32 copy
        fps = matrices(p, 1, m, nb)[0] if not plain_tc else [None] * nb
        los = matrices(p, 2, m, nb, ld // 2)[0] if split else [None] * nb
        low = torch.tril(torch.ones(m, m, dtype=torch.bool))
        for op, fp, lo in zip(ops, fps, los):
            assert torch.equal(op, op.t())
            assert torch.isfinite(op.float()).all()
            if plain_tc:
                continue
            if dt == "bf16":
                assert torch.equal(fp.to(torch.bfloat16)[low], op[low])
            else:
                assert torch.equal(fp, op)
            if split:
                # lo = bf16(R - hi), R - hi exact in fp32; symmetric like hi
                assert torch.equal(lo, lo.t())
                assert torch.equal((fp - op.float()).to(torch.bfloat16)[low], lo[low])


def test_workspace_budget_waves():
    shapes = [(320, 704)] * 5 + [(300, 300)] * 3 + [(48, 200)] * 4
    inputs = make_inputs(shapes, "bf16", 21)
    full, _, _ = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD)
    from matrix_orthogonalising_optimizer_gb300 import Muon
    probe = Muon([(r, c, 0) for r, c in shapes])
    big = max(b["per_matrix_bytes"] for b in probe.buckets())
    waved, _, muon = run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD, workspace_budget=2 * big)
    assert len(muon.waves()) > 2
    for x, y in zip(full, waved):
        assert torch.equal(x, y)


def test_timing_counts_launches():
    shapes = [(320, 704), (48, 200), (300, 300)]
    inputs = make_inputs(shapes, "bf16", 22)
    from matrix_orthogonalising_optimizer_gb300 import Muon
    muon = Muon([(r, c, 0) for r, c in shapes]).bind()
    muon.set_timing(True)
    run_step(shapes, inputs, "bf16", lr=LR, beta=BETA, wd=WD, muon=muon)
    t = muon.timing()
    assert t["momentum"][1] == 1 and t["norm"][1] == 1
    # bf16 mode: every product on tensor cores (small m through split operands)
    assert t["tc"][1] > 0 and t["simt"][1] == 0
    assert all(v[0] >= 0 for v in t.values())


# ------------------------------------------------------------------ configurations


def test_c1_single_fp32():
    cfg = workloads.get("c1")
    inputs = [workloads.make_matrix(cfg, 0, "cpu")]
    errs, _ = check_O(list(cfg.shapes), inputs, "fp32", precision="fp32")
    assert errs[0] <= 1e-4


def test_c2_small_transformer():
    cfg = workloads.get("c2")
    inputs = [workloads.make_matrix(cfg, i, "cpu") for i in range(len(cfg.shapes))]
    errs, muon = check_O(list(cfg.shapes), inputs, "bf16")
    assert len(muon.buckets()) == 3


def test_c4_heterogeneous_sampled():
    cfg = workloads.get("c4")
    shapes = list(cfg.shapes)
    inputs = [workloads.make_matrix(cfg, i, "cpu") for i in range(len(shapes))]
    got, muon = gpu_O(shapes, inputs, "bf16", beta=BETA)
    # every bucket's first member, plus a seeded sample
    picks = {b["members"][0] for b in muon.buckets()}
    rng = np.random.default_rng(3)
    picks |= set(int(i) for i in rng.choice(len(shapes), 60, replace=False))
    picks = sorted(picks)
    want = oracle_O([inputs[i] for i in picks], beta=BETA)
    errs = [rel_fro(got[i], w) for i, w in zip(picks, want)]
    assert max(errs) <= 3e-2, max(errs)


# ------------------------------------------------------------------ full-size sets, sampled


def _full_size_sampled(name, picks):
    """Whole set generated on the GPU and stepped in bench.py's launch
    configuration; sampled matrices checked against the oracle one by one on
    the host.  The first step is the real update (lr, wd of the set): its W'
    is compared with the oracle's W' (check_update_against_oracle).  The
    second step, from W = 0, lr = 1, wd = 0 and the momenta back at their
    initial zeros, exposes O for the O parity."""
    import gc

    from matrix_orthogonalising_optimizer_gb300 import Muon
    from tests.helpers import check_update_against_oracle
    cfg = workloads.get(name)
    assert cfg.mom_std == 0.0  # the momenta start at zero, so they can be reset
    lr, wd = f32(cfg.lr), f32(cfg.wd)
    gc.collect()
    torch.cuda.empty_cache()
    muon = Muon([(r, c, 0) for r, c in cfg.shapes], workspace_budget=int(cfg.budget_gb * (1 << 30))).bind()
    ws, gs, ms = workloads.make_set(cfg, "cuda")
    w_in = {i: ws[i].cpu() for i in picks}
    muon.step(ws, gs, ms, lr, BETA, wd, cfg.ns_steps)
    torch.cuda.synchronize()
    assert muon.device_status() == 0
    w_new = {i: ws[i].cpu() for i in picks}
    for w in ws:
        w.zero_()
    for m in ms:
        m.zero_()
    muon.step(ws, gs, ms, 1.0, BETA, 0.0, cfg.ns_steps)
    torch.cuda.synchronize()
    assert muon.device_status() == 0
    errs = {}
    for i in picks:
        r, c = cfg.shapes[i]
        g = gs[i].cpu()
        o_gpu = -ws[i].double().cpu().numpy() / oracle.shape_scale(r, c)
        # momenta were zero: M' = grad bitwise
        assert torch.equal(ms[i].cpu(), g)
        want = oracle.muon_step(w_in[i].double().numpy(), g.double().numpy(), np.zeros((r, c)), lr=lr, beta=BETA,
                                wd=wd, ns_steps=cfg.ns_steps)
        errs[(i, r, c)] = rel_fro(o_gpu, want["O"])
        check_update_against_oracle(w_new[i], w_in[i], want["W"], want["O"], lr=lr, wd=wd,
                                    scale=oracle.shape_scale(r, c), dtype="bf16", tau=TOL["bf16"])
    del ws, gs, ms, muon
    gc.collect()
    torch.cuda.empty_cache()
    assert max(errs.values()) <= 3e-2, errs
    return errs


def test_c3_llama_full_size_sampled():
    # one matrix per bucket: k (1024x4096, Gram), q (4096^2, direct), gate (14336x4096, tall, Gram),
    # down (4096x14336, wide, Gram)
    _full_size_sampled("c3", [1, 0, 4, 6])


def test_c5_large_layers_full_size_sampled():
    free, total = torch.cuda.mem_get_info()
    if free < 280e9:
        pytest.skip(f"needs about 280 GB free, {free / 1e9:.0f} GB free")
    # 8192^2 (direct) and 28672x8192 (tall, Gram)
    _full_size_sampled("c5", [0, 1])


def test_step_replays_from_a_cuda_graph():
    # After one eager step has uploaded the pointer table, dmuon_step issues
    # only stream work (memsets and launches): it can be captured once and
    # replayed, with bitwise the same results as eager steps.
    from matrix_orthogonalising_optimizer_gb300 import Muon
    shapes = [(320, 704), (704, 320), (300, 300), (64, 256), (1100, 520)]
    inputs = make_inputs(shapes, "bf16", 41)
    state = []
    for _ in range(2):
        muon = Muon([(r, c, 0) for r, c in shapes]).bind()
        ws = [w.cuda() for w, _, _ in inputs]
        gs = [g.cuda() for _, g, _ in inputs]
        ms = [m.cuda().clone() for _, _, m in inputs]
        state.append((muon, ws, gs, ms))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for muon, ws, gs, ms in state:
            muon.step(ws, gs, ms, LR, BETA, WD, 5, side)
        muon, ws, gs, ms = state[1]
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            muon.step(ws, gs, ms, LR, BETA, WD, 5, side)
    torch.cuda.current_stream().wait_stream(side)
    e_muon, e_ws, e_gs, e_ms = state[0]
    for _ in range(3):
        e_muon.step(e_ws, e_gs, e_ms, LR, BETA, WD, 5)
        graph.replay()
    torch.cuda.synchronize()
    assert e_muon.device_status() == 0 and state[1][0].device_status() == 0
    for a, b in zip(e_ws + e_ms, ws + ms):
        assert torch.equal(a, b)


def test_step_ex_waits_for_params_ready_before_the_update():
    # dmuon_step_ex: the stream waits for params_ready only before the first
    # parameter write.  An event held back ~50 ms by a spin kernel on another
    # stream delays the step's end by about that much, and the result equals
    # dmuon_step's.
    from matrix_orthogonalising_optimizer_gb300 import Muon
    shapes = [(320, 704), (300, 300)]
    inputs = make_inputs(shapes, "bf16", 43)
    outs = []
    for use_event in (False, True):
        muon = Muon([(r, c, 0) for r, c in shapes]).bind()
        ws = [w.cuda() for w, _, _ in inputs]
        gs = [g.cuda() for _, g, _ in inputs]
        ms = [m.cuda().clone() for _, _, m in inputs]
        muon.step(ws, gs, ms, LR, BETA, WD, 5)  # uploads the pointer table
        torch.cuda.synchronize()
        other = torch.cuda.Stream()
        ready = torch.cuda.Event()
        with torch.cuda.stream(other):
            torch.cuda._sleep(100_000_000)  # about 50 ms of spinning
            ready.record(other)
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        muon.step(ws, gs, ms, LR, BETA, WD, 5, params_ready=ready if use_event else None)
        t1.record()
        torch.cuda.synchronize()
        assert muon.device_status() == 0
        outs.append((t0.elapsed_time(t1), [w.cpu() for w in ws]))
    (t_plain, w_plain), (t_wait, w_wait) = outs
    assert t_wait > t_plain + 20.0, (t_plain, t_wait)
    for a, b in zip(w_plain, w_wait):
        assert torch.equal(a, b)
