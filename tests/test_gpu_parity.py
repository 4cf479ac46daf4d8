"""GPU parity: every entry point of libattnres.so against the fp64 oracle.

Inputs come from transformer_depth_wise_gb300.workloads (seeded); the oracle
sees the exact same values widened to float64.  Tolerances (max |error|):
fp32 I/O 1e-5 * max|v|, bf16 I/O 8e-3 * max|v|, max|v| over the call's
input sources.  Statistics (m, lse): 2e-5 * max(1, |lse|) where the scores
are fp32 dot products; 1e-4 * max(1, |lse|) for bf16 phase 1, whose scores
use the query split into bf16 hi + lo parts (about 2^-17 relative per
element, summed over D terms).  Small cases span
several CTAs and a ragged tail of rows; full-size cases run the launch the
benchmark times and compare sampled token rows, which the oracle computes
one by one (depth attention never mixes tokens).
"""
import numpy as np
import pytest
import torch

import oracle
from transformer_depth_wise_gb300 import _lib, api
from transformer_depth_wise_gb300 import workloads as wk

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 8e-3}
ODT = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16}


def f64(t):
    return t.detach().double().cpu().numpy()


def vmax(tensors):
    return max(float(t.abs().max()) for t in tensors)


def check(got, want, tol_abs, what=""):
    err = float(np.max(np.abs(f64(got) - want))) if want.size else 0.0
    assert err <= tol_abs, f"{what}: max |err| {err:.3e} > {tol_abs:.3e}"
    return err


# Regression guard for the bf16 block chains, beside the chain tolerance of
# 8e-3 * max|v| over the summaries (about 0.29 at their scale).  The GPU and
# the oracle round at the same points and differ only where fp32 and fp64
# land on either side of a rounding boundary; such a flip in p_k carries on
# through the later updates, so single elements can end a few ulps apart
# (up to 2^-6 * max|p| has been seen over 100k sampled elements), but most
# elements agree exactly.  The guard bounds the root-mean-square error by
# 2^-8 of the compared tensor's own RMS: a few-percent error in one merge's
# weights shifts most elements of every later sublayer by several ulps and
# fails it, while the rare flips stay far below it.
CHAIN_RMS_GUARD = 2.0 ** -8


def check_chain(got, want, what=""):
    d = f64(got) - want
    rms_err = float(np.sqrt(np.mean(d * d)))
    rms = float(np.sqrt(np.mean(want * want)))
    assert rms_err <= CHAIN_RMS_GUARD * rms, \
        f"{what} (regression guard): rms err {rms_err:.3e} > {CHAIN_RMS_GUARD:.3g} * rms {rms:.3e}"
    return rms_err


STATS_TOL = 2e-5           # fp32 score arithmetic
STATS_TOL_SPLIT_Q = 1e-4   # bf16 phase 1: query as bf16 hi + lo


def check_stats(got, want, what="", tol=STATS_TOL):
    g = f64(got)
    err = np.abs(g - want) / np.maximum(1.0, np.abs(want))
    assert float(err.max()) <= tol, f"{what}: stats rel err {float(err.max()):.3e} > {tol:.1e}"


def rand_sources(n, shape, dtype, dev, seed, lo=0.5, hi=8.0):
    g = wk.generator(seed, dev)
    srcs, _ = wk.scaled_normal_sources(g, n, shape, lo, hi, dtype, dev)
    w, gam = wk.queries_and_gains(g, 1, shape[-1], dev)
    return srcs, w[0].contiguous(), gam[0].contiguous()


# --------------------------------------------------------------------------
# depth aggregation
# --------------------------------------------------------------------------
def test_aggregate_full_single_f32_config(gpu):
    wl = wk.WORKLOADS["full_single_f32"]
    for zero in (False, True):
        inp = wk.single_aggregation_inputs(wl, device=gpu, zero_query=zero)
        out, m, lse = api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"],
                                          stats=True)
        V = np.stack([f64(s) for s in inp["sources"]])
        h, om, olse = oracle.depth_aggregate(V, f64(inp["query"]), f64(inp["gain"]), inp["eps"])
        tol = TOL[torch.float32] * vmax(inp["sources"])
        check(out, oracle.round_to(h, oracle.F32), tol, "cfg1")
        check_stats(m, om, "m")
        check_stats(lse, olse, "lse")
        if zero:   # zero query: the mean of the sources
            check(out, V.mean(0), tol, "zero query mean")


CASES = [  # (dtype, D, n, rows) -- covers warp teams of 4..32 lanes and CTA teams, ragged rows
    (torch.bfloat16, 8, 3, 37), (torch.bfloat16, 24, 2, 65), (torch.bfloat16, 64, 5, 33),
    (torch.bfloat16, 256, 4, 129), (torch.bfloat16, 520, 7, 19), (torch.bfloat16, 1032, 9, 23),
    (torch.bfloat16, 2048, 10, 300), (torch.bfloat16, 4096, 9, 41), (torch.bfloat16, 7168, 10, 17),
    (torch.bfloat16, 8192, 3, 5), (torch.float32, 4, 2, 9), (torch.float32, 12, 5, 50),
    (torch.float32, 256, 5, 64), (torch.float32, 264, 6, 31), (torch.float32, 4096, 4, 13),
    # several source groups with a ragged tail, and a Full-stack-sized source list
    (torch.float32, 1024, 37, 7), (torch.float32, 2056, 19, 21), (torch.bfloat16, 2048, 187, 6),
]


@pytest.mark.parametrize("dtype,D,n,rows", CASES)
def test_aggregate_shapes(gpu, dtype, D, n, rows):
    srcs, q, g = rand_sources(n, (1, rows, D), dtype, gpu, seed=D * 31 + n * 7 + rows)
    out, m, lse = api.depth_aggregate(srcs, q, g, 1e-8, stats=True)
    V = np.stack([f64(s) for s in srcs])
    h, om, olse = oracle.depth_aggregate(V, f64(q), f64(g), 1e-8)
    check(out, oracle.round_to(h, ODT[dtype]), TOL[dtype] * vmax(srcs), f"D={D} n={n}")
    check_stats(lse, olse, "lse")
    check_stats(m, om, "m")


# Few sources over short bf16 rows of 2048 (the pipelined kernel's group
# chain at 1..13 sources, several rows per CTA, a ragged last round).
@pytest.mark.parametrize("n,rows", [(1, 1000), (5, 457), (8, 1000), (9, 1000), (13, 2049)])
def test_aggregate_short_rows(gpu, n, rows):
    srcs, q, g = rand_sources(n, (1, rows, 2048), torch.bfloat16, gpu, seed=5 * n + rows)
    out, m, lse = api.depth_aggregate(srcs, q, g, 1e-8, stats=True)
    V = np.stack([f64(s) for s in srcs])
    h, om, olse = oracle.depth_aggregate(V, f64(q), f64(g), 1e-8)
    check(out, oracle.round_to(h, oracle.BF16), TOL[torch.bfloat16] * vmax(srcs), f"n={n} rows={rows}")
    check_stats(lse, olse, "lse")
    check_stats(m, om, "m")


def _random_shapes(seed, count, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(count)]


def test_aggregate_random_shapes(gpu):
    """Seeded random shapes (dtype, D, n, token rows) against the oracle: widths from 4 to 8192 elements,
    1..40 sources, 1..3000 rows, kept to a few million elements each."""
    def draw(rng):
        dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
        step, top = (8, 8192) if dtype == torch.bfloat16 else (4, 4096)
        D = int(rng.integers(1, top // step + 1)) * step
        n = int(rng.integers(1, 41))
        rows = int(rng.integers(1, 3001))
        rows = max(1, min(rows, 4_000_000 // (n * D)))
        return dtype, D, n, rows
    for i, (dtype, D, n, rows) in enumerate(_random_shapes(2024, 40, draw)):
        srcs, q, g = rand_sources(n, (1, rows, D), dtype, gpu, seed=900 + i)
        out, m, lse = api.depth_aggregate(srcs, q, g, 1e-8, stats=True)
        h, om, olse = oracle.depth_aggregate(np.stack([f64(s) for s in srcs]), f64(q), f64(g), 1e-8)
        check(out, oracle.round_to(h, ODT[dtype]), TOL[dtype] * vmax(srcs), f"case {i}: {dtype} D={D} n={n} rows={rows}")
        check_stats(lse, olse, f"case {i} lse")


def test_phase1_random_shapes(gpu):
    """Seeded random phase-1 shapes against the oracle: bf16 and fp32, 1..16 summaries, 1..24 queries,
    widths up to 4096, 1..1200 rows (the tensor-core path from 512 bf16 rows, split mode from 64, the
    per-row kernel below)."""
    def draw(rng):
        dtype = torch.bfloat16 if rng.random() < 0.75 else torch.float32
        elt = 2 if dtype == torch.bfloat16 else 4
        n = int(rng.integers(1, 17))
        S = int(rng.integers(1, 25))
        D = int(rng.integers(1, 65)) * 64
        D = min(D, (200 * 1024) // (n * elt) // 64 * 64) or 64
        rows = int(rng.integers(1, 1201))
        rows = max(1, min(rows, 60_000_000 // (n * S * D)))
        return dtype, D, n, S, rows
    ran = 0
    for i, (dtype, D, n, S, rows) in enumerate(_random_shapes(2025, 30, draw)):
        g = wk.generator(700 + i, gpu)
        blocks, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, dtype, gpu)
        W, G = wk.queries_and_gains(g, S, D, gpu)
        try:
            o, m, lse = api.block_phase1(blocks, W, G, 1e-8, want_max=True)
        except _lib.AttnResError as e:   # a shape no phase-1 kernel takes (refused before anything runs)
            assert "SHAPE" in str(e), str(e)
            continue
        ran += 1
        O, M, LSE = oracle.block_phase1([f64(b) for b in blocks], f64(W), f64(G), 1e-8)
        tol = TOL[dtype] * vmax(blocks)
        what = f"case {i}: {dtype} D={D} n={n} S={S} rows={rows}"
        check(o.reshape(S, rows, D), oracle.round_to(O, ODT[dtype]), tol, what)
        check_stats(lse.reshape(S, rows), LSE, what + " lse", STATS_TOL_SPLIT_Q)
    assert ran >= 25, ran


def test_full_two_phase_random_shapes(gpu):
    """Seeded random Full two-phase schedules against the oracle: bf16, widths a multiple of 64 up to 2048,
    2..30 sublayers in blocks of 1..24, 48..400 token rows."""
    def draw(rng):
        D = int(rng.integers(1, 33)) * 64
        L = int(rng.integers(2, 31))
        S = int(rng.integers(1, 25))
        rows = int(rng.integers(48, 401))
        rows = max(48, min(rows, 30_000_000 // (L * L * D)))
        return D, L, S, rows
    wl = wk.WORKLOADS["full_stack_bf16"]
    for i, (D, L, S, rows) in enumerate(_random_shapes(2026, 10, draw)):
        inp = wk.full_stack_inputs(wl, rows=rows, device=gpu, L=L, D=D)
        y, srcs = api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"])
        V, oy = oracle.full_stack_two_phase(f64(inp["v0"]).reshape(rows, D), f64(inp["queries"]),
                                            f64(inp["gains"]), f64(inp["u"]), S, inp["eps"], oracle.BF16)
        tol = TOL[torch.bfloat16] * float(inp["v0"].abs().max())
        what = f"case {i}: D={D} L={L} S={S} rows={rows}"
        for l in (1, L // 2, L):
            check(srcs[l].reshape(rows, D), V[l], tol, f"{what} v_{l}")
        check(y.reshape(rows, D), oracle.round_to(oy, oracle.BF16), tol, f"{what} y")


def test_aggregate_one_source_is_identity_bitwise(gpu):
    for dtype, D in ((torch.bfloat16, 2048), (torch.float32, 256), (torch.bfloat16, 40)):
        srcs, q, g = rand_sources(1, (2, 33, D), dtype, gpu, seed=5)
        out = api.depth_aggregate(srcs, q, g, 1e-8)
        assert torch.equal(out, srcs[0])


def test_aggregate_no_mixing_across_tokens_bitwise(gpu):
    srcs, q, g = rand_sources(10, (4, 64, 2048), torch.bfloat16, gpu, seed=11)
    out0 = api.depth_aggregate(srcs, q, g, 1e-8).clone()
    srcs2 = [s.clone() for s in srcs]
    for s in srcs2:
        s[2, 17] = -s[2, 17] * 3
    out1 = api.depth_aggregate(srcs2, q, g, 1e-8)
    mask = torch.ones(4, 64, dtype=torch.bool, device=gpu)
    mask[2, 17] = False
    assert torch.equal(out0[mask], out1[mask])
    assert not torch.equal(out0[2, 17], out1[2, 17])


def test_aggregate_empty_rows_is_a_noop(gpu):
    srcs = [torch.empty((0, 5, 256), dtype=torch.bfloat16, device=gpu) for _ in range(3)]
    q = torch.zeros(256, device=gpu)
    out = api.depth_aggregate(srcs, q, None, 1e-8)
    assert out.shape == (0, 5, 256)


def test_empty_rows_every_entry_point(gpu):
    """B*T = 0: every entry point returns at once (empty tensors may carry NULL data), and the backward's
    parameter gradients come back as zeros."""
    D, shape, bf = 256, (0, 5, 256), torch.bfloat16
    srcs = [torch.empty(shape, dtype=bf, device=gpu) for _ in range(3)]
    q = torch.randn(D, device=gpu)
    g = torch.ones(D, device=gpu)
    qs = torch.randn((4, D), device=gpu)
    o, _, lse = api.block_phase1(srcs, qs, None, 1e-8)
    assert o.shape == (4, 0, 5, D) and lse.shape == (4, 0, 5)
    x = torch.empty(shape, dtype=bf, device=gpu)
    lse1 = torch.empty((0, 5), dtype=torch.float32, device=gpu)
    assert api.block_phase2_merge(x, lse1, x, q, g, 1e-8).shape == shape
    p_out, h_out, _ = api.block_merge_update(x, lse1, x, x, q, q, g, 1e-8)
    assert p_out.shape == shape and h_out.shape == shape
    assert api.rms_norm(x, g).shape == shape
    assert api.partial_update(x, x, q).shape == shape
    qL, uL = torch.randn((7, D), device=gpu), torch.randn((6, D), device=gpu)
    y, vs = api.full_stack_forward(x, qL, None, uL, 1e-8)
    assert y.shape == shape and len(vs) == 7
    y, vs = api.full_stack_two_phase(x, qL, None, uL, 3, 1e-8)
    assert y.shape == shape and len(vs) == 7
    gs, gq, gg = api.depth_aggregate_backward(srcs, q, g, 1e-8, x)
    assert len(gs) == 3 and gs[0].shape == shape
    assert torch.count_nonzero(gq) == 0 and torch.count_nonzero(gg) == 0


def test_aggregate_many_sources(gpu):
    srcs, q, g = rand_sources(187, (1, 9, 256), torch.bfloat16, gpu, seed=187)
    out = api.depth_aggregate(srcs, q, g, 1e-8)
    h, _, _ = oracle.depth_aggregate(np.stack([f64(s) for s in srcs]), f64(q), f64(g), 1e-8)
    check(out, h, TOL[torch.bfloat16] * vmax(srcs), "n=187")


def test_gain_absent_is_a_gain_of_one_bitwise(gpu):
    """gain = NULL is a gain of one: the folded query w (.) 1 is w exactly, so every path gives bitwise the
    result of an all-ones gain (the aggregation on its pipelined and team kernels, phase 1 on the tensor
    cores and per row, the fused step on its few-row and CTA kernels, and the backward's gradients)."""
    for D, n, rows, dtype in ((2048, 10, 600, torch.bfloat16), (256, 5, 33, torch.bfloat16),
                              (512, 4, 70, torch.float32)):
        srcs, q, _ = rand_sources(n, (1, rows, D), dtype, gpu, seed=D + n)
        ones = torch.ones(D, device=gpu)
        assert torch.equal(api.depth_aggregate(srcs, q, None, 1e-8), api.depth_aggregate(srcs, q, ones, 1e-8))
    for rows in (600, 40):
        blocks, _, _ = rand_sources(9, (1, rows, 4096), torch.bfloat16, gpu, seed=rows)
        W, _ = wk.queries_and_gains(wk.generator(rows + 1, gpu), 24, 4096, gpu)
        a = api.block_phase1(blocks, W, None, 1e-8)
        b = api.block_phase1(blocks, W, torch.ones_like(W), 1e-8)
        assert torch.equal(a[0], b[0]) and torch.equal(a[2], b[2]), f"phase 1, {rows} rows"
    for rows in (45, 700):
        g = wk.generator(rows + 2, gpu)
        (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, 4096), 0.5, 3.0, torch.bfloat16, gpu)
        W, _ = wk.queries_and_gains(g, 1, 4096, gpu)
        u = wk.sublayer_u(g, 1, 4096, gpu)[0].contiguous()
        lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
        a = api.block_merge_update(o, lse, pin, sub, u, W[0], None, 1e-8)
        b = api.block_merge_update(o, lse, pin, sub, u, W[0], torch.ones(4096, device=gpu), 1e-8)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]), f"fused step, {rows} rows"
    srcs, q, _ = rand_sources(4, (1, 300, 2048), torch.bfloat16, gpu, seed=77)
    dh = wk.upstream_grad(wk.generator(78, gpu), (1, 300, 2048), torch.bfloat16, gpu)
    ga, qa, gga = api.depth_aggregate_backward(srcs, q, None, 1e-8, dh)
    gb, qb, ggb = api.depth_aggregate_backward(srcs, q, torch.ones(2048, device=gpu), 1e-8, dh)
    assert all(torch.equal(x, y) for x, y in zip(ga, gb)) and torch.equal(qa, qb) and torch.equal(gga, ggb)


def test_stream_order_with_dependent_launches(gpu):
    """The library's kernels start as programmatic dependents of the kernel before them on the stream and
    wait for it before touching memory: a query or a source rewritten by a torch kernel right before the call
    is what the call reads.  Ten rewrite-then-call rounds queued back to back, on the pipelined aggregation and
    on the fused step, against the same calls made after a full synchronisation."""
    srcs, q, g = rand_sources(6, (1, 2000, 2048), torch.bfloat16, gpu, seed=31)
    qs = [q * (1.0 + 0.5 * k) for k in range(10)]
    outs, qbuf = [], torch.empty_like(q)
    for k in range(10):
        qbuf.copy_(qs[k])                                  # a torch kernel, then the library's on the same stream
        srcs[0].mul_(-1.0)
        outs.append(api.depth_aggregate(srcs, qbuf, g, 1e-8).clone())
    torch.cuda.synchronize()                               # ten sign flips: srcs[0] is back to its start
    for k in range(10):
        srcs[0].mul_(-1.0)
        torch.cuda.synchronize()
        want = api.depth_aggregate(srcs, qs[k], g, 1e-8)
        torch.cuda.synchronize()
        assert torch.equal(outs[k], want), f"aggregation round {k}"
    gen = wk.generator(32, gpu)
    (o, pin, sub), _ = wk.scaled_normal_sources(gen, 3, (1, 3000, 4096), 0.5, 3.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(gen, 1, 4096, gpu)
    u = wk.sublayer_u(gen, 1, 4096, gpu)[0].contiguous()
    lse = torch.empty(3000, device=gpu).normal_(0.0, 2.0, generator=gen)
    res, wbuf = [], torch.empty_like(W[0])
    for k in range(10):
        wbuf.copy_(W[0] * (1.0 + 0.25 * k))
        res.append(api.block_merge_update(o, lse, pin, sub, u, wbuf, G[0], 1e-8)[1].clone())
    torch.cuda.synchronize()
    for k in range(10):
        want = api.block_merge_update(o, lse, pin, sub, u, (W[0] * (1.0 + 0.25 * k)).contiguous(), G[0], 1e-8)[1]
        torch.cuda.synchronize()
        assert torch.equal(res[k], want), f"fused step round {k}"


def pick(t, rows, D):
    """Rows (numpy indices) of a [.., D] CUDA tensor viewed as [rows, D]."""
    return t.reshape(-1, D)[torch.as_tensor(rows, device=t.device)]


def sample_rows(B, T, k, seed):
    rng = np.random.default_rng(seed)
    rows = {0, B * T - 1}
    for b in range(B):
        rows |= {b * T, b * T + T - 1}
    rows |= set(rng.integers(0, B * T, size=k).tolist())
    return np.array(sorted(rows))


def test_aggregate_block_single_full_size_sampled(gpu):
    wl = wk.WORKLOADS["block_single_bf16"]
    inp = wk.single_aggregation_inputs(wl, device=gpu)
    out, m, lse = api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"], stats=True)
    rows = sample_rows(wl.B, wl.T, 48, 2)
    V = np.stack([f64(pick(s, rows, wl.D)) for s in inp["sources"]])
    h, om, olse = oracle.depth_aggregate(V, f64(inp["query"]), f64(inp["gain"]), inp["eps"])
    check(pick(out, rows, wl.D), h, TOL[torch.bfloat16] * vmax(inp["sources"]), "cfg2")
    check_stats(lse.reshape(-1)[torch.as_tensor(rows, device=gpu)], olse, "lse")


# Shapes that reach the aggregation's instantiations with the CTA width
# built in and the many-rows shape (from 32 rows per SM on a 152-SM GPU,
# 4864 rows): rows that exactly fill 64, 128, 224 or 256 threads, and a
# ragged width for contrast; rows compared on a sample (rows are independent).
@pytest.mark.parametrize("dtype,D,n,rows", [
    (torch.bfloat16, 4096, 5, 4900), (torch.bfloat16, 1024, 7, 5000), (torch.bfloat16, 8192, 3, 4870),
    (torch.float32, 2048, 4, 4900), (torch.bfloat16, 1024, 3, 2000), (torch.bfloat16, 2056, 6, 4900),
    (torch.bfloat16, 7168, 10, 4900), (torch.float32, 3584, 3, 4871),
])
def test_aggregate_exact_widths_sampled(gpu, dtype, D, n, rows):
    srcs, q, g = rand_sources(n, (1, rows, D), dtype, gpu, seed=D + 3 * n + rows)
    out, m, lse = api.depth_aggregate(srcs, q, g, 1e-8, stats=True)
    sample = sample_rows(1, rows, 40, D + rows)
    V = np.stack([f64(pick(s, sample, D)) for s in srcs])
    h, om, olse = oracle.depth_aggregate(V, f64(q), f64(g), 1e-8)
    check(pick(out, sample, D), oracle.round_to(h, ODT[dtype]), TOL[dtype] * vmax(srcs), f"D={D} rows={rows}")
    check_stats(lse.reshape(-1)[torch.as_tensor(sample, device=gpu)], olse, "lse")


# --------------------------------------------------------------------------
# Backward of the depth aggregation
# --------------------------------------------------------------------------
# Gradient bounds, against the gradient's own scale (the inputs are the same
# bytes on both sides; only fp32 against fp64 arithmetic differs):
# - source gradients: fp32 2e-5 * max|g| (dots over D <= 8192 terms, typical
#   error sqrt(D) * 2^-24 ~ 5e-6, times 4); bf16 8e-3 * max|g| (one rounding
#   of the stored gradient, as the forward outputs);
# - query / gain gradients: 2e-4 * max|g| (fp32 partial sums over up to
#   1e5 row-source terms, then over the partial rows).
GRAD_TOL = {torch.float32: 2e-5, torch.bfloat16: 8e-3}
GRAD_SUM_TOL = 2e-4


def _bwd_case(gpu, dtype, D, n, rows, seed, accumulate=False):
    g = wk.generator(seed, gpu)
    srcs, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, dtype, gpu)
    W, G = wk.queries_and_gains(g, 1, D, gpu)
    dh = wk.upstream_grad(g, (1, rows, D), dtype, gpu)
    prior = [wk.upstream_grad(g, (1, rows, D), dtype, gpu) for _ in range(n)] if accumulate else None
    gs = [p.clone() for p in prior] if accumulate else None
    gs, gq, gg = api.depth_aggregate_backward(srcs, W[0], G[0], 1e-8, dh, grad_sources=gs, accumulate=accumulate)
    dV, dw, dg = oracle.depth_aggregate_backward([f64(s).reshape(rows, D) for s in srcs], f64(W[0]), f64(G[0]),
                                                 1e-8, f64(dh).reshape(rows, D))
    if accumulate:
        dV = np.stack([oracle.round_to(f64(p).reshape(rows, D) + dV[i], ODT[dtype]) for i, p in enumerate(prior)])
    else:
        dV = oracle.round_to(dV, ODT[dtype])
    check(torch.stack(gs).reshape(n, rows, D), dV, GRAD_TOL[dtype] * np.abs(dV).max(), "grad sources")
    check(gq, dw, GRAD_SUM_TOL * np.abs(dw).max(), "grad query")
    check(gg, dg, GRAD_SUM_TOL * np.abs(dg).max(), "grad gain")
    return srcs, W, G, dh, gs, gq, gg


def test_aggregate_backward_random_shapes(gpu):
    """Seeded random backward shapes against the oracle: bf16 and fp32, widths from 4 to 8192 elements,
    1..24 sources, 1..2000 rows, overwriting or accumulating the source gradients."""
    def draw(rng):
        dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
        step, top = (8, 8192) if dtype == torch.bfloat16 else (4, 4096)
        D = int(rng.integers(1, top // step + 1)) * step
        n = int(rng.integers(1, 25))
        rows = max(1, min(int(rng.integers(1, 2001)), 3_000_000 // (n * D)))
        return dtype, D, n, rows, bool(rng.random() < 0.3)
    for i, (dtype, D, n, rows, acc) in enumerate(_random_shapes(2028, 16, draw)):
        _bwd_case(gpu, dtype, D, n, rows, seed=600 + i, accumulate=acc)


@pytest.mark.parametrize("dtype,D,n,rows", [
    (torch.bfloat16, 16, 3, 33), (torch.float32, 64, 5, 20), (torch.bfloat16, 512, 7, 45),
    (torch.float32, 256, 2, 70), (torch.bfloat16, 2048, 10, 37), (torch.bfloat16, 8192, 4, 9),
    (torch.float32, 4096, 17, 13), (torch.bfloat16, 1024, 256, 3), (torch.bfloat16, 4096, 9, 130),
])
def test_aggregate_backward_small(gpu, dtype, D, n, rows):
    _bwd_case(gpu, dtype, D, n, rows, D + n + rows)


def test_aggregate_backward_accumulate_and_special_cases(gpu):
    _bwd_case(gpu, torch.bfloat16, 2048, 6, 21, 5, accumulate=True)
    _bwd_case(gpu, torch.float32, 64, 3, 50, 6, accumulate=True)
    # one source: alpha = 1 and ds = 0 exactly -> the gradient is dh, bitwise; no query gradient
    g = wk.generator(7, gpu)
    (v,), _ = wk.scaled_normal_sources(g, 1, (2, 9, 1024), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, 1, 1024, gpu)
    dh = wk.upstream_grad(g, (2, 9, 1024), torch.bfloat16, gpu)
    (gv,), gq, gg = api.depth_aggregate_backward([v], W[0], G[0], 1e-8, dh)
    assert torch.equal(gv, dh) and not torch.any(gq) and not torch.any(gg)
    # empty: the parameter gradients are zero
    e = torch.empty((0, 5, 1024), dtype=torch.bfloat16, device=gpu)
    _, gq, gg = api.depth_aggregate_backward([e, e], W[0], G[0], 1e-8, e, grad_sources=[e.clone(), e.clone()])
    assert not torch.any(gq) and not torch.any(gg)


def test_aggregate_backward_full_size_sampled(gpu):
    wl = wk.WORKLOADS["block_single_bf16"]               # 10 x [4, 4096, 2048] bf16
    inp = wk.single_aggregation_inputs(wl, device=gpu)
    dh = wk.upstream_grad(wk.generator(4242, gpu), (wl.B, wl.T, wl.D), wl.dtype, gpu)
    gs, gq, gg = api.depth_aggregate_backward(inp["sources"], inp["query"], inp["gain"], inp["eps"], dh)
    rows = sample_rows(wl.B, wl.T, 24, 7)
    dV, _, _ = oracle.depth_aggregate_backward([f64(pick(s, rows, wl.D)) for s in inp["sources"]],
                                               f64(inp["query"]), f64(inp["gain"]), inp["eps"],
                                               f64(pick(dh, rows, wl.D)))
    got = torch.stack([pick(x, rows, wl.D) for x in gs])
    dV = oracle.round_to(dV, oracle.BF16)
    check(got, dV, GRAD_TOL[torch.bfloat16] * np.abs(dV).max(), "cfg2 grad sources")
    # the query gradient sums over every row: the sum over two halves must agree,
    # and a second call gives the same bits (fixed reduction order)
    half = wl.B // 2
    parts = [api.depth_aggregate_backward([s[sl] for s in inp["sources"]], inp["query"], inp["gain"], inp["eps"],
                                          dh[sl])[1] for sl in (slice(0, half), slice(half, wl.B))]
    check(gq, f64(parts[0] + parts[1]), GRAD_SUM_TOL * float(gq.abs().max()), "cfg2 grad query split")
    _, gq2, gg2 = api.depth_aggregate_backward(inp["sources"], inp["query"], inp["gain"], inp["eps"], dh)
    assert torch.equal(gq, gq2) and torch.equal(gg, gg2)


# --------------------------------------------------------------------------
# two-phase Block: phase 1, phase 2 merge, partial update, one block chain
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,D,n,S,rows", [
    # tensor-core path (bf16, D a multiple of 64, n <= 10, S <= 24, at least 512 rows): one / several / ragged
    # 128-row tiles; rows wider than 4096 formed in two pieces
    (torch.bfloat16, 512, 9, 24, 600), (torch.bfloat16, 1024, 5, 7, 520), (torch.bfloat16, 2048, 9, 24, 700),
    (torch.bfloat16, 4096, 9, 24, 520), (torch.bfloat16, 4096, 2, 3, 1000), (torch.bfloat16, 4096, 8, 24, 4103),
    (torch.bfloat16, 7168, 9, 24, 530), (torch.bfloat16, 8192, 5, 7, 515), (torch.bfloat16, 5120, 9, 24, 600),
    # the per-row kernel: few rows, fp32, n > 10
    (torch.bfloat16, 512, 1, 1, 1), (torch.bfloat16, 512, 9, 24, 37), (torch.bfloat16, 512, 3, 5, 130),
    (torch.bfloat16, 4096, 9, 24, 8), (torch.bfloat16, 7168, 9, 4, 9), (torch.float32, 256, 5, 7, 66),
    (torch.bfloat16, 64, 1, 3, 20), (torch.bfloat16, 2048, 16, 2, 11), (torch.bfloat16, 4096, 10, 24, 21),
    (torch.float32, 2048, 5, 7, 1600), (torch.bfloat16, 2048, 16, 2, 900),
    # S = 2 on the tensor-core path: the scores kernel with the softmax in its epilogue (ten
    # summaries, one CTA per SM) writes alpha itself; and rows in two pieces with ten summaries
    (torch.bfloat16, 4096, 9, 2, 600), (torch.bfloat16, 7168, 10, 2, 530), (torch.bfloat16, 1024, 10, 2, 1300),
    # the largest S one call takes (the per-row kernel), bf16 and fp32
    (torch.bfloat16, 1024, 5, 64, 40), (torch.float32, 512, 3, 64, 19), (torch.bfloat16, 4096, 9, 64, 7),
    # few rows (64..511) on the tensor cores with the scores split over feature slices: the decode
    # shape, one partly filled tile, an odd S (pad query), ten summaries at S = 3
    (torch.bfloat16, 7168, 9, 24, 256), (torch.bfloat16, 4096, 9, 24, 100), (torch.bfloat16, 2048, 5, 7, 300),
    (torch.bfloat16, 1024, 10, 3, 64),
    # the widest rows: nine summaries at D = 8192 fill kernel B's shared memory (two pieces of 4096); ten
    # do not fit it, and those rows take the per-row kernel
    (torch.bfloat16, 8192, 9, 24, 520), (torch.bfloat16, 8192, 10, 24, 512),
    # the most summaries a call takes, sixteen (more than ten take the per-row kernel), at S = 16
    (torch.bfloat16, 2048, 16, 16, 160),
])
def test_phase1_small(gpu, dtype, D, n, S, rows):
    g = wk.generator(D + n + S, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, dtype, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    o, m, lse = api.block_phase1(blocks, W, G, 1e-8, want_max=True)
    O, M, LSE = oracle.block_phase1([f64(b) for b in blocks], f64(W), f64(G), 1e-8)
    tol = TOL[dtype] * vmax(blocks)
    check(o.reshape(S, -1, D), oracle.round_to(O, ODT[dtype]), tol, "phase1 o")
    stol = STATS_TOL_SPLIT_Q if dtype == torch.bfloat16 else STATS_TOL
    check_stats(lse.reshape(S, -1), LSE, "phase1 lse", stol)
    check_stats(m.reshape(S, -1), M, "phase1 m", stol)


def test_phase1_two_phase_config_full_size_sampled(gpu):
    wl = wk.WORKLOADS["two_phase_bf16"]
    inp = wk.two_phase_inputs(wl, device=gpu)
    o, _, lse = api.block_phase1(inp["blocks"], inp["queries"], inp["gains"], inp["eps"])
    rows = sample_rows(wl.B, wl.T, 24, 3)
    O, _, LSE = oracle.block_phase1([f64(pick(b, rows, wl.D)) for b in inp["blocks"]],
                                    f64(inp["queries"]), f64(inp["gains"]), inp["eps"])
    ix = torch.as_tensor(rows, device=gpu)
    check(o.reshape(wl.S, -1, wl.D)[:, ix], O, TOL[torch.bfloat16] * vmax(inp["blocks"]), "cfg3 p1")
    check_stats(lse.reshape(wl.S, -1)[:, ix], LSE, "cfg3 lse", STATS_TOL_SPLIT_Q)


def test_phase2_merge_small(gpu):
    for dtype, D, rows in ((torch.bfloat16, 4096, 45), (torch.float32, 256, 70), (torch.bfloat16, 16, 33)):
        g = wk.generator(D + rows, gpu)
        (o, p), _ = wk.scaled_normal_sources(g, 2, (1, rows, D), 0.5, 8.0, dtype, gpu)
        W, G = wk.queries_and_gains(g, 1, D, gpu)
        lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
        lse_out = torch.empty_like(lse)
        h = api.block_phase2_merge(o, lse, p, W[0], G[0], 1e-8, out_lse=lse_out)
        want, wl = oracle.block_phase2_merge(f64(o).reshape(rows, D), f64(lse), f64(p).reshape(rows, D),
                                             f64(W[0]), f64(G[0]), 1e-8)
        check(h.reshape(rows, D), oracle.round_to(want, ODT[dtype]), TOL[dtype] * vmax([o, p]), "merge")
        check_stats(lse_out, wl, "merged lse")
        h0 = api.block_phase2_merge(o, lse, None, W[0], G[0], 1e-8, out_lse=lse_out)
        assert torch.equal(h0, o) and torch.equal(lse_out, lse)


def test_partial_update(gpu):
    for dtype, D, rows in ((torch.bfloat16, 4096, 21), (torch.float32, 12, 7)):
        g = wk.generator(D, gpu)
        (h, p), _ = wk.scaled_normal_sources(g, 2, (1, rows, D), 0.5, 3.0, dtype, gpu)
        u = wk.sublayer_u(g, 1, D, gpu)[0].contiguous()
        f = oracle.synthetic_sublayer(f64(u), f64(h).reshape(rows, D))
        first = api.partial_update(h, None, u)
        check(first.reshape(rows, D), oracle.round_to(f, ODT[dtype]), TOL[dtype] * 0.5, "update first")
        want = oracle.round_to(f64(p).reshape(rows, D) + f, ODT[dtype])
        pin = p.clone()
        api.partial_update(h, pin, u, out=pin)                  # in place
        check(pin.reshape(rows, D), want, TOL[dtype] * vmax([p]), "update in place")


def test_synthetic_sublayer_nonlinearity_error_bound(gpu):
    # 0.5 tanh(z) is formed as 0.5 - 1 / (e^{2z} + 1) with fast exp / reciprocal: its absolute
    # error must stay near fp32 rounding over the whole range, tails and tiny arguments included.
    z = np.concatenate([np.linspace(-60.0, 60.0, 120000), np.linspace(-1e-3, 1e-3, 4001),
                        np.array([0.0, 1e-30, -1e-30, 88.0, -88.0, 200.0, -200.0])])
    D = 256
    R = (z.size + D - 1) // D
    zz = np.zeros(R * D)
    zz[: z.size] = z
    h = torch.tensor(zz, dtype=torch.float32, device=gpu).reshape(1, R, D)
    u = torch.ones(D, dtype=torch.float32, device=gpu)
    y = api.partial_update(h, None, u)                       # first sublayer: p = f(h) exactly once
    want = 0.5 * np.tanh(f64(h).reshape(-1))
    err = np.abs(f64(y).reshape(-1) - want).max()
    assert err <= 3e-7, err


def test_merge_update_fused_step(gpu):
    # Up to 4 rows per SM, rows of 65..1024 16-byte vectors take the few-rows kernel, two rows a
    # CTA (4096 bf16, 2048 fp32, 7168 bf16, and 1032 bf16 = 129 vectors, not a multiple of a
    # warp; odd row counts leave the last CTA one row); rows of at most 64 vectors the team kernel
    for dtype, D, rows in ((torch.bfloat16, 4096, 45), (torch.float32, 256, 70), (torch.bfloat16, 16, 33),
                           (torch.float32, 2048, 37), (torch.bfloat16, 1032, 300), (torch.bfloat16, 7168, 5)):
        for synth, with_pin in ((True, True), (True, False), (False, True)):
            g = wk.generator(D + rows + 3 * synth + with_pin, gpu)
            (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, D), 0.5, 3.0, dtype, gpu)
            W, G = wk.queries_and_gains(g, 1, D, gpu)
            u = wk.sublayer_u(g, 1, D, gpu)[0].contiguous() if synth else None
            lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
            p_in = pin if with_pin else None
            lse_out = torch.full((rows,), float("nan"), device=gpu)
            p_out, h, _ = api.block_merge_update(o, lse, p_in, sub, u, W[0], G[0], 1e-8, out_lse=lse_out)
            subn = f64(sub).reshape(rows, D)
            out = oracle.synthetic_sublayer(f64(u), subn) if synth else subn
            want_p = oracle.round_to((f64(pin).reshape(rows, D) if with_pin else 0.0) + out, ODT[dtype])
            want_h, _ = oracle.block_phase2_merge(f64(o).reshape(rows, D), f64(lse), want_p, f64(W[0]),
                                                  f64(G[0]), 1e-8)
            tol = TOL[dtype] * vmax([o, pin, sub])
            check(p_out.reshape(rows, D), want_p, tol, "fused p")
            check(h.reshape(rows, D), oracle.round_to(want_h, ODT[dtype]), tol, "fused h")
            # the merged lse, from the partial as stored: the fast tanh may round a few elements of p to
            # the neighbouring value (within p's tolerance above), which moves s_p with them
            _, want_lse = oracle.block_phase2_merge(f64(o).reshape(rows, D), f64(lse), f64(p_out).reshape(rows, D),
                                                    f64(W[0]), f64(G[0]), 1e-8)
            check_stats(lse_out, want_lse, "fused merged lse")
            if with_pin:                                       # in place: p_out aliases p_in,
                pi, hs = pin.clone(), sub.clone()              # h_out aliases sub_out
                api.block_merge_update(o, lse, pi, hs, u, W[0], G[0], 1e-8, partial_out=pi, h_out=hs)
                assert torch.equal(pi, p_out) and torch.equal(hs, h)


def test_merge_update_random_shapes(gpu):
    """Seeded random fused update+merge steps against the oracle: bf16 and fp32, widths from 4 to 8192
    elements, 1..3000 rows (the team, few-rows and general kernels), with and without the sublayer and the
    incoming partial."""
    def draw(rng):
        dtype = torch.bfloat16 if rng.random() < 0.7 else torch.float32
        step, top = (8, 8192) if dtype == torch.bfloat16 else (4, 4096)
        D = int(rng.integers(1, top // step + 1)) * step
        rows = max(1, min(int(rng.integers(1, 3001)), 6_000_000 // D))
        return dtype, D, rows, bool(rng.random() < 0.7), bool(rng.random() < 0.8)
    for i, (dtype, D, rows, synth, with_pin) in enumerate(_random_shapes(2027, 24, draw)):
        g = wk.generator(500 + i, gpu)
        (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, D), 0.5, 3.0, dtype, gpu)
        W, G = wk.queries_and_gains(g, 1, D, gpu)
        u = wk.sublayer_u(g, 1, D, gpu)[0].contiguous() if synth else None
        lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
        p_out, h, _ = api.block_merge_update(o, lse, pin if with_pin else None, sub, u, W[0], G[0], 1e-8)
        subn = f64(sub).reshape(rows, D)
        out = oracle.synthetic_sublayer(f64(u), subn) if synth else subn
        want_p = oracle.round_to((f64(pin).reshape(rows, D) if with_pin else 0.0) + out, ODT[dtype])
        want_h, _ = oracle.block_phase2_merge(f64(o).reshape(rows, D), f64(lse), want_p, f64(W[0]), f64(G[0]), 1e-8)
        tol = TOL[dtype] * vmax([o, pin, sub])
        what = f"case {i}: {dtype} D={D} rows={rows} synth={synth} p_in={with_pin}"
        check(p_out.reshape(rows, D), want_p, tol, what + " p")
        check(h.reshape(rows, D), oracle.round_to(want_h, ODT[dtype]), tol, what + " h")


# The next sublayer's pre-norm, standalone and fused into the update+merge.
# Its output is a normalised row (values of order |w_n|), so the bound is
# the dtype tolerance times the largest |y| rather than the sources' scale.
def test_rms_norm(gpu):
    for dtype, D, rows in ((torch.bfloat16, 4096, 45), (torch.float32, 256, 70), (torch.bfloat16, 16, 33),
                           (torch.bfloat16, 16384, 5), (torch.float32, 8192, 3), (torch.bfloat16, 7168, 9)):
        g = wk.generator(D + rows + 5, gpu)
        (x,), _ = wk.scaled_normal_sources(g, 1, (1, rows, D), 0.5, 8.0, dtype, gpu)
        _, Wn = wk.queries_and_gains(g, 1, D, gpu)
        y = api.rms_norm(x, Wn[0], 1e-6)
        want = oracle.rms_norm(f64(x).reshape(rows, D), f64(Wn[0]), 1e-6)
        check(y.reshape(rows, D), oracle.round_to(want, ODT[dtype]), TOL[dtype] * np.abs(want).max(), "rms_norm")
        xi = x.clone()
        api.rms_norm(xi, Wn[0], 1e-6, out=xi)                  # in place
        assert torch.equal(xi, y)


def test_merge_update_with_prenorm(gpu):
    for dtype, D, rows in ((torch.bfloat16, 4096, 45), (torch.float32, 256, 70), (torch.bfloat16, 16, 33),
                           (torch.bfloat16, 16384, 6), (torch.bfloat16, 7168, 11), (torch.float32, 2048, 37)):
        for synth, with_pin in ((True, True), (True, False), (False, True)):
            g = wk.generator(D + rows + 3 * synth + with_pin + 11, gpu)
            (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, D), 0.5, 3.0, dtype, gpu)
            W, G = wk.queries_and_gains(g, 1, D, gpu)
            _, Wn = wk.queries_and_gains(g, 1, D, gpu)
            u = wk.sublayer_u(g, 1, D, gpu)[0].contiguous() if synth else None
            lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
            p_in = pin if with_pin else None
            p_out, h, y = api.block_merge_update(o, lse, p_in, sub, u, W[0], G[0], 1e-8,
                                                 norm_weight=Wn[0], norm_eps=1e-5)
            subn = f64(sub).reshape(rows, D)
            out = oracle.synthetic_sublayer(f64(u), subn) if synth else subn
            want_p = oracle.round_to((f64(pin).reshape(rows, D) if with_pin else 0.0) + out, ODT[dtype])
            want_h, _ = oracle.block_phase2_merge(f64(o).reshape(rows, D), f64(lse), want_p, f64(W[0]),
                                                  f64(G[0]), 1e-8)
            want_y = oracle.rms_norm(want_h, f64(Wn[0]), 1e-5)      # from the unrounded h
            tol = TOL[dtype] * vmax([o, pin, sub])
            check(p_out.reshape(rows, D), want_p, tol, "prenorm p")
            check(h.reshape(rows, D), oracle.round_to(want_h, ODT[dtype]), tol, "prenorm h")
            check(y.reshape(rows, D), oracle.round_to(want_y, ODT[dtype]), TOL[dtype] * np.abs(want_y).max(),
                  "prenorm y")
            # h not stored; y written over the sublayer row it was computed from
            pi, ys = (pin.clone() if with_pin else torch.empty_like(pin)), sub.clone()
            api.block_merge_update(o, lse, pi if with_pin else None, ys, u, W[0], G[0], 1e-8, partial_out=pi,
                                   norm_weight=Wn[0], norm_eps=1e-5, normed_out=ys, write_h=False)
            assert torch.equal(pi, p_out) and torch.equal(ys, y)


@pytest.mark.parametrize("D,rows", [(4096, 700), (7168, 650), (8192, 620)])
def test_merge_update_many_rows_sampled(gpu, D, rows):
    """Past 4 rows per SM the fused step takes four vectors per thread; these
    widths fill 128, 224 and 256 threads exactly, the instantiations with the
    CTA width built in (with and without the pre-norm).  Sampled rows."""
    dtype = torch.bfloat16
    sample = sample_rows(1, rows, 24, D)
    for norm in (True, False):
        g = wk.generator(D + rows + 7 * norm, gpu)
        (o, pin, sub), _ = wk.scaled_normal_sources(g, 3, (1, rows, D), 0.5, 3.0, dtype, gpu)
        W, G = wk.queries_and_gains(g, 1, D, gpu)
        _, Wn = wk.queries_and_gains(g, 1, D, gpu)
        u = wk.sublayer_u(g, 1, D, gpu)[0].contiguous()
        lse = torch.empty(rows, device=gpu).normal_(0.0, 2.0, generator=g)
        kw = dict(norm_weight=Wn[0], norm_eps=1e-5) if norm else {}
        lse_out = torch.full((rows,), float("nan"), device=gpu)
        res = api.block_merge_update(o, lse, pin, sub, u, W[0], G[0], 1e-8, out_lse=lse_out, **kw)
        p_out, h = res[0], res[1]
        idx = torch.as_tensor(sample, device=gpu)
        subn = f64(pick(sub, sample, D))
        want_p = oracle.round_to(f64(pick(pin, sample, D)) + oracle.synthetic_sublayer(f64(u), subn), ODT[dtype])
        want_h, _ = oracle.block_phase2_merge(f64(pick(o, sample, D)), f64(lse[idx]), want_p, f64(W[0]),
                                              f64(G[0]), 1e-8)
        tol = TOL[dtype] * vmax([o, pin, sub])
        check(pick(p_out, sample, D), want_p, tol, f"p D={D} norm={norm}")
        check(pick(h, sample, D), oracle.round_to(want_h, ODT[dtype]), tol, f"h D={D} norm={norm}")
        _, want_lse = oracle.block_phase2_merge(f64(pick(o, sample, D)), f64(lse[idx]), f64(pick(p_out, sample, D)),
                                                f64(W[0]), f64(G[0]), 1e-8)   # from the partial as stored
        check_stats(lse_out[idx], want_lse, f"merged lse D={D} norm={norm}")
        if norm:
            want_y = oracle.rms_norm(want_h, f64(Wn[0]), 1e-5)
            check(pick(res[2], sample, D), oracle.round_to(want_y, ODT[dtype]),
                  TOL[dtype] * np.abs(want_y).max(), f"y D={D}")


@pytest.mark.parametrize("fused", [True, False])
def test_two_phase_block_chain_with_prenorm(gpu, fused):
    D, n, S, rows = 2048, 9, 6, 40
    g = wk.generator(78, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    U = wk.sublayer_u(g, S, D, gpu)
    _, NW = wk.queries_and_gains(g, S, D, gpu)
    p, Y = api.block_two_phase(blocks, W, G, U, 1e-8, fused=fused, norm_weights=NW, norm_eps=1e-6)
    OY, OP = oracle.block_two_phase_chain([f64(b) for b in blocks], f64(W), f64(G), f64(U), 1e-8,
                                          oracle.BF16, NW=f64(NW), norm_eps=1e-6)
    # fused: y_k from the unrounded h_k (as the oracle); unfused: from the stored h_k,
    # one bf16 rounding apart, inside the same bound
    check(Y.reshape(S, rows, D), OY, TOL[torch.bfloat16] * np.abs(OY).max(), "chain y")
    check(p.reshape(rows, D), OP, TOL[torch.bfloat16] * vmax(blocks), "chain p")
    check_chain(Y.reshape(S, rows, D), OY, "chain y")
    check_chain(p.reshape(rows, D), OP, "chain p")


@pytest.mark.parametrize("fused", [True, False])
def test_two_phase_block_chain_small(gpu, fused):
    D, n, S, rows = 1024, 9, 6, 50
    g = wk.generator(77, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    U = wk.sublayer_u(g, S, D, gpu)
    p, H = api.block_two_phase(blocks, W, G, U, 1e-8, fused=fused)
    OH, OP = oracle.block_two_phase_chain([f64(b) for b in blocks], f64(W), f64(G), f64(U), 1e-8,
                                          oracle.BF16)
    tol = TOL[torch.bfloat16] * vmax(blocks)
    check(H.reshape(S, rows, D), OH, tol, "chain h")
    check(p.reshape(rows, D), OP, tol, "chain p")
    check_chain(H.reshape(S, rows, D), OH, "chain h")
    check_chain(p.reshape(rows, D), OP, "chain p")


@pytest.mark.parametrize("fused,prenorm", [(False, False), (True, True)])
def test_two_phase_block_groups_other_forms(gpu, fused, prenorm):
    """groups=2 for the unfused pass and for the fused pass with the sublayer pre-norm: bitwise the
    partial of one pass over the whole batch (9728 rows a group, as below)."""
    D, n, S, B, T = 512, 9, 6, 4, 4864
    g = wk.generator(81, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (B, T, D), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    U = wk.sublayer_u(g, S, D, gpu)
    NW = wk.queries_and_gains(g, S, D, gpu)[1] if prenorm else None
    p1 = api.TwoPhaseBlock(blocks, W, G, U, 1e-8, fused=fused, norm_weights=NW).run().clone()
    p2 = api.TwoPhaseBlock(blocks, W, G, U, 1e-8, fused=fused, norm_weights=NW, groups=2).run().clone()
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)


def test_two_phase_block_groups_of_sequences(gpu):
    """groups=2: the batch's sequences in two groups on two streams give bitwise the partial of one pass over
    the whole batch, eagerly and as one CUDA graph, and match the oracle.  9728 rows a group take the same
    kernels as one pass: below 76 tiles of 128 rows phase 1 splits its scores over feature slices, and below
    four rows per SM the update+merge takes its few-rows kernel, each with a reduction order of its own."""
    D, n, S, B, T = 512, 9, 6, 4, 4864
    g = wk.generator(79, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (B, T, D), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    U = wk.sublayer_u(g, S, D, gpu)
    one = api.TwoPhaseBlock(blocks, W, G, U, 1e-8)
    p1 = one.run().clone()
    two = api.TwoPhaseBlock(blocks, W, G, U, 1e-8, groups=2)
    p2 = two.run().clone()
    torch.cuda.synchronize()
    assert torch.equal(p1, p2)
    two.capture()
    two.partial.zero_()
    assert torch.equal(two.replay(), p1)
    torch.cuda.synchronize()
    _, OP = oracle.block_two_phase_chain([f64(b).reshape(B * T, D) for b in blocks], f64(W), f64(G), f64(U),
                                         1e-8, oracle.BF16)
    check(p2.reshape(B * T, D), OP, TOL[torch.bfloat16] * vmax(blocks), "groups=2 p")
    with pytest.raises(ValueError):
        api.TwoPhaseBlock(blocks, W, G, U, 1e-8, groups=3)
    with pytest.raises(ValueError):                       # the partial must match the summaries
        api.TwoPhaseBlock(blocks, W, G, U, 1e-8, partial=torch.empty(1, device=gpu))


@pytest.mark.parametrize("fused", [True, False])
def test_two_phase_block_chain_full_size_sampled(gpu, fused):
    wl = wk.WORKLOADS["two_phase_bf16"]
    inp = wk.two_phase_inputs(wl, device=gpu)
    blk = api.TwoPhaseBlock(inp["blocks"], inp["queries"], inp["gains"], inp["u"], inp["eps"], fused=fused)
    p = blk.run()
    torch.cuda.synchronize()
    rows = sample_rows(wl.B, wl.T, 16, 4)
    _, OP = oracle.block_two_phase_chain([f64(pick(b, rows, wl.D)) for b in inp["blocks"]],
                                         f64(inp["queries"]), f64(inp["gains"]), f64(inp["u"]),
                                         inp["eps"], oracle.BF16)
    check(pick(p, rows, wl.D), OP, TOL[torch.bfloat16] * vmax(inp["blocks"]), "cfg3 chain")
    check_chain(pick(p, rows, wl.D), OP, "cfg3 chain")


@pytest.mark.parametrize("name", ["long_prefill_bf16", "decode_bf16"])
def test_d7168_configs_sampled(gpu, name):
    wl = wk.WORKLOADS[name]
    inp = wk.single_aggregation_inputs(wl, device=gpu)
    out = api.depth_aggregate(inp["sources"], inp["query"], inp["gain"], inp["eps"])
    rows = sample_rows(wl.B, wl.T, 12, 5)
    V = np.stack([f64(pick(s, rows, wl.D)) for s in inp["sources"]])
    h, _, _ = oracle.depth_aggregate(V, f64(inp["query"]), f64(inp["gain"]), inp["eps"])
    check(pick(out, rows, wl.D), h, TOL[torch.bfloat16] * vmax(inp["sources"]), name)
    del out, inp
    tp = wk.two_phase_inputs(wl, device=gpu)           # 9 summaries + S = 24 chain
    blk = api.TwoPhaseBlock(tp["blocks"], tp["queries"], tp["gains"], tp["u"], tp["eps"])
    p = blk.run()
    torch.cuda.synchronize()
    _, OP = oracle.block_two_phase_chain([f64(pick(b, rows, wl.D)) for b in tp["blocks"]],
                                         f64(tp["queries"]), f64(tp["gains"]), f64(tp["u"]),
                                         tp["eps"], oracle.BF16)
    check(pick(p, rows, wl.D), OP, TOL[torch.bfloat16] * vmax(tp["blocks"]), name + " chain")
    check_chain(pick(p, rows, wl.D), OP, name + " chain")


# --------------------------------------------------------------------------
# Decode: side-stream inter-block pass, and the block pass as one CUDA graph
# --------------------------------------------------------------------------
def test_decode_overlap_and_graph(gpu):
    wl = wk.WORKLOADS["decode_bf16"]                     # [256, 1, 7168], 9 summaries, S = 24
    tp = wk.two_phase_inputs(wl, device=gpu)
    args = (tp["blocks"], tp["queries"], tp["gains"], tp["u"], tp["eps"])
    eager = api.TwoPhaseBlock(*args, keep_h=True)
    p_eager = eager.run().clone()
    ov = api.TwoPhaseBlock(*args, keep_h=True, overlap=True)
    p_ov = ov.run().clone()
    torch.cuda.synchronize()
    rows = sample_rows(wl.B, wl.T, 16, 6)
    OH, OP = oracle.block_two_phase_chain([f64(pick(b, rows, wl.D)) for b in tp["blocks"]],
                                          f64(tp["queries"]), f64(tp["gains"]), f64(tp["u"]),
                                          tp["eps"], oracle.BF16)
    tol = TOL[torch.bfloat16] * vmax(tp["blocks"])
    ix = torch.as_tensor(rows, device=gpu)
    for p, H, name in ((p_eager, eager.h, "eager"), (p_ov, ov.h, "overlap")):
        check(pick(p, rows, wl.D), OP, tol, name + " p")
        check(H.reshape(wl.S, -1, wl.D)[:, ix], OH, tol, name + " h")
        check_chain(pick(p, rows, wl.D), OP, name + " p")
        check_chain(H.reshape(wl.S, -1, wl.D)[:, ix], OH, name + " h")
    # graphs replay exactly the eager launches: bitwise equal
    for blk, want in ((eager, p_eager), (ov, p_ov)):
        blk.capture()
        got = blk.replay().clone()
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    # a replay reads the live buffers: new summaries in place, new result
    for b in tp["blocks"]:
        b.mul_(-0.5)
    p_new = eager.replay().clone()
    ref = api.TwoPhaseBlock(*args).run()
    torch.cuda.synchronize()
    assert torch.equal(p_new, ref) and not torch.equal(p_new, p_eager)


def test_two_phase_stream_pipelined_passes(gpu):
    """api.TwoPhaseStream: host inputs copied in on a copy stream, the block
    pass on the current stream, the partial copied back on a third, two
    device buffer sets in turn.  Four passes over different host inputs, all
    submitted before any is awaited: each host result equals, bitwise, a
    plain TwoPhaseBlock pass on the same inputs (a set reused too early, or a
    partial read back before its pass ended, would show)."""
    wl = wk.WORKLOADS["two_phase_bf16"]
    rows, S, n = 640, 6, 9
    passes = []
    for j in range(4):
        tp = wk.two_phase_inputs(wl, rows=rows + j, device="cpu", S=S, n=n)
        tp["blocks"] = [b[:, :rows] for b in tp["blocks"]]          # same shape every pass
        passes.append(tp)
    host = [{"blocks": [b.contiguous().pin_memory() for b in tp["blocks"]],
             "queries": tp["queries"].pin_memory(), "gains": tp["gains"].pin_memory(),
             "u": tp["u"].pin_memory()} for tp in passes]
    shape = tuple(host[0]["blocks"][0].shape)
    pipe = api.TwoPhaseStream(n, shape, torch.bfloat16, S, gpu, wk.EPS)
    outs = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in host]
    for h, out in zip(host, outs):
        done = pipe.submit(h["blocks"], h["queries"], h["gains"], h["u"], out)
    done.synchronize()
    torch.cuda.synchronize()
    for h, out in zip(host, outs):
        want = api.TwoPhaseBlock([b.to(gpu) for b in h["blocks"]], h["queries"].to(gpu), h["gains"].to(gpu),
                                 h["u"].to(gpu), wk.EPS).run().cpu()
        assert torch.equal(out, want)
    assert not torch.equal(outs[0], outs[1])


# --------------------------------------------------------------------------
# Full stack
# --------------------------------------------------------------------------
def test_full_stack_small(gpu):
    for dtype, D, L, rows in ((torch.bfloat16, 256, 12, 40), (torch.float32, 128, 7, 19)):
        wl = wk.WORKLOADS["full_stack_bf16"]
        inp = wk.full_stack_inputs(wl, rows=rows, device=gpu, L=L, D=D)
        v0 = inp["v0"].to(dtype)
        y, srcs = api.full_stack_forward(v0, inp["queries"], inp["gains"], inp["u"], inp["eps"])
        V, oy = oracle.full_stack_forward(f64(v0).reshape(rows, D), f64(inp["queries"]),
                                          f64(inp["gains"]), f64(inp["u"]), inp["eps"], ODT[dtype])
        tol = TOL[dtype] * float(v0.abs().max())
        for l in range(1, L + 1):
            check(srcs[l].reshape(rows, D), V[l], tol, f"v_{l}")
        check(y.reshape(rows, D), oracle.round_to(oy, ODT[dtype]), tol, "y")


def test_full_stack_as_one_cuda_graph(gpu):
    """api.FullStack: the plain stack and the two-phase schedule captured as one
    CUDA graph each replay bitwise the eager run, and a replay reads the live
    v_0 (changed in place after the capture)."""
    wl = wk.WORKLOADS["full_stack_bf16"]
    inp = wk.full_stack_inputs(wl, rows=300, device=gpu, L=30, D=1024)
    for S in (None, 6):
        fs = api.FullStack(inp["v0"].clone(), inp["queries"], inp["gains"], inp["u"], inp["eps"], S=S)
        want = fs.run().clone()
        fs.capture()
        got = fs.replay().clone()
        torch.cuda.synchronize()
        assert torch.equal(got, want), f"S={S}"
        fs.v0.mul_(-1.0)
        got2 = fs.replay().clone()
        ref = api.FullStack(fs.v0.clone(), inp["queries"], inp["gains"], inp["u"], inp["eps"], S=S).run()
        torch.cuda.synchronize()
        assert torch.equal(got2, ref) and not torch.equal(got2, want), f"S={S} after v0 changed"


def test_full_stack_config_full_size_sampled(gpu):
    wl = wk.WORKLOADS["full_stack_bf16"]
    inp = wk.full_stack_inputs(wl, device=gpu)
    y, srcs = api.full_stack_forward(inp["v0"], inp["queries"], inp["gains"], inp["u"], inp["eps"])
    rows = sample_rows(wl.B, wl.T, 6, 6)
    V, oy = oracle.full_stack_forward(f64(pick(inp["v0"], rows, wl.D)), f64(inp["queries"]),
                                      f64(inp["gains"]), f64(inp["u"]), inp["eps"], oracle.BF16)
    tol = TOL[torch.bfloat16] * float(inp["v0"].abs().max())
    for l in (1, 2, 50, 186):
        check(pick(srcs[l], rows, wl.D), V[l], tol, f"v_{l}")
    check(pick(y, rows, wl.D), oy, tol, "y")


# Full stack with the two-phase schedule: blocks up to ten sources take the
# block phase-1 kernels, wider ones the raw-score path (scores ten at a time,
# softmax, outputs over all sources); the oracle rounds o_l and v_l where the
# GPU stores them.
# Wide blocks with S <= 16 (and D a multiple of 256) take the tensor-core outputs kernel, wider S the packed-FMA one.
@pytest.mark.parametrize("S,D,L,rows", [(4, 1024, 23, 130), (12, 2048, 30, 70), (1, 512, 14, 64),
                                        (40, 1024, 25, 50), (24, 2048, 27, 129), (20, 1024, 45, 64),
                                        (16, 256, 40, 33),
                                        # S = 2 over 512+ rows: blocks of up to ten sources take the
                                        # tensor-core phase 1 with the softmax in the scores kernel,
                                        # wider ones the raw-score path
                                        (2, 1024, 9, 600), (2, 512, 25, 520),
                                        # the last block over 241 sources at D = 2048: three copy slots no
                                        # longer fit two CTAs per SM there, and the outputs take two
                                        (16, 2048, 250, 48)])
def test_full_two_phase_small(gpu, S, D, L, rows):
    wl = wk.WORKLOADS["full_stack_bf16"]
    inp = wk.full_stack_inputs(wl, rows=rows, device=gpu, L=L, D=D)
    y, srcs = api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"])
    V, oy = oracle.full_stack_two_phase(f64(inp["v0"]).reshape(rows, D), f64(inp["queries"]), f64(inp["gains"]),
                                        f64(inp["u"]), S, inp["eps"], oracle.BF16)
    tol = TOL[torch.bfloat16] * float(inp["v0"].abs().max())
    for l in range(1, L + 1):
        check(srcs[l].reshape(rows, D), V[l], tol, f"S={S} v_{l}")
    check(y.reshape(rows, D), oracle.round_to(oy, oracle.BF16), tol, f"S={S} y")


# bf16 rows of 2048: the intra-block steps merge into the phase-1 state with
# the two-pass kernel that holds each row in shared memory (up to seven rows
# in flight with one intra source, one from eight; 15 intra sources at S = 16),
# over several rows per CTA.
@pytest.mark.parametrize("S,L,rows", [(7, 20, 1000), (14, 29, 600), (16, 33, 500),
                                      # a grid of one and of five CTAs
                                      (7, 12, 1), (16, 32, 5)])
def test_full_two_phase_short_rows(gpu, S, L, rows):
    wl = wk.WORKLOADS["full_stack_bf16"]
    D = 2048
    inp = wk.full_stack_inputs(wl, rows=rows, device=gpu, L=L, D=D)
    y, srcs = api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"])
    V, oy = oracle.full_stack_two_phase(f64(inp["v0"]).reshape(rows, D), f64(inp["queries"]), f64(inp["gains"]),
                                        f64(inp["u"]), S, inp["eps"], oracle.BF16)
    tol = TOL[torch.bfloat16] * float(inp["v0"].abs().max())
    for l in range(1, L + 1):
        check(srcs[l].reshape(rows, D), V[l], tol, f"S={S} v_{l}")
    check(y.reshape(rows, D), oracle.round_to(oy, oracle.BF16), tol, f"S={S} y")


def test_full_two_phase_shape_limits(gpu):
    # fp32 works while every block has at most ten sources; wider blocks need bf16
    wl = wk.WORKLOADS["full_stack_bf16"]
    inp = wk.full_stack_inputs(wl, rows=20, device=gpu, L=9, D=256)
    v0 = inp["v0"].float()
    y, srcs = api.full_stack_two_phase(v0, inp["queries"], inp["gains"], inp["u"], 3, inp["eps"])
    V, oy = oracle.full_stack_two_phase(f64(v0).reshape(20, 256), f64(inp["queries"]), f64(inp["gains"]),
                                        f64(inp["u"]), 3, inp["eps"], oracle.F32)
    check(y.reshape(20, 256), oracle.round_to(oy, oracle.F32), TOL[torch.float32] * float(v0.abs().max()), "fp32 y")
    inp = wk.full_stack_inputs(wl, rows=20, device=gpu, L=25, D=256)
    with pytest.raises(_lib.AttnResError):
        api.full_stack_two_phase(inp["v0"].float(), inp["queries"], inp["gains"], inp["u"], 3, inp["eps"])


@pytest.mark.parametrize("S", [14, 16])
def test_full_two_phase_config_full_size_sampled(gpu, S):
    wl = wk.WORKLOADS["full_stack_bf16"]                 # [1, 2048, 2048], L = 186
    inp = wk.full_stack_inputs(wl, device=gpu)
    y, srcs = api.full_stack_two_phase(inp["v0"], inp["queries"], inp["gains"], inp["u"], S, inp["eps"])
    rows = sample_rows(wl.B, wl.T, 6, 8)
    V, oy = oracle.full_stack_two_phase(f64(pick(inp["v0"], rows, wl.D)), f64(inp["queries"]), f64(inp["gains"]),
                                        f64(inp["u"]), S, inp["eps"], oracle.BF16)
    tol = TOL[torch.bfloat16] * float(inp["v0"].abs().max())
    for l in (1, S, S + 1, 2 * S + 1, 100, 186):
        check(pick(srcs[l], rows, wl.D), V[l], tol, f"S={S} v_{l}")
    check(pick(y, rows, wl.D), oy, tol, f"S={S} y")


def test_no_kernel_wait_ran_out(gpu):
    """Every bounded in-kernel wait of the runs above completed in time."""
    from transformer_depth_wise_gb300 import _lib
    assert _lib.lib().attnres_take_device_error() == 0


def test_wait_that_runs_out_reports_timeout(gpu):
    """A bounded in-kernel wait that runs out, on purpose and without a fault:
    with a limit of one clock cycle the tensor-core phase 1's waits give up
    (each CTA takes several 128-row tiles, so at least its wait for the
    epilogue of an earlier tile cannot have completed).  The part of a CTA
    whose wait gave up stops, the CTA drains its copies and tensor-core
    operations in flight, and attnres_take_device_error reports
    ATTNRES_ERR_TIMEOUT.  The device stays usable: the same call with the
    default limit then matches the oracle, with no error."""
    L = _lib.lib()
    D, n, S, rows = 2048, 9, 2, 128 * 152 * 2
    g = wk.generator(99, gpu)
    blocks, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, torch.bfloat16, gpu)
    W, G = wk.queries_and_gains(g, S, D, gpu)
    assert L.attnres_take_device_error() == 0
    assert L.attnres_set_wait_limit(1) == 0
    try:
        api.block_phase1(blocks, W, G, 1e-8)
        rc = L.attnres_take_device_error()
    finally:
        assert L.attnres_set_wait_limit(0) == 0
    assert rc == -9, _lib.STATUS.get(rc, rc)                  # ATTNRES_ERR_TIMEOUT
    o, _, lse = api.block_phase1(blocks, W, G, 1e-8)
    assert L.attnres_take_device_error() == 0
    sample = sample_rows(1, rows, 24, 99)
    O, _, LSE = oracle.block_phase1([f64(pick(b, sample, D)) for b in blocks], f64(W), f64(G), 1e-8)
    ix = torch.as_tensor(sample, device=gpu)
    check(o.reshape(S, -1, D)[:, ix], O, TOL[torch.bfloat16] * vmax(blocks), "phase1 after a timeout")
    check_stats(lse.reshape(S, -1)[:, ix], LSE, "lse after a timeout", STATS_TOL_SPLIT_Q)
