"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each pin is either a result worked out by hand from the pages' equations
(exact closed forms for tiny inputs), an invariant the pages state, a
special case that reduces to a library routine, or a second, independently
written formulation.  Together they are chosen so that a plausible slip in
the oracle -- a dropped eps, sum instead of mean, scoring the raw instead
of the normalised source (or summing the normalised instead of the raw),
a lost gain, a wrong sign, a transposed operand, an off-by-one in the
block bookkeeping -- fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def agg(V, w, gamma=None, eps=0.0):
    h, m, lse = oracle.depth_aggregate(np.asarray(V, dtype=np.float64)[:, None, :], w, gamma, eps)
    return h[0], float(m[0]), float(lse[0])


# --------------------------------------------------------------------------
# Closed forms worked by hand (eq. A1-A3)
# --------------------------------------------------------------------------
def test_two_sources_closed_form():
    # v0 = (1,1): mean square 1 -> RMS(v0) = (1,1); v1 = (3,-3): mean square 9 -> RMS(v1) = (1,-1).
    # w = (a, b): s0 = a + b, s1 = a - b, alpha0 = sigmoid(s0 - s1) = sigmoid(2b).
    # With b = ln(3)/2: alpha0 = 3/4, h = 3/4 (1,1) + 1/4 (3,-3) = (1.5, 0) (RAW sources).
    a, b = 0.7, math.log(3.0) / 2
    h, m, lse = agg([[1.0, 1.0], [3.0, -3.0]], [a, b])
    assert np.allclose(h, [1.5, 0.0], atol=1e-15)
    assert m == pytest.approx(a + b, abs=1e-15)
    assert lse == pytest.approx(a + math.log(4 / math.sqrt(3.0)), abs=1e-15)


def test_eps_inside_the_root_of_the_mean_square():
    # eps = 3: v0 = (1,1) -> 1/sqrt(1 + 3) = 1/2 -> key (1/2, 1/2); v1 = (-1,-1) -> (-1/2, -1/2).
    # w = (c, c): s0 = c, s1 = -c, alpha0 = sigmoid(2c); c = ln(2)/2 -> alpha0 = 2/3,
    # h = 2/3 (1,1) + 1/3 (-1,-1) = (1/3, 1/3).
    c = math.log(2.0) / 2
    h, _, _ = agg([[1.0, 1.0], [-1.0, -1.0]], [c, c], eps=3.0)
    assert np.allclose(h, [1 / 3, 1 / 3], atol=1e-15)


def test_three_sources_softmax_and_raw_weighted_sum():
    # D = 1, eps = 0: RMS(v) = sign(v).  v = (2, -5, 0.5), w = ln 2:
    # s = (ln2, -ln2, ln2), weights (2, 1/2, 2)/4.5 = (4/9, 1/9, 4/9),
    # h = 8/9 - 5/9 + 2/9 = 5/9.
    h, m, lse = agg([[2.0], [-5.0], [0.5]], [math.log(2.0)])
    assert h[0] == pytest.approx(5 / 9, abs=1e-15)
    assert m == pytest.approx(math.log(2.0), abs=1e-15)
    assert lse == pytest.approx(math.log(4.5), abs=1e-15)


def test_gain_folds_into_the_query():
    # gamma = (2, 1/2), w = (x, y): w~ = (2x, y/2).  With the sources of the first
    # test, s0 - s1 = y, so y = ln 3 gives alpha0 = 3/4 and h = (1.5, 0) again.
    h, _, _ = agg([[1.0, 1.0], [3.0, -3.0]], [0.3, math.log(3.0)], gamma=[2.0, 0.5])
    assert np.allclose(h, [1.5, 0.0], atol=1e-15)


def test_gain_on_keys_formulation_agrees():
    # An independent formulation: apply gamma to the normalised keys (the
    # "norm(V)" of block_attn_res), then dot with the unfolded w.
    rng = np.random.default_rng(5)
    V = rng.normal(size=(4, 3, 16)) * rng.uniform(0.5, 4, size=(4, 1, 1))
    w, g = rng.normal(0, 0.3, 16), rng.normal(1, 0.1, 16)
    K = V / np.sqrt((V ** 2).mean(-1, keepdims=True) + 1e-8) * g
    logits = np.einsum("d,nrd->nr", w, K)
    alpha = np.exp(logits - logits.max(0)) / np.exp(logits - logits.max(0)).sum(0)
    want = np.einsum("nr,nrd->rd", alpha, V)
    h, _, _ = oracle.depth_aggregate(V, w, g, 1e-8)
    assert np.allclose(h, want, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Invariants and special cases the pages state
# --------------------------------------------------------------------------
def test_zero_query_gives_the_source_mean():
    rng = np.random.default_rng(1)
    V = rng.normal(size=(7, 2, 3, 5))
    h, _, lse = oracle.depth_aggregate(V, np.zeros(5), None, 1e-8)
    assert np.allclose(h, V.mean(0), rtol=0, atol=1e-15)
    assert np.allclose(lse, math.log(7.0), atol=1e-15)


def test_one_source_is_the_identity_bitwise():
    rng = np.random.default_rng(2)
    V = rng.normal(size=(1, 4, 9))
    h, m, lse = oracle.depth_aggregate(V, rng.normal(size=9), rng.normal(1, 0.1, 9), 1e-8)
    assert np.array_equal(h, V[0])
    assert np.array_equal(m, lse)


def test_identical_sources_return_that_source():
    rng = np.random.default_rng(3)
    v = rng.normal(size=(2, 6))
    V = np.stack([v, v, v])
    h, _, _ = oracle.depth_aggregate(V, rng.normal(size=6), None, 1e-8)
    assert np.allclose(h, v, rtol=0, atol=1e-15)


def test_scale_invariance_of_the_weights_at_eps_zero():
    rng = np.random.default_rng(4)
    V = rng.normal(size=(5, 3, 8))
    w = rng.normal(size=8)
    h0, m0, lse0 = oracle.depth_aggregate(V, w, None, 0.0)
    V2 = V.copy()
    V2[2] *= 7.5
    h1, m1, lse1 = oracle.depth_aggregate(V2, w, None, 0.0)
    assert np.allclose(lse1, lse0, rtol=0, atol=1e-13)       # scores unchanged
    # weights unchanged: h1 - h0 = alpha_2 (7.5 - 1) v_2, alpha_2 from the pinned scores
    _, m2, _ = oracle.depth_aggregate(V[2:3], w, None, 0.0)   # s_2 (one source: m = s)
    alpha2 = np.exp(m2 - lse0)
    assert np.allclose(h1 - h0, alpha2[:, None] * 6.5 * V[2], atol=1e-12)


def test_source_permutation_invariance():
    rng = np.random.default_rng(6)
    V = rng.normal(size=(6, 4, 10))
    w, g = rng.normal(size=10), rng.normal(1, 0.1, 10)
    h0, _, l0 = oracle.depth_aggregate(V, w, g, 1e-8)
    h1, _, l1 = oracle.depth_aggregate(V[[3, 0, 5, 1, 4, 2]], w, g, 1e-8)
    assert np.allclose(h0, h1, rtol=0, atol=1e-14)
    assert np.allclose(l0, l1, rtol=0, atol=1e-14)


def test_no_mixing_across_tokens():
    rng = np.random.default_rng(7)
    V = rng.normal(size=(4, 6, 12))
    w = rng.normal(size=12)
    h0, _, _ = oracle.depth_aggregate(V, w, None, 1e-8)
    V2 = V.copy()
    V2[:, 3] += rng.normal(size=(4, 12))
    h1, _, _ = oracle.depth_aggregate(V2, w, None, 1e-8)
    keep = [0, 1, 2, 4, 5]
    assert np.array_equal(h0[keep], h1[keep])
    assert not np.allclose(h0[3], h1[3])


def test_high_precision_brute_force_tiny():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(8)
    V = rng.normal(size=(3, 2, 4)) * 3
    w, g = rng.normal(size=4), rng.normal(1, 0.2, size=4)
    eps = 1e-3
    h, _, lse = oracle.depth_aggregate(V, w, g, eps)
    for r in range(2):
        s = []
        for i in range(3):
            v = [mp.mpf(float(x)) for x in V[i, r]]
            rms = mp.sqrt(sum(x * x for x in v) / 4 + mp.mpf(eps))
            s.append(sum(mp.mpf(float(w[d])) * mp.mpf(float(g[d])) * v[d] / rms for d in range(4)))
        z = sum(mp.e ** si for si in s)
        for d in range(4):
            hd = sum(mp.e ** s[i] / z * mp.mpf(float(V[i, r, d])) for i in range(3))
            assert abs(float(hd) - h[r, d]) < 1e-14
        assert abs(float(mp.log(z)) - lse[r]) < 1e-14


# --------------------------------------------------------------------------
# Online softmax: OS1, OS2, single_source_stats, phase 2
# --------------------------------------------------------------------------
def test_merge_of_any_split_equals_the_whole():
    rng = np.random.default_rng(0)
    V = rng.normal(size=(7, 5)) * rng.uniform(0.5, 4, size=(7, 1))
    q = rng.normal(size=5)
    whole = oracle.os1_stats(V, q)
    for cut in range(1, 7):
        merged = oracle.os2_merge(oracle.os1_stats(V[:cut], q), oracle.os1_stats(V[cut:], q))
        assert np.allclose(merged[1] / merged[2], whole[1] / whole[2], rtol=0, atol=1e-14)
        assert merged[0] + math.log(merged[2]) == pytest.approx(whole[0] + math.log(whole[2]),
                                                                abs=1e-14)


def test_single_source_stats_has_unit_denominator():
    rng = np.random.default_rng(9)
    p = rng.normal(size=6)
    q = rng.normal(size=6)
    m, numer, den = oracle.single_source_stats(p, q)
    assert den == 1.0 and np.array_equal(numer, p)
    assert m == pytest.approx(float(q @ (p / np.sqrt((p ** 2).mean() + 1e-8))), abs=1e-14)


def test_phase2_merge_closed_form():
    # o = (1, 2), lse = ln 3; p = (2, 2) -> RMS(p) = (1, 1); w = (t, -t) -> s_p = 0.
    # M = ln 3: weights 1 and 1/3 -> h = (3 o + p) / 4 = (5/4, 2); merged lse = ln 4.
    h, lse = oracle.block_phase2_merge([[1.0, 2.0]], [math.log(3.0)], [[2.0, 2.0]], [0.4, -0.4],
                                       None, 0.0)
    assert np.allclose(h, [[1.25, 2.0]], atol=1e-15)
    assert lse[0] == pytest.approx(math.log(4.0), abs=1e-15)


def test_phase2_without_partial_passes_through():
    h, lse = oracle.block_phase2_merge([[1.0, -2.0, 3.0]], [0.25], None, [1.0, 1.0, 1.0])
    assert np.array_equal(h, [[1.0, -2.0, 3.0]]) and lse[0] == 0.25


def test_two_phase_equals_monolithic_aggregation():
    rng = np.random.default_rng(10)
    blocks = rng.normal(size=(4, 5, 8)) * rng.uniform(0.5, 8, size=(4, 1, 1))
    p = rng.normal(size=(5, 8)) * 2
    W, G = rng.normal(0, 0.3, size=(3, 8)), rng.normal(1, 0.1, size=(3, 8))
    O, M, LSE = oracle.block_phase1(blocks, W, G)
    for s in range(3):
        h, lse = oracle.block_phase2_merge(O[s], LSE[s], p, W[s], G[s])
        want, _, want_lse = oracle.depth_aggregate(np.concatenate([blocks, p[None]]), W[s], G[s])
        assert np.allclose(h, want, rtol=0, atol=1e-12)
        assert np.allclose(lse, want_lse, rtol=0, atol=1e-12)
        assert np.all(M[s] <= LSE[s]) and np.all(LSE[s] <= M[s] + math.log(4) + 1e-12)


def test_block_two_phase_forward_equals_naive_forward():
    rng = np.random.default_rng(11)
    N, S, R, D = 9, 4, 3, 8
    x = rng.normal(size=(R, D))
    W, G = rng.normal(0, 0.5, size=(N + 1, D)), rng.normal(1, 0.1, size=(N + 1, D))
    U = rng.normal(1, 0.25, size=(N, D))
    H0, y0 = oracle.block_forward_naive(x, W, G, U, S)
    H1, y1 = oracle.block_forward_two_phase(x, W, G, U, S)
    assert np.allclose(H0, H1, rtol=0, atol=1e-12)
    assert np.allclose(y0, y1, rtol=0, atol=1e-12)


def test_block_size_one_is_the_full_stack():
    rng = np.random.default_rng(12)
    N, R, D = 6, 2, 8
    x = rng.normal(size=(R, D))
    W, G = rng.normal(0, 0.5, size=(N + 1, D)), rng.normal(1, 0.1, size=(N + 1, D))
    U = rng.normal(1, 0.25, size=(N, D))
    H, y_block = oracle.block_forward_naive(x, W, G, U, 1)
    V, y_full = oracle.full_stack_forward(x, W, G, U, 1e-8, oracle.F64)
    for l in range(1, N + 1):
        assert np.allclose(V[l], 0.5 * np.tanh(U[l - 1] * H[l - 1]), rtol=0, atol=1e-14)
    assert np.allclose(y_block, y_full, rtol=0, atol=1e-13)


def test_one_block_is_embedding_plus_running_sum():
    rng = np.random.default_rng(13)
    N, R, D = 5, 2, 6
    x = rng.normal(size=(R, D))
    W, G = rng.normal(0, 0.5, size=(N + 1, D)), rng.normal(1, 0.1, size=(N + 1, D))
    U = rng.normal(1, 0.25, size=(N, D))
    H, y = oracle.block_forward_naive(x, W, G, U, N)
    partial = None
    for l in range(N):
        srcs = [x] if partial is None else [x, partial]
        h, _, _ = oracle.depth_aggregate(np.stack(srcs), W[l], G[l])
        assert np.allclose(H[l], h, rtol=0, atol=1e-14)
        out = 0.5 * np.tanh(U[l] * h)
        partial = out if partial is None else partial + out
    want, _, _ = oracle.depth_aggregate(np.stack([x, partial]), W[N], G[N])
    assert np.allclose(y, want, rtol=0, atol=1e-14)


def test_full_stack_first_layers_by_hand():
    rng = np.random.default_rng(14)
    R, D, L = 3, 8, 3
    v0 = rng.normal(size=(R, D))
    W = np.zeros((L + 1, D))                       # zero queries: every h is a plain mean
    U = rng.normal(1, 0.25, size=(L, D))
    V, y = oracle.full_stack_forward(v0, W, None, U, 1e-8, oracle.F64)
    v1 = 0.5 * np.tanh(U[0] * v0)                  # one source -> h_1 = v0
    v2 = 0.5 * np.tanh(U[1] * (v0 + v1) / 2)
    v3 = 0.5 * np.tanh(U[2] * (v0 + v1 + v2) / 3)
    assert np.allclose(V[1], v1, atol=1e-15) and np.allclose(V[2], v2, atol=1e-15)
    assert np.allclose(V[3], v3, atol=1e-15)
    assert np.allclose(y, (v0 + v1 + v2 + v3) / 4, atol=1e-15)


@pytest.mark.parametrize("S", [1, 2, 3, 5, 7, 9, 12])
def test_full_two_phase_schedule_equals_the_naive_full_stack(S):
    # Phase 1 over the completed sources + OS2 merges of the intra-block ones reach,
    # in exact arithmetic, the direct aggregation over every earlier source.
    rng = np.random.default_rng(20 + S)
    L, R, D = 9, 3, 8
    v0 = rng.normal(size=(R, D)) * 2
    W, G = rng.normal(0, 0.5, size=(L + 1, D)), rng.normal(1, 0.1, size=(L + 1, D))
    U = rng.normal(1, 0.25, size=(L, D))
    V0, y0 = oracle.full_stack_forward(v0, W, G, U, 1e-8, oracle.F64)
    V1, y1 = oracle.full_stack_two_phase(v0, W, G, U, S, 1e-8, oracle.F64)
    assert np.allclose(V1, V0, rtol=0, atol=1e-12)
    assert np.allclose(y1, y0, rtol=0, atol=1e-12)


def test_full_two_phase_rounds_what_it_materialises():
    rng = np.random.default_rng(30)
    L, R, D = 7, 2, 16
    v0 = oracle.round_to(rng.normal(size=(R, D)), oracle.BF16)
    W, G = rng.normal(0, 0.5, size=(L + 1, D)), rng.normal(1, 0.1, size=(L + 1, D))
    U = rng.normal(1, 0.25, size=(L, D))
    V, y = oracle.full_stack_two_phase(v0, W, G, U, 3, 1e-8, oracle.BF16)
    assert np.array_equal(V, oracle.round_to(V, oracle.BF16))       # every v_l is a bf16 tensor
    Vn, yn = oracle.full_stack_forward(v0, W, G, U, 1e-8, oracle.BF16)
    assert np.allclose(V, Vn, atol=0.02) and np.allclose(y, yn, atol=0.02)  # a few bf16 ulps apart


def test_chain_rounding_points():
    # The two-phase chain rounds o, h and p to the I/O dtype; in F64 mode it is exact
    # and must equal the unrounded two-phase recurrence of one block.
    rng = np.random.default_rng(15)
    n, S, R, D = 3, 4, 2, 8
    blocks = [rng.normal(size=(R, D)) * 3 for _ in range(n)]
    W, G, U = rng.normal(0, 0.3, (S, D)), rng.normal(1, 0.1, (S, D)), rng.normal(1, 0.25, (S, D))
    H, P = oracle.block_two_phase_chain(blocks, W, G, U, 1e-8, oracle.F64)
    partial = None
    for k in range(S):
        srcs = blocks if partial is None else blocks + [partial]
        h, _, _ = oracle.depth_aggregate(np.stack(srcs), W[k], G[k])
        assert np.allclose(H[k], h, rtol=0, atol=1e-12)
        out = 0.5 * np.tanh(U[k] * h)
        partial = out if partial is None else partial + out
    assert np.allclose(P, partial, rtol=0, atol=1e-12)
    Hb, Pb = oracle.block_two_phase_chain(blocks, W, G, U, 1e-8, oracle.BF16)
    assert np.array_equal(Pb, oracle.round_to(Pb, oracle.BF16))   # stored partial is bf16
    assert np.allclose(Pb, P, atol=0.05)


# --------------------------------------------------------------------------
# The sublayer pre-norm fused into the merge ("Depth attention 与 online merge
# reference": optional fused output RMSNorm; "Kimi Linear 与 K3 中的接入":
# merge + partial update + RMSNorm fused on the decode path)
# --------------------------------------------------------------------------
def test_rms_norm_closed_forms():
    # x = (2, 0): mean square 2; with eps = 2 the root is 2, so y = (1, 0) (.) w.
    assert np.array_equal(oracle.rms_norm([[2.0, 0.0]], [3.0, 5.0], 2.0), [[3.0, 0.0]])
    # eps inside the root, added to the MEAN (not the sum): x = (3, 4), eps = 0 -> root sqrt(12.5).
    y = oracle.rms_norm([[3.0, 4.0]], None, 0.0)
    assert np.allclose(y, [[3 / math.sqrt(12.5), 4 / math.sqrt(12.5)]], rtol=0, atol=1e-15)
    # a constant row normalises to the weight (eps = 0), whatever its scale and sign
    w = np.array([0.5, -1.0, 2.0, 3.0])
    assert np.allclose(oracle.rms_norm([[7.0] * 4], w, 0.0), [w], rtol=0, atol=1e-15)
    assert np.allclose(oracle.rms_norm([[-0.25] * 4], w, 0.0), [-w], rtol=0, atol=1e-15)


def test_rms_norm_invariants():
    rng = np.random.default_rng(16)
    x = rng.normal(size=(5, 32)) * rng.uniform(0.1, 10, size=(5, 1))
    y = oracle.rms_norm(x, None, 0.0)
    assert np.allclose((y ** 2).mean(axis=1), 1.0, rtol=0, atol=1e-13)      # unit mean square
    assert np.allclose(oracle.rms_norm(3.5 * x, None, 0.0), y, rtol=0, atol=1e-13)  # scale-free
    assert np.allclose(y * np.sign(x), np.abs(y), rtol=0, atol=0)           # sign kept per element
    w = rng.normal(1, 0.2, size=32)
    yw = oracle.rms_norm(x, w, 1e-6)
    # a second formulation: numpy's norm of the row, sqrt(||x||^2 / D + eps)
    want = x / np.sqrt(np.linalg.norm(x, axis=1, keepdims=True) ** 2 / 32 + 1e-6) * w
    assert np.allclose(yw, want, rtol=1e-14, atol=0)
    assert np.array_equal(oracle.rms_norm(x[2:3], w, 1e-6), yw[2:3])        # rows independent


def test_normed_chain_equals_normed_naive_stack():
    # One block over the embedding alone: the two-phase chain (phase 1 + merges) with
    # pre-norm weights equals forward_naive (direct aggregation) with the same weights.
    rng = np.random.default_rng(17)
    S, R, D = 4, 3, 8
    x = rng.normal(size=(R, D)) * 2
    W, G = rng.normal(0, 0.5, size=(S + 1, D)), rng.normal(1, 0.1, size=(S + 1, D))
    U, NW = rng.normal(1, 0.25, size=(S, D)), rng.normal(1, 0.1, size=(S, D))
    Hn, _ = oracle.block_forward_naive(x, W, G, U, S, NW=NW, norm_eps=1e-5)
    Hc, Pc = oracle.block_two_phase_chain([x], W[:S], G[:S], U, 1e-8, oracle.F64, NW=NW, norm_eps=1e-5)
    assert np.allclose(Hc, Hn, rtol=0, atol=1e-12)
    # the sublayer inputs are normalised rows: mean square of y / NW is 1 up to eps
    assert np.allclose(((Hc / NW[:, None, :]) ** 2).mean(axis=2), 1.0, atol=1e-4)
    # and the norm changes the recurrence (not silently ignored)
    H0, P0 = oracle.block_two_phase_chain([x], W[:S], G[:S], U, 1e-8, oracle.F64)
    assert not np.allclose(P0, Pc, atol=1e-3)
    # step by step by hand: partial = sum_k 0.5 tanh(u_k (.) y_k)
    assert np.allclose(Pc, sum(0.5 * np.tanh(U[k] * Hc[k]) for k in range(S)), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Backward of the depth aggregation (the operator's forward/backward,
# "Depth attention 与 online merge reference", "公开实现边界")
# --------------------------------------------------------------------------
def test_backward_closed_form_two_sources():
    # D = 1, eps = 0: RMS(v) = sign(v), so with v0 = 1, v1 = -2 and q~ = ln(3)/2 the scores are
    # +-ln(3)/2, alpha = (3/4, 1/4), h = 1/4.  With dh = 1: da = (1, -2), sum alpha da = 1/4,
    # ds = (3/4 * 3/4, 1/4 * -9/4) = (9/16, -9/16), dq~ = 9/16 * 1 + (-9/16) * (-1) = 9/8.
    # The scores do not depend on |v| (D = 1, eps = 0), so dv is the direct term alpha dh.
    q = math.log(3) / 2
    dV, dw, dg = oracle.depth_aggregate_backward([[[1.0]], [[-2.0]]], [q / 2], [2.0], 0.0, [[1.0]])
    assert np.allclose(dV.ravel(), [0.75, 0.25], rtol=0, atol=1e-15)
    assert np.allclose(dw, [9 / 8 * 2.0], rtol=0, atol=1e-14)          # dw = dq~ * gamma
    assert np.allclose(dg, [9 / 8 * q / 2], rtol=0, atol=1e-14)        # dgamma = dq~ * w


def test_backward_matches_central_differences_of_the_forward():
    rng = np.random.default_rng(18)
    n, R, D, eps = 3, 2, 5, 1e-2
    V = rng.normal(size=(n, R, D)) * rng.uniform(0.5, 3, size=(n, 1, 1))
    w, gam = rng.normal(0, 0.7, size=D), rng.normal(1, 0.2, size=D)
    dh = rng.normal(size=(R, D))

    def loss(V_, w_, g_):
        h, _, _ = oracle.depth_aggregate(V_, w_, g_, eps)
        return float(np.sum(dh * h))

    dV, dw, dg = oracle.depth_aggregate_backward(list(V), w, gam, eps, dh)
    step = 1e-6
    num = np.zeros_like(V)
    for idx in np.ndindex(V.shape):
        Vp, Vm = V.copy(), V.copy()
        Vp[idx] += step
        Vm[idx] -= step
        num[idx] = (loss(Vp, w, gam) - loss(Vm, w, gam)) / (2 * step)
    assert np.allclose(dV, num, rtol=0, atol=1e-8)
    for arr, grad, which in ((w, dw, "w"), (gam, dg, "gamma")):
        num = np.zeros(D)
        for d in range(D):
            ap, am = arr.copy(), arr.copy()
            ap[d] += step
            am[d] -= step
            args_p = (V, ap, gam) if which == "w" else (V, w, ap)
            args_m = (V, am, gam) if which == "w" else (V, w, am)
            num[d] = (loss(*args_p) - loss(*args_m)) / (2 * step)
        assert np.allclose(grad, num, rtol=0, atol=1e-8), which


def test_backward_invariants():
    rng = np.random.default_rng(19)
    n, R, D = 4, 3, 16
    V = rng.normal(size=(n, R, D)) * rng.uniform(0.5, 8, size=(n, 1, 1))
    w, gam = rng.normal(0, 0.3, size=D), rng.normal(1, 0.1, size=D)
    dh = rng.normal(size=(R, D))
    # one source: h = v whatever the query -> dv = dh exactly, no query gradient
    dV1, dw1, dg1 = oracle.depth_aggregate_backward([V[0]], w, gam, 1e-8, dh)
    assert np.array_equal(dV1[0], dh) and not np.any(dw1) and not np.any(dg1)
    # no upstream gradient -> no gradient
    dV0, dw0, _ = oracle.depth_aggregate_backward(list(V), w, gam, 1e-8, np.zeros((R, D)))
    assert not np.any(dV0) and not np.any(dw0)
    # eps = 0: each score is invariant to the scale of its own source, so the radial part of
    # dv_i is only the direct term: sum_i v_i . dv_i = sum_i alpha_i dh . v_i = dh . h
    dV, _, _ = oracle.depth_aggregate_backward(list(V), w, gam, 0.0, dh)
    h, _, _ = oracle.depth_aggregate(V, w, gam, 0.0)
    assert np.allclose(np.einsum("nrd,nrd->r", V, dV), np.sum(dh * h, axis=1), rtol=1e-12, atol=0)
    # identical sources: equal scores whatever the query, so alpha = 1/n and every ds is 0:
    # no query gradient, and each source gets dh / n
    same = [V[0]] * n
    dVs, dws, _ = oracle.depth_aggregate_backward(same, w, gam, 1e-8, dh)
    assert np.allclose(dws, 0.0, atol=1e-15) and np.allclose(dVs, dh / n, rtol=0, atol=1e-15)


# --------------------------------------------------------------------------
# Rounding to the I/O dtype
# --------------------------------------------------------------------------
def test_bf16_rounding_ties_and_ranges():
    r = oracle.round_bf16_scalar
    assert r(1 + 2 ** -8) == 1.0                       # tie -> even (mantissa 0)
    assert r(1 + 3 * 2 ** -8) == 1 + 2 ** -6           # tie -> even (mantissa 2)
    assert r(1 + 2 ** -8 + 2 ** -20) == 1 + 2 ** -7    # above the tie
    assert r(2.0 ** -133) == 2.0 ** -133               # smallest subnormal
    assert r(2.0 ** -134) == 0.0                       # tie with zero -> even
    assert r(3 * 2.0 ** -134) == 2.0 ** -132
    assert r(2.0 ** 128) == math.inf
    assert r(-(2 - 2 ** -7) * 2.0 ** 127) == -(2 - 2 ** -7) * 2.0 ** 127


def test_bf16_rounding_matches_torch_on_fp32_values():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(20000, generator=g) * torch.exp(torch.randn(20000, generator=g) * 8)
    want = x.to(torch.bfloat16).double().numpy()
    got = oracle.round_to(x.double().numpy(), oracle.BF16)
    assert np.array_equal(got, want)
    got32 = oracle.round_to(x.double().numpy() * (1 + 1e-9), oracle.F32)
    assert np.array_equal(got32, (x.double() * (1 + 1e-9)).float().double().numpy())


# --------------------------------------------------------------------------
# Bookkeeping
# --------------------------------------------------------------------------
def test_atomic_block_size_examples_from_the_pages():
    assert oracle.atomic_block_size(24) == 6           # ceil(24/8) = 3 DecoderBlocks -> 6
    assert oracle.atomic_block_size(93) == 24          # K3: 12 DecoderBlocks -> 24
    assert oracle.atomic_block_size(4, 2) == 4         # --attnres-block-size 2
    assert oracle.atomic_block_size(4) == 2
    assert 48 // oracle.atomic_block_size(24) == 8     # N/S = 8 blocks


def test_schedule_block_size_one_reproduces_full():
    sched = oracle.block_schedule(7, 1)
    for l in range(7):
        assert sched[l] == list(range(l + 1))         # sublayer l+1 sees v_0..v_l
    assert sched[7] == list(range(8))


def test_schedule_single_block_is_embedding_plus_partial():
    sched = oracle.block_schedule(5, 5)
    assert sched[0] == [0] and all(s == [0, -1] for s in sched[1:5]) and sched[5] == [0, 1]


def test_schedule_k3_counts():
    sched = oracle.block_schedule(186, 24)
    assert len(sched[186]) == 9                        # embedding + 8 blocks (last one short)
    assert max(len(s) for s in sched[:186]) == 9
    assert sched[168] == list(range(8))                # first sublayer of the short block
    assert sched[169] == list(range(8)) + [-1]
