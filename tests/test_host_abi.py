"""CPU-only checks of libattnres.so: it loads, exports every declared symbol,
rejects bad arguments before launching anything, and its host bookkeeping
matches the oracle bit for bit.  No compute entry point runs here."""
import ctypes
import json
import math
import os
import re

import pytest

import oracle
from transformer_depth_wise_gb300 import _lib, accounting, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x7F0000000000      # 16-byte aligned stand-in for a device pointer (never dereferenced)
OK, NULL, SHAPE, DTYPE, ALIGN, MANY, CUDA, CAP, VALUE = 0, -1, -2, -3, -4, -5, -6, -7, -8


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "attnres.h")).read()
    return sorted(set(re.findall(r"^(?:int|int64_t|const char \*)\s*(attnres_\w+)\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    L = _lib.lib()
    names = declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SIGNATURES)


def test_status_strings():
    L = _lib.lib()
    for code in _lib.STATUS:
        s = L.attnres_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.attnres_status_string(12345).decode() == "unknown status"


def agg(sources, n=None, B=2, T=3, D=64, dtype=1, q=FAKE, g=None, eps=1e-8, out=FAKE):
    L = _lib.lib()
    arr = None if sources is None else _lib.ptr_array(sources)
    return L.attnres_depth_aggregate(arr, len(sources) if n is None else n, B, T, D, dtype, q, g, eps,
                                     out, None, None, None)


def test_depth_aggregate_argument_checks():
    assert agg([FAKE] * 3, dtype=7) == DTYPE
    assert agg([FAKE] * 3, D=0) == SHAPE
    assert agg([FAKE] * 3, B=-1) == SHAPE
    assert agg([FAKE] * 3, D=36, dtype=1) == ALIGN           # bf16 needs D % 8 == 0
    assert agg([FAKE] * 3, D=34, dtype=0) == ALIGN           # fp32 needs D % 4 == 0
    assert agg(None, n=3) == NULL
    assert agg([FAKE] * 3, q=None) == NULL
    assert agg([FAKE] * 3, out=None) == NULL
    assert agg([FAKE, 0, FAKE]) == NULL
    assert agg([FAKE] * 3, n=0) == SHAPE
    assert agg([FAKE] * 257) == MANY
    assert agg([FAKE] * 3, eps=-1.0) == VALUE
    assert agg([FAKE] * 3, eps=math.nan) == VALUE
    assert agg([FAKE] * 3, eps=math.inf) == VALUE
    assert agg([FAKE, FAKE + 8, FAKE]) == ALIGN
    assert agg([FAKE] * 3, q=FAKE + 4) == ALIGN
    assert agg([FAKE] * 3, g=FAKE + 4) == ALIGN
    assert agg([FAKE] * 3, D=16384, dtype=1) == SHAPE        # beyond the kernel family
    assert agg([FAKE] * 3, B=0) == OK                         # empty: nothing launched
    assert agg([FAKE] * 3, T=0) == OK


def test_phase1_argument_checks():
    L = _lib.lib()
    arr = _lib.ptr_array([FAKE] * 9)

    def p1(n=9, S=24, lse=FAKE, out=FAKE, B=1, D=4096, dtype=1, q=FAKE):
        return L.attnres_block_phase1(arr, n, B, 4, D, dtype, q, None, S, 1e-8, out, None, lse, None)

    assert p1(lse=None) == NULL
    assert p1(out=None) == NULL
    assert p1(q=None) == NULL
    assert p1(S=0) == SHAPE
    assert p1(S=65) == SHAPE
    assert p1(n=0) == SHAPE
    arr17 = _lib.ptr_array([FAKE] * 17)
    assert L.attnres_block_phase1(arr17, 17, 1, 4, 4096, 1, FAKE, None, 24, 1e-8, FAKE, None, FAKE, None) == MANY
    assert p1(D=4100) == ALIGN
    assert p1(B=0) == OK


def test_merge_and_update_argument_checks():
    L = _lib.lib()
    m = L.attnres_block_phase2_merge
    assert m(None, FAKE, FAKE, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, None, None) == NULL
    assert m(FAKE, None, FAKE, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, None, None) == NULL
    assert m(FAKE, FAKE, FAKE + 2, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, None, None) == ALIGN
    assert m(FAKE, FAKE, FAKE, 1, 2, 64, 1, FAKE, None, -1.0, FAKE, None, None) == VALUE
    assert m(FAKE, FAKE, None, 0, 2, 64, 1, FAKE, None, 1e-8, FAKE, None, None) == OK
    mu = L.attnres_block_merge_update

    def fused(h=FAKE, nw=None, neps=1e-6, y=None, lse=FAKE, B=1, D=64):
        return mu(FAKE, lse, FAKE, FAKE, None, B, 2, D, 1, FAKE, None, 1e-8, FAKE, h, None, nw, neps, y, None)

    assert fused(lse=None) == NULL
    assert fused(h=None) == NULL                              # nothing to write
    assert fused(nw=FAKE) == NULL                             # weight without an output
    assert fused(y=FAKE) == NULL                              # output without a weight
    assert fused(nw=FAKE, y=FAKE, neps=-1.0) == VALUE
    assert fused(nw=FAKE, y=FAKE, neps=math.nan) == VALUE
    assert fused(nw=FAKE + 4, y=FAKE) == ALIGN
    assert fused(D=60) == ALIGN
    assert fused(D=32768) == SHAPE                            # beyond the kernel family
    assert fused(B=0, h=None) == OK
    n = L.attnres_rms_norm
    assert n(FAKE, 1, 2, 64, 1, None, 1e-6, FAKE, None) == NULL
    assert n(FAKE, 1, 2, 64, 1, FAKE, -1.0, FAKE, None) == VALUE
    assert n(FAKE + 8, 1, 2, 64, 1, FAKE, 1e-6, FAKE, None) == ALIGN
    assert n(FAKE, 1, 2, 64, 9, FAKE, 1e-6, FAKE, None) == DTYPE
    assert n(FAKE, 1, 0, 64, 1, FAKE, 1e-6, FAKE, None) == OK
    u = L.attnres_partial_update
    assert u(FAKE, None, None, 1, 2, 64, 1, FAKE, None) == NULL
    assert u(FAKE, None, FAKE, 1, 2, 60, 1, FAKE, None) == ALIGN
    assert u(FAKE, None, FAKE, 1, 0, 64, 1, FAKE, None) == OK


def test_backward_argument_checks():
    L = _lib.lib()
    arr = _lib.ptr_array([FAKE] * 3)
    garr = _lib.ptr_array([FAKE + 4096] * 3)

    def bwd(n=3, B=1, D=64, dtype=1, q=FAKE, dh=FAKE, g=garr, acc=0, gq=FAKE, ws=FAKE, wsr=64, eps=1e-8):
        return L.attnres_depth_aggregate_backward(arr, n, B, 2, D, dtype, q, None, eps, dh, g, acc, gq, None,
                                                  ws, wsr, None)

    assert bwd(q=None) == NULL
    assert bwd(dh=None) == NULL
    assert bwd(g=None) == NULL
    assert bwd(ws=None) == NULL                          # a query gradient needs the workspace
    assert bwd(wsr=0) == CAP
    assert bwd(acc=2) == VALUE
    assert bwd(eps=-1.0) == VALUE
    assert bwd(n=0) == SHAPE
    assert bwd(n=257) == MANY
    assert bwd(D=36) == ALIGN
    assert bwd(D=16384) == SHAPE                         # beyond the kernel family (bf16: 8192)
    assert bwd(gq=FAKE + 4) == ALIGN
    assert bwd(dh=FAKE + 8) == ALIGN
    na = L.attnres_depth_aggregate_backward_noalloc
    assert na(arr, 3, 1, 2, 16384, 1, FAKE, None, 1e-8, FAKE, garr, 0, FAKE, None, None) == SHAPE
    assert na(arr, 3, 1, 2, 64, 5, FAKE, None, 1e-8, FAKE, garr, 0, FAKE, None, None) == DTYPE
    assert na(arr, 3, 1, 2, 64, 1, None, None, 1e-8, FAKE, garr, 0, None, None, None) == NULL
    # every argument is checked before the scratch is looked up (a CUDA call,
    # which fails here without a GPU): bad arguments report their own status
    assert na(arr, 3, 1, 2, 64, 1, None, None, 1e-8, FAKE, garr, 0, FAKE, None, None) == NULL
    assert na(arr, 3, 1, 2, 64, 1, FAKE, None, 1e-8, None, garr, 0, FAKE, None, None) == NULL
    assert na(arr, 3, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE + 8, garr, 0, FAKE, None, None) == ALIGN
    assert na(arr, 3, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, garr, 0, FAKE + 4, None, None) == ALIGN
    assert na(arr, 3, 1, 2, 64, 1, FAKE, None, -1.0, FAKE, garr, 0, FAKE, None, None) == VALUE
    assert na(arr, 3, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, garr, 3, FAKE, None, None) == VALUE
    assert na(arr, 0, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, garr, 0, FAKE, None, None) == SHAPE
    assert na(arr, 257, 1, 2, 64, 1, FAKE, None, 1e-8, FAKE, garr, 0, FAKE, None, None) == MANY
    assert L.attnres_depth_aggregate_backward_workspace_rows(16384, 1) == SHAPE
    assert L.attnres_depth_aggregate_backward_workspace_rows(64, 7) == DTYPE


def test_wait_limit_knob():
    L = _lib.lib()
    assert L.attnres_set_wait_limit(-1) == VALUE
    assert L.attnres_set_wait_limit(1000) == OK
    assert L.attnres_set_wait_limit(0) == OK                # back to the default


def test_full_stack_argument_checks():
    L = _lib.lib()
    f = L.attnres_full_stack_forward
    arr = _lib.ptr_array([FAKE] * 5)
    assert f(arr, 0, 1, 2, 64, 1, FAKE, None, FAKE, 1e-8, FAKE, None) == SHAPE
    assert f(arr, 4, 1, 2, 64, 1, FAKE, None, None, 1e-8, FAKE, None) == NULL
    big = _lib.ptr_array([FAKE] * 257)
    assert f(big, 256, 1, 2, 64, 1, FAKE, None, FAKE, 1e-8, FAKE, None) == MANY
    assert f(arr, 4, 0, 2, 64, 1, FAKE, None, FAKE, 1e-8, FAKE, None) == OK


def test_full_two_phase_argument_checks():
    # L = 5 sublayers in blocks of S = 2: every block's phase 1 has at most ten
    # sources, so the shape checks need no GPU
    L = _lib.lib()
    wsb = L.attnres_full_stack_two_phase_workspace_bytes
    assert wsb(5, 2, 1, 4, 64, 1) > 0
    assert wsb(0, 2, 1, 4, 64, 1) == SHAPE
    assert wsb(5, 0, 1, 4, 64, 1) == SHAPE
    assert wsb(5, 2, 1, 4, 64, 7) == DTYPE
    assert wsb(5, 2, 1, 4, 36, 1) == ALIGN
    need = wsb(5, 2, 1, 4, 64, 1)
    arr = _lib.ptr_array([FAKE] * 6)
    tp = L.attnres_full_stack_two_phase

    def call(arr=arr, Lsub=5, S=2, B=1, ws=FAKE, wsbytes=need, eps=1e-8, y=FAKE, q=FAKE, u=FAKE):
        return tp(arr, Lsub, S, B, 4, 64, 1, q, None, u, eps, y, ws, wsbytes, None)

    assert call(S=0) == SHAPE
    assert call(S=65) == SHAPE
    assert call(Lsub=0) == SHAPE
    big = _lib.ptr_array([FAKE] * 257)
    assert call(arr=big, Lsub=256) == MANY
    assert call(eps=-1.0) == VALUE
    assert call(B=0, arr=None, ws=None, y=None, q=None, u=None) == OK    # empty: nothing checked or launched
    assert call(arr=None) == NULL
    assert call(ws=None) == NULL
    assert call(q=None) == NULL
    assert call(arr=_lib.ptr_array([FAKE] * 5 + [0])) == NULL
    assert call(arr=_lib.ptr_array([FAKE] * 5 + [FAKE + 8])) == ALIGN
    assert call(ws=FAKE + 16) == ALIGN                                   # the workspace is 256-byte aligned
    assert call(wsbytes=need - 1) == CAP
    # the backward with no token rows: nothing is read, launched or written
    garr = _lib.ptr_array([FAKE + 4096] * 3)
    assert L.attnres_depth_aggregate_backward(_lib.ptr_array([FAKE] * 3), 3, 0, 2, 64, 1, FAKE, None, 1e-8, FAKE,
                                              garr, 0, None, None, None, 0, None) == OK


@pytest.mark.parametrize("N", [1, 2, 5, 8, 23, 48, 93, 186])
def test_schedule_matches_oracle_bit_exact(N):
    for S in sorted({1, 2, 3, 4, 6, 7, 24, N, N + 5}):
        assert api.block_schedule(N, S) == oracle.block_schedule(N, S), (N, S)


def test_schedule_errors():
    L = _lib.lib()
    counts = (ctypes.c_int * 9)()
    ids = (ctypes.c_int * 4)()
    assert L.attnres_block_schedule(8, 2, counts, ids, 4) == CAP
    assert L.attnres_block_schedule(0, 2, counts, ids, 4) == SHAPE
    assert L.attnres_block_schedule(8, 0, counts, ids, 4) == VALUE
    assert L.attnres_block_schedule(8, 2, None, ids, 4) == NULL


def test_atomic_block_size_matches_oracle():
    for layers in range(1, 200):
        assert api.atomic_block_size(layers) == oracle.atomic_block_size(layers)
        for bs in (1, 2, 3, 12, 40):
            assert api.atomic_block_size(layers, bs) == oracle.atomic_block_size(layers, bs)
    assert _lib.lib().attnres_atomic_block_size(24, 0) == VALUE
    assert _lib.lib().attnres_atomic_block_size(0, -1) == SHAPE


# --------------------------------------------------------------------------
# Figures printed on the pages (tests/golden/pages_figures.json)
# --------------------------------------------------------------------------
GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "pages_figures.json")))


def test_golden_atomic_block_size():
    for c in GOLD["atomic_block_size"]["cases"]:
        got = api.atomic_block_size(c["num_hidden_layers"], c["attnres_block_size"])
        assert got == c["atomic"]
        if "blocks_of_48" in c:
            assert 2 * c["num_hidden_layers"] // got == c["blocks_of_48"]


def test_golden_extra_parameter_table():
    for r in GOLD["extra_parameters"]["rows"]:
        N = 2 * r["L"]                                    # atomic sublayers
        assert N == r["N"]
        assert 2 * (N + 1) * r["D"] == r["params"]        # one query + one gain per aggregation


def test_golden_k3_source_count():
    g = GOLD["k3_sources"]
    sched = api.block_schedule(g["num_atomic"], g["block_size"])
    assert len(sched[-1]) == g["final_sources"]


def test_golden_residual_io_model():
    g = GOLD["residual_io_model"]
    assert accounting.residual_io_per_layer("standard", g["L"], g["N"], g["S"]) == g["standard_d"]
    assert accounting.residual_io_per_layer("block", g["L"], g["N"], g["S"]) == g["block_d"]
    assert accounting.residual_io_per_layer("full_two_phase", g["L"], g["N"], g["S"]) == g["full_two_phase_d"]


def test_golden_prefill_cache():
    g = GOLD["prefill_cache"]
    total = accounting.prefill_block_cache_bytes(g["tokens"], g["blocks"], g["D"], g["elt_bytes"])
    assert round(total / 1e9) == g["total_gb_approx"]
    per_rank = accounting.prefill_block_cache_bytes(g["tokens"], g["blocks"], g["D"], g["elt_bytes"],
                                                    g["ranks"])
    assert round(per_rank / 1e9, 1) == g["per_rank_gb_approx"]
    chunk = accounting.prefill_block_cache_bytes(g["chunk_tokens"], g["blocks"], g["D"], g["elt_bytes"],
                                                 g["ranks"])
    assert chunk / 1e9 < g["chunk_gb_below"]


def test_kernel_byte_accounting_by_hand():
    # Block single aggregation [4,4096,2048] bf16, n = 10: 11 rows of 4 KiB per token.
    assert accounting.aggregate_bytes(10, 4 * 4096, 2048, 2) == 11 * 16384 * 4096
    # Backward of that aggregation: 11 rows read, 10 written (+10 read when accumulating).
    assert accounting.aggregate_backward_bytes(10, 4 * 4096, 2048, 2) == 21 * 16384 * 4096
    assert accounting.aggregate_backward_bytes(10, 4 * 4096, 2048, 2, True) == 31 * 16384 * 4096
    # Two-phase block, 9 summaries [8,4096,4096] bf16, S = 24.
    b = accounting.two_phase_block_bytes(9, 24, 32768, 4096, 2)
    assert b["phase1"] == 32768 * (33 * 8192 + 24 * 4)
    assert b["merges"] == 23 * 32768 * (3 * 8192 + 4)
    fb = accounting.two_phase_block_bytes(9, 24, 32768, 4096, 2, fused=True)
    assert fb["merges"] == 32768 * ((4 * 8192 + 4) + 22 * (5 * 8192 + 4))
    assert fb["updates"] == 32768 * 3 * 8192
    # fused: 117 row transfers per token after phase 1, against 140 unfused
    assert (fb["merges"] + fb["updates"]) // 32768 // 8192 == 117
    assert (b["merges"] + b["updates"]) // 32768 // 8192 == 140
    # Full two-phase, S = L: one block, phase 1 over v_0 only (1 read + L writes + lse),
    # sublayer j reads o, lse and j intra sources and writes v_l; then the final L+1 + 1.
    L = 5
    want = (1 + L) * 4096 + L * 4 + sum((j + 2) * 4096 + 4 for j in range(L)) + (L + 2) * 4096
    assert accounting.full_two_phase_bytes(L, L, 1, 2048, 2) == want
    # S = 1 gives back the naive stack's source reads (plus the o row and lse written and read)
    naive = accounting.full_stack_bytes(186, 1, 2048, 2)
    assert accounting.full_two_phase_bytes(186, 1, 1, 2048, 2) == naive + 186 * (2 * 4096 + 8)
    # Full stack, 186 sublayers: 17391 + 187 reads and 187 writes per token row.
    assert accounting.full_stack_bytes(186, 2048, 2048, 2) == 2048 * (17391 + 187 + 187) * 4096
