"""Algorithmic byte counts (what the method itself must read and write).

Used by the benchmark for the roofline ("achieved" = algorithmic bytes per
launch / launch time) and pinned by tests against the figures the pages
print for their residual I/O and prefill-cache models.
"""
from __future__ import annotations

BF16 = 2
F32 = 4


def aggregate_bytes(n: int, rows: int, D: int, elt: int, stats: bool = False) -> int:
    """One depth aggregation: read n source rows, write one output row per token."""
    return rows * (n + 1) * D * elt + (rows * 8 if stats else 0)


def aggregate_backward_bytes(n: int, rows: int, D: int, elt: int, accumulate: bool = False) -> int:
    """Backward of one aggregation: read n sources and dh, write n source
    gradients (and read them first when accumulating).  The [D] query and
    gain gradients and the per-CTA partials are negligible and not counted."""
    return rows * ((n + 1) + n + (n if accumulate else 0)) * D * elt


def phase1_bytes(n: int, S: int, rows: int, D: int, elt: int, with_max: bool = False) -> int:
    """Phase 1: read n summaries once, write S outputs and S lse (and S max) per token."""
    return rows * ((n + S) * D * elt + S * 4 * (2 if with_max else 1))


def merge_bytes(rows: int, D: int, elt: int) -> int:
    """One phase-2 merge: read o and lse and the partial, write h."""
    return rows * (3 * D * elt + 4)


def partial_update_bytes(rows: int, D: int, elt: int, first: bool) -> int:
    """p_k = p_{k-1} + f(h_k): read h (and p unless first), write p."""
    return rows * ((2 if first else 3) * D * elt)


def merge_update_bytes(rows: int, D: int, elt: int, first: bool) -> int:
    """Fused update + merge: read o, the sublayer row and p_in (not on the first
    step), and lse; write p and h."""
    return rows * (((4 if first else 5) * D * elt) + 4)


def two_phase_block_bytes(n: int, S: int, rows: int, D: int, elt: int, fused: bool = False) -> dict:
    """Per-kernel algorithmic bytes of one block pass.

    Unfused: phase 1, S-1 merges, S updates.  Fused: phase 1, S-1 fused
    update+merge steps, 1 final update.
    """
    p1 = phase1_bytes(n, S, rows, D, elt)
    if fused:
        mg = merge_update_bytes(rows, D, elt, True) + (S - 2) * merge_update_bytes(rows, D, elt, False)
        up = partial_update_bytes(rows, D, elt, S == 1)
    else:
        mg = (S - 1) * merge_bytes(rows, D, elt)
        up = partial_update_bytes(rows, D, elt, True) + (S - 1) * partial_update_bytes(rows, D, elt, False)
    return {"phase1": p1, "merges": mg, "updates": up, "attnres": p1 + mg, "total": p1 + mg + up}


def full_stack_bytes(L: int, rows: int, D: int, elt: int) -> int:
    """Full stack, f fused: sublayer l reads l sources and writes v_l; the final reads L+1, writes y."""
    reads = sum(range(1, L + 1)) + (L + 1)
    writes = L + 1
    return rows * (reads + writes) * D * elt


def full_two_phase_bytes(L: int, S: int, rows: int, D: int, elt: int) -> int:
    """Full stack with the two-phase schedule of block size S, f fused.

    Per block of Sb sublayers after `start` completed ones: phase 1 reads the
    start + 1 completed sources once and writes Sb outputs (+ Sb lse); sublayer
    j of the block reads its output and lse and its j intra-block sources and
    writes v_l.  Then the final aggregate reads L + 1 sources and writes y.
    """
    row = D * elt
    total = 0
    for start in range(0, L, S):
        Sb = min(S, L - start)
        total += (start + 1 + Sb) * row + Sb * 4
        total += sum((1 + j + 1) * row + 4 for j in range(Sb))
    total += (L + 2) * row
    return rows * total


# ---------------------------------------------------------------------------
# The pages' analytic models ("推理：block representations 像一份 depth KV cache")
# ---------------------------------------------------------------------------
def residual_io_per_layer(kind: str, L: int, N: int, S: int) -> float:
    """Residual-mechanism I/O per token per layer, in units of d.

    standard residual 3d; Full AttnRes with the two-phase schedule (S + N)d;
    Block AttnRes (N/S + 5)d.  L layers, N blocks, S layers per block.
    """
    if kind == "standard":
        return 3.0
    if kind == "full_two_phase":
        return float(S + N)
    if kind == "block":
        return N / S + 5.0
    raise ValueError(kind)


def prefill_block_cache_bytes(tokens: int, blocks: int, D: int, elt: int = BF16,
                              shards: int = 1) -> float:
    """N*T*d elements of cached block summaries, optionally sharded by token rows."""
    return tokens * blocks * D * elt / shards
