"""Seeded synthetic inputs for the Attention Residuals workloads.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle can be fed
the same bytes from it.  Every tensor is drawn in a fixed order from one
``torch.Generator`` seeded per workload, then cast once to its storage
dtype.  The recipes (sizes, value distributions) are the five benchmark
workloads of the depth-aggregation problem:

* ``full_single_f32``   n=5 sources [1,64,256] fp32, source i = s_i*N(0,1),
  s_i ~ U(0.5, 4); query ~ N(0, 0.02^2); gain ~ N(1, 0.1^2); eps = 1e-8.
* ``block_single_bf16`` n=10 sources [4,4096,2048] bf16, s_i ~ U(0.5, 8).
* ``two_phase_bf16``    S=24 queries [24,4096], 9 cached block summaries
  [8,4096,4096] bf16 (s_i ~ U(0.5, 8)), u_k ~ N(1, 0.25^2) per feature.
* ``full_stack_bf16``   v0 ~ N(0,1) [1,2048,2048] bf16, 186 sublayers, each with
  query, gain and u, plus a final query and gain.
* ``long_prefill_bf16`` / ``decode_bf16``  D=7168, n=10 sources, S=24:
  B=1,T=65536 and B=256,T=1.

``scale_rows`` shrinks the token axis for tests that must stay small while
keeping every other size of the recipe.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

EPS = 1e-8


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    D: int
    n: int                      # sources in one aggregation / cached summaries
    dtype: torch.dtype
    scale_lo: float
    scale_hi: float
    S: int = 0                  # queries per block (two-phase)
    L: int = 0                  # sublayers (full stack)
    seed: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "full_single_f32": Workload("full_single_f32", 1, 64, 256, 5, torch.float32, 0.5, 4.0,
                                seed=1001, note="Full AttnRes single aggregation, fp32"),
    "block_single_bf16": Workload("block_single_bf16", 4, 4096, 2048, 10, torch.bfloat16, 0.5, 8.0,
                                  seed=1002, note="Block AttnRes single aggregation, bf16"),
    "two_phase_bf16": Workload("two_phase_bf16", 8, 4096, 4096, 9, torch.bfloat16, 0.5, 8.0, S=24,
                               seed=1003, note="two-phase Block AttnRes, bf16, S=24, 9 summaries"),
    "full_stack_bf16": Workload("full_stack_bf16", 1, 2048, 2048, 1, torch.bfloat16, 1.0, 1.0,
                                L=186, seed=1004, note="Full AttnRes 186-sublayer forward, bf16"),
    "long_prefill_bf16": Workload("long_prefill_bf16", 1, 65536, 7168, 10, torch.bfloat16, 0.5, 8.0,
                                  S=24, seed=1005, note="Block AttnRes long prefill, D=7168"),
    "decode_bf16": Workload("decode_bf16", 256, 1, 7168, 10, torch.bfloat16, 0.5, 8.0, S=24,
                            seed=1006, note="Block AttnRes decode, D=7168"),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def scaled_normal_sources(g: torch.Generator, n: int, shape, lo: float, hi: float, dtype,
                          device="cpu"):
    """n tensors, source i = s_i * N(0,1) with s_i ~ U(lo, hi), cast to dtype.

    Returns (list of tensors, scales tensor [n] fp64 on CPU).
    """
    scales = torch.empty(n, dtype=torch.float64, device=device).uniform_(lo, hi, generator=g)
    out = []
    for i in range(n):
        z = torch.empty(shape, dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=g)
        out.append((z * float(scales[i])).to(dtype))
    return out, scales.cpu()


def queries_and_gains(g: torch.Generator, count: int, D: int, device="cpu", zero_query=False):
    """count query rows ~ N(0, 0.02^2) and gain rows ~ N(1, 0.1^2), fp32 [count, D]."""
    w = torch.empty((count, D), dtype=torch.float32, device=device).normal_(0.0, 0.02, generator=g)
    gam = torch.empty((count, D), dtype=torch.float32, device=device).normal_(1.0, 0.1, generator=g)
    if zero_query:
        w.zero_()
    return w, gam


def sublayer_u(g: torch.Generator, count: int, D: int, device="cpu"):
    """u rows ~ N(1, 0.25^2), fp32 [count, D] (synthetic sublayer f(h) = 0.5 tanh(u*h))."""
    return torch.empty((count, D), dtype=torch.float32, device=device).normal_(1.0, 0.25, generator=g)


def upstream_grad(g: torch.Generator, shape, dtype, device) -> torch.Tensor:
    """The gradient arriving at an aggregation's output in a backward pass: N(0, 1)."""
    return torch.empty(shape, dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=g).to(dtype)


def single_aggregation_inputs(wl: Workload, rows: int | None = None, device="cpu",
                              zero_query=False, n: int | None = None):
    """Inputs of one depth aggregation: dict(sources, query [D], gain [D], eps)."""
    B, T = (wl.B, wl.T) if rows is None else (1, rows)
    n = wl.n if n is None else n
    g = generator(wl.seed + (0 if rows is None else 7919 * rows), device)
    srcs, scales = scaled_normal_sources(g, n, (B, T, wl.D), wl.scale_lo, wl.scale_hi, wl.dtype,
                                         device)
    w, gam = queries_and_gains(g, 1, wl.D, device, zero_query)
    return {"sources": srcs, "query": w[0].contiguous(), "gain": gam[0].contiguous(), "eps": EPS,
            "scales": scales}


def two_phase_inputs(wl: Workload, rows: int | None = None, device="cpu", S: int | None = None,
                     n: int | None = None):
    """Inputs of one block of the two-phase scheme: n summaries, S queries/gains/u."""
    B, T = (wl.B, wl.T) if rows is None else (1, rows)
    S = wl.S if S is None else S
    n = (wl.n if wl.name == "two_phase_bf16" else wl.n - 1) if n is None else n
    g = generator(wl.seed + 17 + (0 if rows is None else 7919 * rows), device)
    blocks, scales = scaled_normal_sources(g, n, (B, T, wl.D), wl.scale_lo, wl.scale_hi,
                                           wl.dtype, device)
    w, gam = queries_and_gains(g, S, wl.D, device)
    u = sublayer_u(g, S, wl.D, device)
    return {"blocks": blocks, "queries": w, "gains": gam, "u": u, "eps": EPS, "scales": scales}


def full_stack_inputs(wl: Workload, rows: int | None = None, device="cpu", L: int | None = None,
                      D: int | None = None):
    """Inputs of the Full stack: v0 [B,T,D], queries/gains [L+1, D], u [L, D]."""
    B, T = (wl.B, wl.T) if rows is None else (1, rows)
    L = wl.L if L is None else L
    D = wl.D if D is None else D
    g = generator(wl.seed + 31 + (0 if rows is None else 7919 * rows), device)
    v0 = torch.empty((B, T, D), dtype=torch.float32, device=device).normal_(0.0, 1.0, generator=g)
    v0 = v0.to(wl.dtype)
    w, gam = queries_and_gains(g, L + 1, D, device)
    u = sublayer_u(g, L, D, device)
    return {"v0": v0, "queries": w, "gains": gam, "u": u, "eps": EPS}
