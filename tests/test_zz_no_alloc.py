"""The allocation-free backward entry point against the workspace one.

attnres_depth_aggregate_backward_noalloc serves callers that may not allocate
device memory themselves (their device memory is all owned by a pool of
their own, or their loop may not stall on cudaMalloc / cudaFree).  It keeps
its partial sums in a fixed array inside the library instead of a
caller-given workspace.  This file checks, through the C ABI, that its
gradients agree with attnres_depth_aggregate_backward's on several calls in
a row -- different shapes and inputs, so a stale partial row left in the
shared array by one call would show in the next.  It is collected last, so
a run that stops at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

from transformer_depth_wise_gb300 import _lib, api
from transformer_depth_wise_gb300 import workloads as wk

# The bounds of the backward parity tests: source gradients one rounding of
# the dtype (fp32 2e-5, bf16 8e-3 of max|g|), query / gain gradients 2e-4 of
# max|g| (fp32 sums over many rows in a different order).
GRAD_TOL = {torch.float32: 2e-5, torch.bfloat16: 8e-3}
GRAD_SUM_TOL = 2e-4


def _noalloc(srcs, query, gain, eps, dh, grads, gq, gg, accumulate=False):
    B, T, D = srcs[0].shape
    code = 1 if srcs[0].dtype == torch.bfloat16 else 0
    rc = _lib.lib().attnres_depth_aggregate_backward_noalloc(
        _lib.ptr_array([s.data_ptr() for s in srcs]), len(srcs), B, T, D, code, query.data_ptr(),
        gain.data_ptr(), float(eps), dh.data_ptr(), _lib.ptr_array([g.data_ptr() for g in grads]),
        1 if accumulate else 0, None if gq is None else gq.data_ptr(), gg.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    _lib.check("attnres_depth_aggregate_backward_noalloc", rc)


def _close(got, want, rel, what):
    err = float((got.double() - want.double()).abs().max())
    bound = rel * float(want.double().abs().max())
    assert err <= bound, f"{what}: max |err| {err:.3e} > {bound:.3e}"


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward(gpu):
    # The D = 8192 case with 400 rows (more than two per SM) has its grid
    # limited by the scratch: floor(2^21 / 8192) = 256 partial rows, fewer
    # than the resident CTAs, so the reduction runs over all 256 of them.
    # The last case asks for the gain gradient alone.
    cases = [(torch.bfloat16, 2048, 10, 300, 1, False, True), (torch.float32, 256, 5, 777, 2, False, True),
             (torch.bfloat16, 2048, 10, 300, 3, True, True), (torch.bfloat16, 8192, 3, 40, 4, False, True),
             (torch.bfloat16, 8192, 4, 400, 5, False, True), (torch.bfloat16, 1024, 6, 333, 6, False, False)]
    for dtype, D, n, rows, seed, accumulate, want_query in cases:
        g = wk.generator(5000 + seed, gpu)
        srcs, _ = wk.scaled_normal_sources(g, n, (1, rows, D), 0.5, 8.0, dtype, gpu)
        W, G = wk.queries_and_gains(g, 1, D, gpu)
        dh = wk.upstream_grad(g, (1, rows, D), dtype, gpu)
        prior = [wk.upstream_grad(g, (1, rows, D), dtype, gpu) for _ in range(n)]
        want, wq, wg = api.depth_aggregate_backward(srcs, W[0], G[0], 1e-8, dh,
                                                    grad_sources=[p.clone() for p in prior] if accumulate
                                                    else None, accumulate=accumulate)
        grads = [p.clone() for p in prior]
        gq = torch.full((D,), float("nan"), device=gpu) if want_query else None
        gg = torch.full((D,), float("nan"), device=gpu)
        _noalloc(srcs, W[0], G[0], 1e-8, dh, grads, gq, gg, accumulate)
        torch.cuda.synchronize()
        scale = max(float(w.abs().max()) for w in want)
        for got, ref in zip(grads, want):
            err = float((got.double() - ref.double()).abs().max())
            assert err <= GRAD_TOL[dtype] * scale, f"grad sources {dtype} D={D}: {err:.3e}"
        if want_query:
            _close(gq, wq, GRAD_SUM_TOL, f"grad query {dtype} D={D}")
        _close(gg, wg, GRAD_SUM_TOL, f"grad gain {dtype} D={D}")
