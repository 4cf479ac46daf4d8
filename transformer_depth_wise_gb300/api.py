"""PyTorch-facing wrappers of the C ABI (include/attnres.h).

PyTorch supplies device memory and the current CUDA stream; every step of
the computation runs in libattnres.so's kernels.  The wrappers only check
that tensors are CUDA, contiguous and of one dtype, allocate outputs the
caller did not pass, and marshal pointers.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

_CODES = {torch.float32: _lib.ATTNRES_F32, torch.bfloat16: _lib.ATTNRES_BF16}


def _code(t: torch.Tensor) -> int:
    try:
        return _CODES[t.dtype]
    except KeyError:
        raise TypeError(f"dtype {t.dtype} is not supported (float32 or bfloat16)") from None


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _f32(t: torch.Tensor | None, name: str):
    if t is None:
        return None
    _cuda(t, name)
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return t


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _btd(t: torch.Tensor):
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2]
    if t.dim() == 2:
        return 1, t.shape[0], t.shape[1]
    raise ValueError("expected a [B, T, D] (or [rows, D]) tensor")


def depth_aggregate(sources, query, gain=None, eps: float = 1e-8, out=None, stats: bool = False):
    """h = sum_i softmax_i(w~ . RMS(v_i)) v_i over the listed sources (eq. A1-A3).

    Returns out, or (out, m, lse) when stats=True.
    """
    srcs = [_cuda(s, "sources[i]") for s in sources]
    if not srcs:
        raise ValueError("at least one source is required")
    B, T, D = _btd(srcs[0])
    for s in srcs:
        if s.shape != srcs[0].shape or s.dtype != srcs[0].dtype:
            raise ValueError("all sources must share shape and dtype")
    _f32(query, "query")
    _f32(gain, "gain")
    if out is None:
        out = torch.empty_like(srcs[0])
    _cuda(out, "out")
    m = lse = None
    if stats:
        m = torch.empty(srcs[0].shape[:-1], dtype=torch.float32, device=srcs[0].device)
        lse = torch.empty_like(m)
    arr = _lib.ptr_array([s.data_ptr() for s in srcs])
    rc = _lib.lib().attnres_depth_aggregate(arr, len(srcs), B, T, D, _code(srcs[0]), _ptr(query),
                                            _ptr(gain), float(eps), out.data_ptr(), _ptr(m),
                                            _ptr(lse), _stream(out))
    _lib.check("attnres_depth_aggregate", rc)
    return (out, m, lse) if stats else out


def depth_aggregate_backward_workspace_rows(D: int, dtype) -> int:
    """Rows of the fp32 [rows, D] workspace that let the backward fill the current GPU."""
    code = 1 if dtype == torch.bfloat16 else 0
    r = int(_lib.lib().attnres_depth_aggregate_backward_workspace_rows(int(D), code))
    if r < 0:
        _lib.check("attnres_depth_aggregate_backward_workspace_rows", r)
    return r


def depth_aggregate_backward(sources, query, gain, eps: float, grad_out, grad_sources=None,
                             accumulate: bool = False, want_query: bool = True, want_gain: bool = True,
                             workspace=None):
    """Gradients of h = depth_aggregate(sources, query, gain, eps) for the upstream dh = grad_out.

    Returns (grad_sources list, grad_query [D] fp32 or None, grad_gain [D] fp32 or None).
    accumulate=True adds into the given grad_sources.  workspace: fp32 [rows, D]
    (allocated here when None and a parameter gradient is wanted).
    """
    srcs = [_cuda(s, "sources[i]") for s in sources]
    B, T, D = _btd(srcs[0])
    _cuda(grad_out, "grad_out")
    dev = srcs[0].device
    if grad_sources is None:
        if accumulate:
            raise ValueError("accumulate=True needs grad_sources")
        grad_sources = [torch.empty_like(s) for s in srcs]
    gq = torch.empty(D, dtype=torch.float32, device=dev) if want_query else None
    gg = torch.empty(D, dtype=torch.float32, device=dev) if want_gain else None
    if (want_query or want_gain) and workspace is None:
        rows = depth_aggregate_backward_workspace_rows(D, srcs[0].dtype)
        workspace = torch.empty((rows, D), dtype=torch.float32, device=dev)
    arr = _lib.ptr_array([s.data_ptr() for s in srcs])
    garr = _lib.ptr_array([g.data_ptr() for g in grad_sources])
    rc = _lib.lib().attnres_depth_aggregate_backward(
        arr, len(srcs), B, T, D, _code(srcs[0]), _ptr(query), _ptr(gain), float(eps), grad_out.data_ptr(),
        garr, 1 if accumulate else 0, _ptr(gq), _ptr(gg), _ptr(workspace),
        0 if workspace is None else workspace.shape[0], _stream(grad_out))
    _lib.check("attnres_depth_aggregate_backward", rc)
    return grad_sources, gq, gg


def block_phase1(blocks, queries, gains=None, eps: float = 1e-8, out=None, out_max=None,
                 out_lse=None, want_max: bool = False):
    """Phase 1: S queries [S, D] over n summaries; returns (o [S,B,T,D], m or None, lse [S,B,T])."""
    blks = [_cuda(b, "blocks[i]") for b in blocks]
    B, T, D = _btd(blks[0])
    _f32(queries, "queries")
    _f32(gains, "gains")
    S = queries.shape[0]
    dev = blks[0].device
    if out is None:
        out = torch.empty((S, *blks[0].shape), dtype=blks[0].dtype, device=dev)
    if out_lse is None:
        out_lse = torch.empty((S, *blks[0].shape[:-1]), dtype=torch.float32, device=dev)
    if out_max is None and want_max:
        out_max = torch.empty_like(out_lse)
    arr = _lib.ptr_array([b.data_ptr() for b in blks])
    rc = _lib.lib().attnres_block_phase1(arr, len(blks), B, T, D, _code(blks[0]), _ptr(queries),
                                         _ptr(gains), S, float(eps), out.data_ptr(), _ptr(out_max),
                                         out_lse.data_ptr(), _stream(out))
    _lib.check("attnres_block_phase1", rc)
    return out, out_max, out_lse


def block_phase2_merge(inter_out, inter_lse, partial, query, gain=None, eps: float = 1e-8,
                       h_out=None, out_lse=None):
    """Phase 2: merge the running partial into one query's phase-1 state (eq. OS2)."""
    _cuda(inter_out, "inter_out")
    _f32(inter_lse, "inter_lse")
    if partial is not None:
        _cuda(partial, "partial")
    B, T, D = _btd(inter_out)
    if h_out is None:
        h_out = torch.empty_like(inter_out)
    rc = _lib.lib().attnres_block_phase2_merge(inter_out.data_ptr(), inter_lse.data_ptr(),
                                               _ptr(partial), B, T, D, _code(inter_out),
                                               _ptr(query), _ptr(gain), float(eps),
                                               h_out.data_ptr(), _ptr(out_lse), _stream(h_out))
    _lib.check("attnres_block_phase2_merge", rc)
    return h_out


def partial_update(h, partial_in, u, out=None):
    """partial_out = partial_in + 0.5 tanh(u (.) h)  (partial_in None: no addend)."""
    _cuda(h, "h")
    B, T, D = _btd(h)
    if out is None:
        out = torch.empty_like(h)
    rc = _lib.lib().attnres_partial_update(h.data_ptr(), _ptr(partial_in), _ptr(u), B, T, D,
                                           _code(h), out.data_ptr(), _stream(out))
    _lib.check("attnres_partial_update", rc)
    return out


def full_stack_forward(v0, queries, gains, u, eps: float = 1e-8, sources=None, y=None):
    """Full AttnRes stack with the synthetic sublayer; returns (y, [v_0..v_L])."""
    _cuda(v0, "v0")
    B, T, D = _btd(v0)
    L = u.shape[0]
    if sources is None:
        sources = [v0] + [torch.empty_like(v0) for _ in range(L)]
    if y is None:
        y = torch.empty_like(v0)
    arr = _lib.ptr_array([s.data_ptr() for s in sources])
    rc = _lib.lib().attnres_full_stack_forward(arr, L, B, T, D, _code(v0), _ptr(queries),
                                               _ptr(gains), _ptr(u), float(eps), y.data_ptr(),
                                               _stream(y))
    _lib.check("attnres_full_stack_forward", rc)
    return y, sources


def full_stack_two_phase(v0, queries, gains, u, S: int, eps: float = 1e-8, sources=None, y=None,
                         workspace=None):
    """The Full stack with the two-phase schedule of block size S; returns (y, [v_0..v_L]).

    Same arguments as full_stack_forward (sources [L+1] with v_0 given,
    v_1..v_L written); workspace is a uint8 CUDA tensor of the size
    attnres_full_stack_two_phase_workspace_bytes reports (allocated when None).
    """
    _cuda(v0, "v0")
    B, T, D = _btd(v0)
    L = u.shape[0]
    if sources is None:
        sources = [v0] + [torch.empty_like(v0) for _ in range(L)]
    if y is None:
        y = torch.empty_like(v0)
    L_lib = _lib.lib()
    need = int(L_lib.attnres_full_stack_two_phase_workspace_bytes(L, int(S), B, T, D, _code(v0)))
    if need < 0:
        _lib.check("attnres_full_stack_two_phase_workspace_bytes", need)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=v0.device)
    arr = _lib.ptr_array([s.data_ptr() for s in sources])
    rc = L_lib.attnres_full_stack_two_phase(arr, L, int(S), B, T, D, _code(v0), _ptr(queries), _ptr(gains),
                                            _ptr(u), float(eps), y.data_ptr(), workspace.data_ptr(),
                                            workspace.numel(), _stream(y))
    _lib.check("attnres_full_stack_two_phase", rc)
    return y, sources


class FullStack:
    """A whole Full AttnRes stack over preallocated buffers, as one call or as
    one CUDA graph.  S = None runs the plain stack (attnres_full_stack_forward),
    an integer S the two-phase schedule of block size S (with its workspace).
    run() launches it eagerly; capture() records one run as a CUDA graph (after
    one eager run, which settles the library's per-kernel launch settings) and
    replay() launches the graph: the same kernels on the same buffers, so the
    results are bitwise those of run()."""

    def __init__(self, v0, queries, gains, u, eps: float = 1e-8, S=None):
        _cuda(v0, "v0")
        self.v0, self.queries, self.gains, self.u, self.eps, self.S = v0, queries, gains, u, float(eps), S
        L = u.shape[0]
        self.sources = [v0] + [torch.empty_like(v0) for _ in range(L)]
        self.y = torch.empty_like(v0)
        self.workspace = None
        if S is not None:
            B, T, D = _btd(v0)
            need = int(_lib.lib().attnres_full_stack_two_phase_workspace_bytes(L, int(S), B, T, D, _code(v0)))
            if need < 0:
                _lib.check("attnres_full_stack_two_phase_workspace_bytes", need)
            self.workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=v0.device)
        self.graph = None

    def run(self):
        if self.S is None:
            full_stack_forward(self.v0, self.queries, self.gains, self.u, self.eps, self.sources, self.y)
        else:
            full_stack_two_phase(self.v0, self.queries, self.gains, self.u, self.S, self.eps, self.sources, self.y,
                                 self.workspace)
        return self.y

    def capture(self):
        self.run()
        torch.cuda.synchronize(self.v0.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
        return self.y


def block_merge_update(inter_out, inter_lse, partial_in, sub_out, u, query, gain=None,
                       eps: float = 1e-8, partial_out=None, h_out=None, out_lse=None,
                       norm_weight=None, norm_eps: float = 1e-6, normed_out=None, write_h: bool = True):
    """Fused partial update (p = p_in + f(sub_out) or p_in + sub_out) and phase-2 merge.

    With norm_weight, also the next sublayer's pre-norm of the unrounded h:
    normed_out = rms_norm(h) (.) norm_weight.  write_h=False skips storing h.
    Returns (partial_out, h_out, normed_out); h_out / normed_out are None when
    not written.
    """
    _cuda(inter_out, "inter_out")
    _cuda(sub_out, "sub_out")
    B, T, D = _btd(inter_out)
    if partial_out is None:
        partial_out = torch.empty_like(inter_out)
    if h_out is None and write_h:
        h_out = torch.empty_like(inter_out)
    if norm_weight is not None and normed_out is None:
        normed_out = torch.empty_like(inter_out)
    rc = _lib.lib().attnres_block_merge_update(inter_out.data_ptr(), inter_lse.data_ptr(),
                                               _ptr(partial_in), sub_out.data_ptr(), _ptr(u), B, T, D,
                                               _code(inter_out), _ptr(query), _ptr(gain), float(eps),
                                               partial_out.data_ptr(), _ptr(h_out if write_h else None),
                                               _ptr(out_lse), _ptr(norm_weight), float(norm_eps),
                                               _ptr(normed_out), _stream(partial_out))
    _lib.check("attnres_block_merge_update", rc)
    return partial_out, (h_out if write_h else None), normed_out


def rms_norm(x, weight, eps: float = 1e-6, out=None):
    """y = x / sqrt(mean(x^2) + eps) (.) weight per token row (out may be x)."""
    _cuda(x, "x")
    B, T, D = _btd(x)
    if out is None:
        out = torch.empty_like(x)
    rc = _lib.lib().attnres_rms_norm(x.data_ptr(), B, T, D, _code(x), _ptr(weight), float(eps),
                                     out.data_ptr(), _stream(out))
    _lib.check("attnres_rms_norm", rc)
    return out


class TwoPhaseBlock:
    """One block of the two-phase Block scheme over preallocated buffers.

    run() computes phase 1 over the cached summaries for the block's S
    queries, then walks the S sublayers: h_1 is the phase-1 output itself,
    h_k (k >= 2) merges the running partial into the phase-1 state, and
    after each sublayer the partial grows by f_k(h_k) (synthetic sublayer).
    The final partial (the block's summary b_n) is returned.

    fused=False: 23 merges + 24 partial updates (attnres_block_phase2_merge,
    attnres_partial_update).  fused=True: 23 fused update+merge steps
    (attnres_block_merge_update) + 1 final update.  Both give the same values.

    norm_weights ([S, D] fp32 or None): each sublayer reads its pre-norm
    y_k = rms_norm(h_k) (.) norm_weights[k] instead of h_k.  Fused, the norm
    is formed inside the update+merge step from the unrounded h_k (the first
    sublayer's by attnres_rms_norm); unfused, by attnres_rms_norm after each
    merge.  The stored sublayer inputs are then the y_k.

    overlap=True (decode): the batched inter-block pass for sublayers 2..S
    runs on a side stream while the main stream forms sublayer 1's input by
    a direct aggregation over the summaries (the only phase-1 result the
    first sublayer needs); the main stream joins the side stream before the
    first merge.  capture() records the whole pass as one CUDA graph and
    replay() launches it.

    groups=G > 1 (G divides B): the batch's sequences are split into G groups,
    each a block pass of its own over its rows, on G streams forked from the
    current stream and joined back; the returned partial holds every group's
    rows.  Rows never mix in any step of the pass, so the values are those of
    one pass over the whole batch (bitwise where both take the same kernels:
    a group of fewer than 76 x 128 rows splits its phase-1 scores over
    feature slices, one of at most four rows per SM takes the few-rows
    update+merge kernel, each with its own reduction order), and the groups'
    kernels overlap
    (one group's phase-1 scores beside another's outputs).  Per-kernel events
    and overlap=True need groups=1.

    partial ([B,T,D] of the sources' dtype, or None): where the final partial
    is written (allocated when None).
    """

    def __init__(self, blocks, queries, gains, u, eps: float = 1e-8, keep_h: bool = False,
                 fused: bool = True, norm_weights=None, norm_eps: float = 1e-6, overlap: bool = False,
                 groups: int = 1, partial=None):
        self.blocks = list(blocks)
        self.queries, self.gains, self.u, self.eps = queries, gains, u, float(eps)
        self.nw, self.norm_eps = norm_weights, float(norm_eps)
        self.overlap = overlap
        self.graph = None
        self.groups = int(groups)
        ref = self.blocks[0]
        self.device = ref.device
        if partial is not None and (partial.shape != ref.shape or partial.dtype != ref.dtype
                                    or partial.device != ref.device or not partial.is_contiguous()):
            raise ValueError("partial must be a contiguous tensor of the summaries' shape, dtype and device")
        if self.groups > 1:
            if overlap:
                raise ValueError("groups > 1 does not combine with overlap=True")
            Bb = ref.shape[0]
            if Bb % self.groups:
                raise ValueError(f"groups={self.groups} must divide the batch B={Bb}")
            self.partial = torch.empty_like(ref) if partial is None else partial
            bg = Bb // self.groups
            self.parts = [TwoPhaseBlock([b[g * bg:(g + 1) * bg] for b in self.blocks], queries, gains, u, eps,
                                        keep_h=keep_h, fused=fused, norm_weights=norm_weights, norm_eps=norm_eps,
                                        partial=self.partial[g * bg:(g + 1) * bg])
                          for g in range(self.groups)]
            self.streams = [torch.cuda.Stream(device=self.device) for _ in range(self.groups)]
            self.ev_fork = torch.cuda.Event()
            self.ev_parts = [torch.cuda.Event() for _ in range(self.groups)]
            self.S = queries.shape[0]
            self.B, self.T, self.D = _btd(ref)
            self.launches_per_run = sum(p.launches_per_run for p in self.parts)
            return
        if overlap:
            if not fused or norm_weights is not None:
                raise ValueError("overlap=True runs the fused pass without a pre-norm")
            self.side = torch.cuda.Stream(device=blocks[0].device)
            self.ev_fork, self.ev_join = torch.cuda.Event(), torch.cuda.Event()
        S = queries.shape[0]
        self.o = torch.empty((S, *ref.shape), dtype=ref.dtype, device=ref.device)
        self.lse = torch.empty((S, *ref.shape[:-1]), dtype=torch.float32, device=ref.device)
        self.partial = torch.empty_like(ref) if partial is None else partial
        self.h = (torch.empty((S, *ref.shape), dtype=ref.dtype, device=ref.device) if keep_h
                  else torch.empty_like(ref))
        self.keep_h = keep_h
        self.fused = fused
        self._arr = _lib.ptr_array([b.data_ptr() for b in self.blocks])
        self.B, self.T, self.D = _btd(ref)
        self.code = _code(ref)
        self.S = S
        self.launches_per_run = (1 + (S - 1) + 1) if fused else (1 + (S - 1) + S)
        if norm_weights is not None:
            self.launches_per_run += 1 if fused else S
        if overlap:
            self.launches_per_run += 1

    def _hptr(self, k: int) -> int:
        """Device address of sublayer k's input (0-based k); without a pre-norm
        h_0 is the phase-1 output o_0 itself."""
        if k == 0 and not self.keep_h and self.nw is None and not self.overlap:
            return self.o.data_ptr()
        return (self.h[k] if self.keep_h else self.h).data_ptr()

    def run(self, stream=None, events=None):
        if self.groups > 1:
            return self._run_groups(stream, events)
        L = _lib.lib()
        st = stream if stream is not None else torch.cuda.current_stream(self.o.device).cuda_stream
        B, T, D, code, eps = self.B, self.T, self.D, self.code, self.eps
        D4 = self.D * 4
        qp, gp, up = self.queries.data_ptr(), _ptr(self.gains), self.u.data_ptr()
        row_bytes = self.o[0].numel() * self.o.element_size()
        rows = B * T
        rec = ((lambda name, k, i: events[name][k][i].record() if name in events else None) if events
               else (lambda *a: None))
        if self.overlap:
            self._overlapped_phase1(L, st)
        else:
            if events:
                events["phase1"][0].record()
            _lib.check("attnres_block_phase1",
                       L.attnres_block_phase1(self._arr, len(self.blocks), B, T, D, code, qp, gp, self.S, eps,
                                              self.o.data_ptr(), None, self.lse.data_ptr(), st))
            if events:
                events["phase1"][1].record()
        op, lp, pp = self.o.data_ptr(), self.lse.data_ptr(), self.partial.data_ptr()
        nwp, neps = _ptr(self.nw), self.norm_eps
        if self.nw is not None:
            # first sublayer: y_1 = rms_norm(o_1), its pre-norm as a pass of its own
            rec("norm", 0, 0)
            _lib.check("attnres_rms_norm", L.attnres_rms_norm(op, B, T, D, code, nwp, neps, self._hptr(0), st))
            rec("norm", 0, 1)
        elif self.keep_h and not self.overlap:
            self.h[0].copy_(self.o[0])
        gk = (lambda k: None) if gp is None else (lambda k: gp + k * D4)
        if self.fused:
            for k in range(1, self.S):
                rec("merge", k - 1, 0)
                h_dst = self._hptr(k)
                _lib.check("attnres_block_merge_update",
                           L.attnres_block_merge_update(op + k * row_bytes, lp + k * rows * 4,
                                                        None if k == 1 else pp, self._hptr(k - 1),
                                                        up + (k - 1) * D4, B, T, D, code, qp + k * D4,
                                                        gk(k), eps, pp,
                                                        None if nwp else h_dst, None,
                                                        (nwp + k * D4) if nwp else None, neps,
                                                        h_dst if nwp else None, st))
                rec("merge", k - 1, 1)
            rec("update", 0, 0)
            _lib.check("attnres_partial_update",
                       L.attnres_partial_update(self._hptr(self.S - 1), pp if self.S > 1 else None,
                                                up + (self.S - 1) * D4, B, T, D, code, pp, st))
            rec("update", 0, 1)
            return self.partial
        for k in range(self.S):
            if k > 0:
                rec("merge", k - 1, 0)
                _lib.check("attnres_block_phase2_merge",
                           L.attnres_block_phase2_merge(op + k * row_bytes, lp + k * rows * 4, pp, B, T, D,
                                                        code, qp + k * D4, gk(k), eps, self._hptr(k), None,
                                                        st))
                if nwp:
                    _lib.check("attnres_rms_norm",
                               L.attnres_rms_norm(self._hptr(k), B, T, D, code, nwp + k * D4, neps,
                                                  self._hptr(k), st))
                rec("merge", k - 1, 1)
            rec("update", k, 0)
            _lib.check("attnres_partial_update",
                       L.attnres_partial_update(self._hptr(k), None if k == 0 else pp, up + k * D4, B, T, D,
                                                code, pp, st))
            rec("update", k, 1)
        return self.partial


    def _overlapped_phase1(self, L, st):
        """Side stream: phase 1 for queries 2..S.  Main stream: sublayer 1's
        input by a direct aggregation over the summaries; then join."""
        main = torch.cuda.current_stream(self.o.device)
        if st != main.cuda_stream:
            raise ValueError("overlap=True runs on the current stream")
        B, T, D, code, eps, S = self.B, self.T, self.D, self.code, self.eps, self.S
        D4, row_bytes, rows = D * 4, self.o[0].numel() * self.o.element_size(), B * T
        qp, gp = self.queries.data_ptr(), _ptr(self.gains)
        self.ev_fork.record(main)
        self.side.wait_event(self.ev_fork)
        if S > 1:
            _lib.check("attnres_block_phase1",
                       L.attnres_block_phase1(self._arr, len(self.blocks), B, T, D, code, qp + D4,
                                              None if gp is None else gp + D4, S - 1, eps,
                                              self.o.data_ptr() + row_bytes, None,
                                              self.lse.data_ptr() + rows * 4, self.side.cuda_stream))
        self.ev_join.record(self.side)
        _lib.check("attnres_depth_aggregate",
                   L.attnres_depth_aggregate(self._arr, len(self.blocks), B, T, D, code, qp, gp, eps,
                                             self._hptr(0), None, None, st))
        main.wait_event(self.ev_join)

    def _run_groups(self, stream, events):
        """Each group's pass on a stream of its own, forked from the current
        stream and joined back before return."""
        if events:
            raise ValueError("per-kernel events need groups=1")
        main = torch.cuda.current_stream(self.device)
        if stream is not None and stream != main.cuda_stream:
            raise ValueError("groups > 1 runs on the current stream")
        self.ev_fork.record(main)
        for s, p, e in zip(self.streams, self.parts, self.ev_parts):
            s.wait_event(self.ev_fork)
            with torch.cuda.stream(s):
                p.run()
            e.record(s)
        for e in self.ev_parts:
            main.wait_event(e)
        return self.partial

    def capture(self):
        """Record one whole block pass as a CUDA graph (after one eager pass,
        which settles the library's per-kernel launch settings)."""
        self.run()
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run()
        self.graph = g
        return g

    def replay(self):
        """Launch the captured block pass on the current stream; returns the final partial."""
        if self.graph is None:
            raise RuntimeError("capture() first")
        self.graph.replay()
        return self.partial


class TwoPhaseStream:
    """Block passes over a stream of host inputs, pipelined across passes.

    submit() copies one pass's summaries, queries, gains and u from (pinned)
    host memory, runs the fused block pass (TwoPhaseBlock.run) and copies its
    final partial back to a host tensor.  Two device buffer sets alternate:
    the host->device copies of pass k+1 run on a copy stream while pass k's
    kernels run on the current stream, and pass k's partial returns on a
    third stream while pass k+1 runs.  Events order every reuse of a set (its
    inputs are overwritten only after the pass that read them, its partial
    only after it has reached the host), so each pass's result is exactly
    TwoPhaseBlock.run()'s on the same inputs.
    """

    def __init__(self, n: int, shape, dtype, S: int, device, eps: float = 1e-8, with_gains: bool = True):
        device = torch.device(device)
        D = shape[-1]
        self.sets = []
        for _ in range(2):
            blocks = [torch.empty(shape, dtype=dtype, device=device) for _ in range(n)]
            q = torch.empty((S, D), dtype=torch.float32, device=device)
            g = torch.empty((S, D), dtype=torch.float32, device=device) if with_gains else None
            u = torch.empty((S, D), dtype=torch.float32, device=device)
            self.sets.append({"blocks": blocks, "queries": q, "gains": g, "u": u,
                              "blk": TwoPhaseBlock(blocks, q, g, u, eps),
                              "copied": torch.cuda.Event(), "done": torch.cuda.Event(),
                              "returned": torch.cuda.Event()})
        self.device = device
        self.copy_stream = torch.cuda.Stream(device=device)
        self.d2h_stream = torch.cuda.Stream(device=device)
        self.k = 0

    def submit(self, host_blocks, host_queries, host_gains, host_u, out_host):
        """Enqueue one pass; returns the event recorded once out_host holds its
        final partial (out_host must not be reused before)."""
        st = self.sets[self.k % 2]
        self.k += 1
        main = torch.cuda.current_stream(self.device)
        self.copy_stream.wait_event(st["done"])            # the set's last pass has read its inputs
        with torch.cuda.stream(self.copy_stream):
            for dst, src in zip(st["blocks"], host_blocks):
                dst.copy_(src, non_blocking=True)
            st["queries"].copy_(host_queries, non_blocking=True)
            if st["gains"] is not None:
                st["gains"].copy_(host_gains, non_blocking=True)
            st["u"].copy_(host_u, non_blocking=True)
        st["copied"].record(self.copy_stream)
        main.wait_event(st["copied"])
        main.wait_event(st["returned"])                      # its last partial is back on the host
        partial = st["blk"].run(stream=main.cuda_stream)
        st["done"].record(main)
        self.d2h_stream.wait_event(st["done"])
        with torch.cuda.stream(self.d2h_stream):
            out_host.copy_(partial, non_blocking=True)
        st["returned"].record(self.d2h_stream)
        return st["returned"]


def block_two_phase(blocks, queries, gains, u, eps: float = 1e-8, fused: bool = True,
                    norm_weights=None, norm_eps: float = 1e-6):
    """Run one block of the two-phase scheme; returns (final partial, sublayer inputs [S, ...])."""
    blk = TwoPhaseBlock(blocks, queries, gains, u, eps, keep_h=True, fused=fused,
                        norm_weights=norm_weights, norm_eps=norm_eps)
    p = blk.run()
    return p, blk.h


def block_schedule(num_atomic: int, block_size: int):
    """forward_naive's source lists (host bookkeeping): num_atomic+1 lists, -1 = partial."""
    cap = (num_atomic + 1) * (num_atomic + 2)
    counts = (ctypes.c_int * (num_atomic + 1))()
    ids = (ctypes.c_int * cap)()
    w = _lib.check("attnres_block_schedule",
                   _lib.lib().attnres_block_schedule(int(num_atomic), int(block_size), counts, ids,
                                                     cap))
    out, k = [], 0
    for c in counts:
        out.append([ids[k + j] for j in range(c)])
        k += c
    assert k == w
    return out


def atomic_block_size(num_hidden_layers: int, attnres_block_size=None) -> int:
    bs = -1 if attnres_block_size is None else int(attnres_block_size)
    return _lib.check("attnres_atomic_block_size",
                      _lib.lib().attnres_atomic_block_size(int(num_hidden_layers), bs))
