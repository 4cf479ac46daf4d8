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


def block_merge_update(inter_out, inter_lse, partial_in, sub_out, u, query, gain=None,
                       eps: float = 1e-8, partial_out=None, h_out=None, out_lse=None):
    """Fused partial update (p = p_in + f(sub_out) or p_in + sub_out) and phase-2 merge.

    Returns (partial_out, h_out).
    """
    _cuda(inter_out, "inter_out")
    _cuda(sub_out, "sub_out")
    B, T, D = _btd(inter_out)
    if partial_out is None:
        partial_out = torch.empty_like(inter_out)
    if h_out is None:
        h_out = torch.empty_like(inter_out)
    rc = _lib.lib().attnres_block_merge_update(inter_out.data_ptr(), inter_lse.data_ptr(),
                                               _ptr(partial_in), sub_out.data_ptr(), _ptr(u), B, T, D,
                                               _code(inter_out), _ptr(query), _ptr(gain), float(eps),
                                               partial_out.data_ptr(), h_out.data_ptr(), _ptr(out_lse),
                                               _stream(h_out))
    _lib.check("attnres_block_merge_update", rc)
    return partial_out, h_out


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
    """

    def __init__(self, blocks, queries, gains, u, eps: float = 1e-8, keep_h: bool = False,
                 fused: bool = True):
        self.blocks = list(blocks)
        self.queries, self.gains, self.u, self.eps = queries, gains, u, float(eps)
        S = queries.shape[0]
        ref = self.blocks[0]
        self.o = torch.empty((S, *ref.shape), dtype=ref.dtype, device=ref.device)
        self.lse = torch.empty((S, *ref.shape[:-1]), dtype=torch.float32, device=ref.device)
        self.partial = torch.empty_like(ref)
        self.h = (torch.empty((S, *ref.shape), dtype=ref.dtype, device=ref.device) if keep_h
                  else torch.empty_like(ref))
        self.keep_h = keep_h
        self.fused = fused
        self._arr = _lib.ptr_array([b.data_ptr() for b in self.blocks])
        self.B, self.T, self.D = _btd(ref)
        self.code = _code(ref)
        self.S = S
        self.launches_per_run = (1 + (S - 1) + 1) if fused else (1 + (S - 1) + S)

    def _hptr(self, k: int) -> int:
        """Device address of h_k (0-based k); h_0 is the phase-1 output o_0."""
        if k == 0 and not self.keep_h:
            return self.o.data_ptr()
        return (self.h[k] if self.keep_h else self.h).data_ptr()

    def run(self, stream=None, events=None):
        L = _lib.lib()
        st = stream if stream is not None else torch.cuda.current_stream(self.o.device).cuda_stream
        B, T, D, code, eps = self.B, self.T, self.D, self.code, self.eps
        D4 = self.D * 4
        qp, gp, up = self.queries.data_ptr(), _ptr(self.gains), self.u.data_ptr()
        row_bytes = self.o[0].numel() * self.o.element_size()
        rows = B * T
        rec = (lambda name, k, i: events[name][k][i].record()) if events else (lambda *a: None)
        if events:
            events["phase1"][0].record()
        _lib.check("attnres_block_phase1",
                   L.attnres_block_phase1(self._arr, len(self.blocks), B, T, D, code, qp, gp, self.S, eps,
                                          self.o.data_ptr(), None, self.lse.data_ptr(), st))
        if events:
            events["phase1"][1].record()
        op, lp, pp = self.o.data_ptr(), self.lse.data_ptr(), self.partial.data_ptr()
        if self.keep_h:
            self.h[0].copy_(self.o[0])
        gk = (lambda k: None) if gp is None else (lambda k: gp + k * D4)
        if self.fused:
            for k in range(1, self.S):
                rec("merge", k - 1, 0)
                _lib.check("attnres_block_merge_update",
                           L.attnres_block_merge_update(op + k * row_bytes, lp + k * rows * 4,
                                                        None if k == 1 else pp, self._hptr(k - 1),
                                                        up + (k - 1) * D4, B, T, D, code, qp + k * D4,
                                                        gk(k), eps, pp, self._hptr(k), None, st))
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
                rec("merge", k - 1, 1)
            rec("update", k, 0)
            _lib.check("attnres_partial_update",
                       L.attnres_partial_update(self._hptr(k), None if k == 0 else pp, up + k * D4, B, T, D,
                                                code, pp, st))
            rec("update", k, 1)
        return self.partial


def block_two_phase(blocks, queries, gains, u, eps: float = 1e-8, fused: bool = True):
    """Run one block of the two-phase scheme; returns (final partial, [h_1..h_S])."""
    blk = TwoPhaseBlock(blocks, queries, gains, u, eps, keep_h=True, fused=fused)
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
