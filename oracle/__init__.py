"""fp64 CPU oracle for the Attention Residuals depth aggregation.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg are the only callers.  The CUDA
product path (``transformer_depth_wise_gb300``) never imports this package,
and this package never imports the product.

The arithmetic lives in ``attnres_oracle.c`` (plain single-threaded C, fp64).
This module only builds it, loads it and marshals numpy float64 arrays.
Each wrapper names the passage of the pages it follows:

* "Attention Residual 深度残差" (K3 course notes, sec-09): eq. A1-A4, OS1-OS2,
  listings DepthResidual, forward_naive, _run_block_two_phase,
  atomic_block_size.
* "Attention Residuals：当网络深度也拥有寻址能力": sections "Full AttnRes" and
  "Online softmax 让两阶段计算保持精确".

Parity is pinned for every function here (see tests/test_oracle_pins.py);
none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attnres_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1
F64 = 2  # keep exact values (no rounding)

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_I = ctypes.POINTER(ctypes.c_int)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math: IEEE fp64 semantics)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, c_int, c_dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        PP = ctypes.POINTER(_D)
        sig = {
            "oracle_round_bf16": (c_dbl, [c_dbl]),
            "oracle_round_f32": (c_dbl, [c_dbl]),
            "oracle_round_array": (None, [i64, _D, c_int, _D]),
            "oracle_fold_query": (None, [i64, _D, _D, _D]),
            "oracle_depth_aggregate": (c_int, [c_int, i64, i64, _D, _D, _D, c_dbl, _D, _D, _D]),
            "oracle_depth_aggregate_list": (c_int, [c_int, i64, i64, PP, _D, _D, c_dbl, _D, _D, _D]),
            "oracle_depth_aggregate_backward": (c_int, [c_int, i64, i64, PP, _D, _D, c_dbl, _D, PP,
                                                        _D, _D]),
            "oracle_os1_stats": (None, [c_int, i64, PP, _D, c_dbl, _D, _D, _D]),
            "oracle_single_source_stats": (None, [i64, _D, _D, c_dbl, _D, _D, _D]),
            "oracle_os2_merge": (None, [i64, c_dbl, _D, c_dbl, c_dbl, _D, c_dbl, _D, _D, _D]),
            "oracle_block_phase1": (c_int, [c_int, i64, i64, PP, c_int, _D, _D, c_dbl, _D, _D, _D]),
            "oracle_block_phase2_merge": (c_int, [i64, i64, _D, _D, _D, _D, _D, c_dbl, _D, _D]),
            "oracle_synthetic_sublayer": (None, [i64, i64, _D, _D, _D]),
            "oracle_rms_norm": (None, [i64, i64, _D, _D, c_dbl, _D]),
            "oracle_block_two_phase_chain": (c_int, [c_int, i64, i64, PP, c_int, _D, _D, _D, _D, c_dbl,
                                                     c_dbl, c_int, _D, _D]),
            "oracle_block_forward_naive": (c_int, [c_int, c_int, i64, i64, _D, _D, _D, _D, _D, c_dbl,
                                                   c_dbl, _D, _D]),
            "oracle_block_forward_two_phase": (c_int, [c_int, c_int, i64, i64, _D, _D, _D, _D,
                                                       c_dbl, _D, _D]),
            "oracle_full_stack_forward": (c_int, [c_int, i64, i64, _D, _D, _D, _D, c_dbl, c_int,
                                                  _D, _D]),
            "oracle_full_stack_two_phase": (c_int, [c_int, c_int, i64, i64, _D, _D, _D, _D, c_dbl, c_int,
                                                    _D, _D]),
            "oracle_atomic_block_size": (c_int, [c_int, c_int, c_int]),
            "oracle_block_schedule": (c_int, [c_int, c_int, _I, _I, c_int]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _arr(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _plist(arrs):
    ptrs = (_D * len(arrs))(*[a.ctypes.data_as(_D) for a in arrs])
    return ptrs


def _check(rc):
    if rc != 0:
        raise RuntimeError(f"oracle call failed ({rc})")


# --------------------------------------------------------------------------
# Rounding to the I/O dtype
# --------------------------------------------------------------------------
def round_to(x, dtype: int) -> np.ndarray:
    """Round every element once, to nearest even, to fp32 or bf16 (kept as float64)."""
    a = _arr(x)
    out = np.empty_like(a)
    _load().oracle_round_array(a.size, _p(a), int(dtype), _p(out))
    return out


def round_bf16_scalar(x: float) -> float:
    return _load().oracle_round_bf16(float(x))


# --------------------------------------------------------------------------
# A1-A3 (DepthResidual.forward)
# --------------------------------------------------------------------------
def fold_query(w, gamma=None) -> np.ndarray:
    """Gain folding w~ = w (.) gamma ("DepthResidual", paragraph (1))."""
    w = _arr(w)
    g = None if gamma is None else _arr(gamma)
    out = np.empty_like(w)
    _load().oracle_fold_query(w.size, _p(w), _p(g), _p(out))
    return out


def depth_aggregate(sources, w, gamma=None, eps: float = 1e-8):
    """Eq. A1-A3 over sources [n, ..., D]; returns (h unrounded, m, lse).

    Rows are every leading index after the source axis (B, T flattened).
    """
    V = _arr(sources)
    n, D = V.shape[0], V.shape[-1]
    lead = V.shape[1:-1]
    R = int(np.prod(lead)) if lead else 1
    w = _arr(w)
    g = None if gamma is None else _arr(gamma)
    h = np.empty((R, D))
    m = np.empty(R)
    lse = np.empty(R)
    _check(_load().oracle_depth_aggregate(n, R, D, _p(V), _p(w), _p(g), float(eps), _p(h), _p(m),
                                          _p(lse)))
    return h.reshape(*lead, D), m.reshape(lead), lse.reshape(lead)


# --------------------------------------------------------------------------
# OS1 / OS2 / single_source_stats
# --------------------------------------------------------------------------
def depth_aggregate_backward(sources, w, gamma, eps: float, dh):
    """Gradients of the depth aggregation for the upstream gradient dh:
    returns (dV [n, ..., D], dw [D], dgamma [D] or None).  Exact fp64."""
    srcs = [_arr(s) for s in sources]
    shape = srcs[0].shape
    D = shape[-1]
    src2 = [s.reshape(-1, D) for s in srcs]
    R = src2[0].shape[0]
    dh = _arr(dh).reshape(R, D)
    w = _arr(w)
    gamma = None if gamma is None else _arr(gamma)
    dV = [np.empty((R, D)) for _ in src2]
    dw = np.empty(D)
    dg = None if gamma is None else np.empty(D)
    _check(_load().oracle_depth_aggregate_backward(len(src2), R, D, _plist(src2), _p(w), _p(gamma),
                                                   float(eps), _p(dh), _plist(dV), _p(dw), _p(dg)))
    return np.stack([x.reshape(shape) for x in dV]), dw, dg


def os1_stats(sources_row, q_eff, eps: float = 1e-8):
    """Eq. OS1 for one token: sources_row [n, D] -> (m, numer [D], denom)."""
    V = _arr(sources_row)
    n, D = V.shape
    rows = [np.ascontiguousarray(V[i]) for i in range(n)]
    q = _arr(q_eff)
    m, d = ctypes.c_double(), ctypes.c_double()
    numer = np.empty(D)
    _load().oracle_os1_stats(n, D, _plist(rows), _p(q), float(eps), ctypes.byref(m), _p(numer),
                             ctypes.byref(d))
    return m.value, numer, d.value


def single_source_stats(p_row, q_eff, eps: float = 1e-8):
    """single_source_stats: (s_p, p, 1)."""
    p = _arr(p_row)
    q = _arr(q_eff)
    m, d = ctypes.c_double(), ctypes.c_double()
    numer = np.empty_like(p)
    _load().oracle_single_source_stats(p.size, _p(p), _p(q), float(eps), ctypes.byref(m),
                                       _p(numer), ctypes.byref(d))
    return m.value, numer, d.value


def os2_merge(a, b):
    """Eq. OS2: merge two (m, numer, denom) triples."""
    na, nb = _arr(a[1]), _arr(b[1])
    m, d = ctypes.c_double(), ctypes.c_double()
    out = np.empty_like(na)
    _load().oracle_os2_merge(na.size, float(a[0]), _p(na), float(a[2]), float(b[0]), _p(nb),
                             float(b[2]), ctypes.byref(m), _p(out), ctypes.byref(d))
    return m.value, out, d.value


# --------------------------------------------------------------------------
# Two-phase Block inference
# --------------------------------------------------------------------------
def block_phase1(blocks, W, G=None, eps: float = 1e-8):
    """Phase 1: S queries W [S, D] over n summaries blocks [n, R, D].

    Returns (O [S, R, D] unrounded, M [S, R], LSE [S, R]).
    """
    Bk = [_arr(b).reshape(-1, _arr(b).shape[-1]) for b in blocks]
    n = len(Bk)
    R, D = Bk[0].shape
    W = _arr(W)
    S = W.shape[0]
    G = None if G is None else _arr(G)
    O = np.empty((S, R, D))
    M = np.empty((S, R))
    LSE = np.empty((S, R))
    _check(_load().oracle_block_phase1(n, R, D, _plist(Bk), S, _p(W), _p(G), float(eps), _p(O),
                                       _p(M), _p(LSE)))
    return O, M, LSE


def block_phase2_merge(o, lse, partial, w, gamma=None, eps: float = 1e-8):
    """Phase 2 merge for one sublayer: returns (h unrounded [R, D], merged lse [R])."""
    o = _arr(o)
    R, D = o.reshape(-1, o.shape[-1]).shape
    lse = _arr(lse)
    p = None if partial is None else _arr(partial)
    w = _arr(w)
    g = None if gamma is None else _arr(gamma)
    h = np.empty((R, D))
    lse_out = np.empty(R)
    _check(_load().oracle_block_phase2_merge(R, D, _p(o), _p(lse), _p(p), _p(w), _p(g), float(eps),
                                             _p(h), _p(lse_out)))
    return h, lse_out


def synthetic_sublayer(u, h) -> np.ndarray:
    """f(h) = 0.5 tanh(u (.) h), the benchmark recipes' stand-in sublayer."""
    h = _arr(h)
    R, D = h.reshape(-1, h.shape[-1]).shape
    u = _arr(u)
    out = np.empty((R, D))
    _load().oracle_synthetic_sublayer(R, D, _p(u), _p(h), _p(out))
    return out


def rms_norm(x, weight=None, eps: float = 1e-6) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) (.) weight, row by row (the sublayer pre-norm)."""
    x = _arr(x)
    shape = x.shape
    x2 = x.reshape(-1, shape[-1])
    R, D = x2.shape
    weight = None if weight is None else _arr(weight)
    y = np.empty((R, D))
    _load().oracle_rms_norm(R, D, _p(x2), _p(weight), float(eps), _p(y))
    return y.reshape(shape)


def block_two_phase_chain(blocks, W, G, U, eps: float, dtype: int, NW=None, norm_eps: float = 1e-6):
    """One block of the two-phase recurrence with materialisation rounding.

    NW ([S, D] or None): the sublayers' pre-norm weights; with them each
    sublayer reads rms_norm(h_k) (formed from the unrounded h_k).
    Returns (H [S, R, D] rounded sublayer inputs, P [R, D] rounded final partial).
    """
    Bk = [_arr(b).reshape(-1, _arr(b).shape[-1]) for b in blocks]
    R, D = Bk[0].shape
    W = _arr(W)
    S = W.shape[0]
    G = None if G is None else _arr(G)
    U = _arr(U)
    H = np.empty((S, R, D))
    P = np.empty((R, D))
    NW = None if NW is None else _arr(NW)
    _check(_load().oracle_block_two_phase_chain(len(Bk), R, D, _plist(Bk), S, _p(W), _p(G), _p(U),
                                                _p(NW), float(norm_eps), float(eps), int(dtype),
                                                _p(H), _p(P)))
    return H, P


def block_forward_naive(x, W, G, U, S: int, eps: float = 1e-8, NW=None, norm_eps: float = 1e-6):
    """forward_naive with the synthetic sublayer, exact fp64: returns (H [N,R,D], y [R,D]).

    NW ([N, D] or None): pre-norm weights; sublayer l then reads rms_norm(h_l).
    """
    x = _arr(x)
    R, D = x.reshape(-1, x.shape[-1]).shape
    U = _arr(U)
    N = U.shape[0]
    W = _arr(W)
    G = None if G is None else _arr(G)
    H = np.empty((N, R, D))
    y = np.empty((R, D))
    NW = None if NW is None else _arr(NW)
    _check(_load().oracle_block_forward_naive(N, S, R, D, _p(x), _p(W), _p(G), _p(U), _p(NW),
                                              float(norm_eps), float(eps), _p(H), _p(y)))
    return H, y


def block_forward_two_phase(x, W, G, U, S: int, eps: float = 1e-8):
    """_run_block_two_phase per block, exact fp64: returns (H [N,R,D], y [R,D])."""
    x = _arr(x)
    R, D = x.reshape(-1, x.shape[-1]).shape
    U = _arr(U)
    N = U.shape[0]
    W = _arr(W)
    G = None if G is None else _arr(G)
    H = np.empty((N, R, D))
    y = np.empty((R, D))
    _check(_load().oracle_block_forward_two_phase(N, S, R, D, _p(x), _p(W), _p(G), _p(U),
                                                  float(eps), _p(H), _p(y)))
    return H, y


def full_stack_forward(v0, W, G, U, eps: float, dtype: int):
    """Full stack with the synthetic sublayer: returns (V [L+1,R,D] rounded, y [R,D] unrounded)."""
    v0 = _arr(v0)
    R, D = v0.reshape(-1, v0.shape[-1]).shape
    U = _arr(U)
    L = U.shape[0]
    W = _arr(W)
    G = None if G is None else _arr(G)
    V = np.empty((L + 1, R, D))
    y = np.empty((R, D))
    _check(_load().oracle_full_stack_forward(L, R, D, _p(v0), _p(W), _p(G), _p(U), float(eps),
                                             int(dtype), _p(V), _p(y)))
    return V, y


# --------------------------------------------------------------------------
# Bookkeeping
# --------------------------------------------------------------------------
def full_stack_two_phase(v0, W, G, U, S: int, eps: float, dtype: int):
    """Full stack with the two-phase schedule of block size S: returns (V [L+1, R, D], y [R, D])."""
    v0 = _arr(v0)
    R, D = v0.reshape(-1, v0.shape[-1]).shape
    U = _arr(U)
    L = U.shape[0]
    W = _arr(W)
    G = None if G is None else _arr(G)
    V = np.empty((L + 1, R, D))
    y = np.empty((R, D))
    _check(_load().oracle_full_stack_two_phase(L, int(S), R, D, _p(v0), _p(W), _p(G), _p(U), float(eps),
                                               int(dtype), _p(V), _p(y)))
    return V, y


def atomic_block_size(num_hidden_layers: int, attnres_block_size=None) -> int:
    has = attnres_block_size is not None
    return int(_load().oracle_atomic_block_size(int(num_hidden_layers), int(has),
                                                int(attnres_block_size or 0)))


def block_schedule(num_atomic: int, block_size: int):
    """forward_naive's source lists: list of num_atomic+1 lists (-1 = running partial)."""
    cap = (num_atomic + 1) * (num_atomic + 2)
    counts = (ctypes.c_int * (num_atomic + 1))()
    ids = (ctypes.c_int * cap)()
    w = _load().oracle_block_schedule(int(num_atomic), int(block_size), counts, ids, cap)
    if w < 0:
        raise RuntimeError("schedule capacity")
    out, k = [], 0
    for c in counts:
        out.append([ids[k + j] for j in range(c)])
        k += c
    return out
