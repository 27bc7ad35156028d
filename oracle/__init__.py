"""FP64 CPU oracle for the KDA core -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library never does.  The arithmetic lives in
``kda_oracle.c`` (plain C, double precision); this module only marshals numpy
or torch CPU arrays into it.

Functions return float64 numpy arrays.  Inputs may be float32, bfloat16 or
float64 tensors/arrays: they are widened exactly to float64 first, so the
oracle sees the very values the GPU was given.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None
_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int)


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.kda_oracle_default_q_scale.restype = ctypes.c_double
        L.kda_oracle_default_q_scale.argtypes = [ctypes.c_int]
        L.kda_oracle_threads.restype = ctypes.c_int
        L.kda_oracle_recurrent.restype = None
        L.kda_oracle_recurrent.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double] + [_dp] * 8
        L.kda_oracle_chunk_prepare.restype = None
        L.kda_oracle_chunk_prepare.argtypes = ([ctypes.c_int, ctypes.c_int, ctypes.c_double]
                                               + [_dp] * 5 + [ctypes.c_int, ctypes.c_int]
                                               + [_dp] * 9)
        L.kda_oracle_chunk_scan.restype = None
        L.kda_oracle_chunk_scan.argtypes = ([ctypes.c_int, ctypes.c_int] + [_dp] * 7
                                            + [ctypes.c_int, _dp, _dp, ctypes.c_int])
        L.kda_oracle_chunked.restype = None
        L.kda_oracle_chunked.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double] + [_dp] * 7
        L.kda_oracle_conv_silu_l2.restype = None
        L.kda_oracle_conv_silu_l2.argtypes = ([ctypes.c_int, _ip] + [ctypes.c_int] * 3
                                              + [ctypes.c_double] + [_dp] * 4)
        L.kda_oracle_o_norm_gated.restype = None
        L.kda_oracle_o_norm_gated.argtypes = ([ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_double] + [_dp] * 4)
        L.kda_oracle_gate.restype = None
        L.kda_oracle_gate.argtypes = ([ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double] + [_dp] * 6)
        _LIB = L
    return _LIB


def f64(x) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype) or array to float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().to("cpu", torch.float64).numpy())
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_dp)


def q_scale(head_dim: int = 128) -> float:
    """The query scale the oracle fixes: 1/sqrt(head_dim)."""
    return float(lib().kda_oracle_default_q_scale(head_dim))


def threads() -> int:
    return int(lib().kda_oracle_threads())


def recurrent(q, k, v, g, beta, state, scale=None, snapshots=False):
    """Token-by-token recurrence.

    q, k, v, g: [N, T, H, D]; beta: [N, T, H]; state: [N, H, D, D].
    Returns (o [N, T, H, D], final state [N, H, D, D]) and, with
    ``snapshots=True``, also the state after every token [T, N, H, D, D].
    """
    q, k, v, g, beta = (f64(a) for a in (q, k, v, g, beta))
    S = f64(state).copy()
    N, T, H, D = q.shape
    assert k.shape == v.shape == g.shape == q.shape and beta.shape == (N, T, H)
    assert S.shape == (N, H, D, D)
    if scale is None:
        scale = q_scale(D)
    o = np.zeros_like(q)
    snaps = np.zeros((T, N, H, D, D)) if snapshots else None
    lib().kda_oracle_recurrent(N, T, H, D, float(scale), _p(q), _p(k), _p(v), _p(g),
                               _p(beta), _p(S), _p(o),
                               _p(snaps) if snapshots else ctypes.cast(None, _dp))
    if snapshots:
        return o, S, snaps
    return o, S


def prefill(q, k, v, g, beta, state, scale=None):
    """One sequence: q, k, v, g [T, H, D], beta [T, H], state [H, D, D]."""
    o, S = recurrent(f64(q)[None], f64(k)[None], f64(v)[None], f64(g)[None],
                     f64(beta)[None], f64(state)[None], scale)
    return o[0], S[0]


def chunked(q, k, v, g, beta, state, chunk, scale=None):
    """Chunked form of one sequence (prepare + scan per chunk), FP64."""
    q, k, v, g, beta = (f64(a) for a in (q, k, v, g, beta))
    S = f64(state).copy()
    T, H, D = q.shape
    if scale is None:
        scale = q_scale(D)
    o = np.zeros_like(q)
    lib().kda_oracle_chunked(T, H, D, int(chunk), float(scale), _p(q), _p(k), _p(v),
                             _p(g), _p(beta), _p(S), _p(o))
    return o, S


def chunk_prepare(q, k, v, g, beta, scale=None):
    """Intra-chunk stage of one chunk of one head: q, k, v, g [L, D], beta [L].
    Returns a dict of Gamma, A, T, W, Ut, P, Qt, Kh, dec."""
    q, k, v, g, beta = (f64(a) for a in (q, k, v, g, beta))
    L, D = q.shape
    if scale is None:
        scale = q_scale(D)
    out = {n: np.zeros((L, D)) for n in ("Gamma", "W", "Ut", "Qt", "Kh")}
    out.update({n: np.zeros((L, L)) for n in ("A", "T", "P")})
    out["dec"] = np.zeros(D)
    lib().kda_oracle_chunk_prepare(L, D, float(scale), _p(q), _p(k), _p(v), _p(g), _p(beta),
                                   D, 1, _p(out["Gamma"]), _p(out["A"]), _p(out["T"]),
                                   _p(out["W"]), _p(out["Ut"]), _p(out["P"]), _p(out["Qt"]),
                                   _p(out["Kh"]), _p(out["dec"]))
    return out


def chunk_scan(prep: dict, beta, state):
    """Inter-chunk stage: carries state [D, D] across one prepared chunk."""
    beta = f64(beta)
    S = f64(state).copy()
    L, D = prep["W"].shape
    o = np.zeros((L, D))
    lib().kda_oracle_chunk_scan(L, D, _p(prep["W"]), _p(prep["Ut"]), _p(prep["P"]),
                                _p(prep["Qt"]), _p(prep["Kh"]), _p(prep["dec"]), _p(beta), 1,
                                _p(S), _p(o), D)
    return o, S


def conv_silu_l2(x, w, conv_state, cu_seqlens, heads, head_dim=128, l2_eps=1e-6):
    """Depthwise causal conv + SiLU + L2(q, k).  x [T_total, 3*H*D], w [3*H*D, K],
    conv_state [N, 3*H*D, K]; returns (out [T_total, 3*H*D], new conv_state)."""
    x, w = f64(x), f64(w)
    st = f64(conv_state).copy()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    N = cu.shape[0] - 1
    K = w.shape[1]
    assert x.shape[1] == 3 * heads * head_dim and st.shape == (N, x.shape[1], K)
    out = np.zeros_like(x)
    lib().kda_oracle_conv_silu_l2(N, cu.ctypes.data_as(_ip), heads, head_dim, K,
                                  float(l2_eps), _p(x), _p(w), _p(st), _p(out))
    return out, st


def o_norm_gated(core, gate, w, eps=1e-6):
    """Sigmoid-gated RMSNorm: core [rows, H, D] (pre-norm core output), gate
    [rows, H*D] or [rows, H, D], w [D]; returns out [rows, H, D] (FP64)."""
    core, gate, w = f64(core), f64(gate), f64(w)
    rows, H, D = core.shape
    gate = np.ascontiguousarray(gate.reshape(rows, H, D))
    assert w.shape == (D,)
    out = np.zeros_like(core)
    lib().kda_oracle_o_norm_gated(rows, H, D, float(eps), _p(core), _p(gate), _p(w), _p(out))
    return out


def gate(g_raw, dt_bias, a_log, lower_bound, b):
    """Forget gate and beta (the reading stated in kda_oracle.c): g_raw
    [rows, H*D] or [rows, H, D], dt_bias [H*D], a_log [H], b [rows, H];
    returns g [rows, H, D] and beta [rows, H] (FP64)."""
    a_log, b = f64(a_log), f64(b)
    H = a_log.shape[0]
    rows = b.shape[0]
    g_raw = np.ascontiguousarray(f64(g_raw).reshape(rows, H, -1))
    D = g_raw.shape[2]
    dt_bias = np.ascontiguousarray(f64(dt_bias).reshape(H * D))
    assert b.shape == (rows, H)
    g = np.zeros_like(g_raw)
    beta = np.zeros_like(b)
    lib().kda_oracle_gate(rows, H, D, float(lower_bound), _p(g_raw), _p(dt_bias), _p(a_log),
                          _p(b), _p(g), _p(beta))
    return g, beta
