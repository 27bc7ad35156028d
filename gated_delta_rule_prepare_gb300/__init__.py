"""Python binding of libkda, the GB300 (sm_103a) KDA core library.

Argument marshalling only: every function here checks tensor dtypes, shapes
and devices, then calls the C ABI declared in ``include/kda.h`` with raw
device pointers and the current CUDA stream.  All arithmetic runs in the
library's CUDA kernels; there is no fallback.  Importing this package on a
machine without the built library raises immediately.

Entry points (same names as the C ABI): ``kda_decode``, ``kda_decode_k``,
``kda_prefill``, ``kda_prefill_gated``, ``kda_prefill_o_norm``, ``kda_conv_silu_l2``,
``kda_conv_silu_l2_k``,
``kda_gate``, ``kda_o_norm_gated``, ``kda_prefill_workspace_size``, ``kda_sync_status``.
``kda_prefill_static_ws`` is reached through ``LIB`` (its callers hold raw pointers).
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

HEAD_DIM = 128
Q_SCALE = 0.08838834764831845
MAX_K = 8
F32, BF16 = 0, 1

_c = ctypes
_vp, _i, _u64, _i64, _f, _sz = _c.c_void_p, _c.c_int, _c.c_uint64, _c.c_int64, _c.c_float, _c.c_size_t


class KdaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("kda status %d: %s" % (status, message))
        self.status = status


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError("libkda.so is not built (%s); run __graft_entry__.build() first" % path)
    lib = _c.CDLL(path)
    sig = {
        "kda_decode": [_vp] * 7 + [_i] * 3 + [_u64],
        "kda_decode_k": [_vp] * 7 + [_i] * 4 + [_vp, _i, _u64],
        "kda_prefill": [_vp] * 7 + [_i, _i, _i, _f, _i, _i, _i, _i64, _vp, _i, _vp, _sz, _u64],
        "kda_conv_silu_l2": [_vp] * 4 + [_i, _i, _vp, _i, _f, _i, _i, _u64],
        "kda_sync_status": [_u64],
        "kda_o_norm_gated": [_vp] * 4 + [_i64, _i, _i, _f, _u64],
        "kda_gate": [_vp, _i64, _vp, _vp, _f, _vp, _i64, _vp, _vp, _i, _i64, _i, _i, _u64],
        "kda_prefill_gated": [_vp] * 5 + [_i64, _vp, _vp, _f, _vp, _i64, _vp, _i, _i, _i, _i,
                                          _i64, _vp, _i, _vp, _sz, _u64],
        "kda_conv_silu_l2_k": [_vp] * 4 + [_i, _i, _i, _f, _i, _i, _vp, _i, _u64],
        "kda_prefill_o_norm": [_vp] * 7 + [_i64, _vp, _f, _vp, _i64, _i, _i, _i, _i, _i, _i,
                                           _i64, _vp, _i, _vp, _sz, _u64],
    }
    for name, args in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = _i
    lib.kda_prefill_workspace_size.argtypes = [_i64, _i, _i, _i, _i, _i]
    lib.kda_prefill_workspace_size.restype = _sz
    lib.kda_last_error.argtypes = []
    lib.kda_last_error.restype = _c.c_char_p
    lib.kda_version.argtypes = []
    lib.kda_version.restype = _c.c_char_p
    return lib


LIB = _load()


def _check(status: int):
    if status != 0:
        raise KdaError(status, LIB.kda_last_error().decode())


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _contig(t, name):
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def version() -> str:
    return LIB.kda_version().decode()


def kda_decode(state, q, k, v, g, beta, o):
    """One token per sequence: state [N,H,128,128] FP32 in place; q, k, v, g, o
    [N,H,128] FP32; beta [N,H] FP32."""
    N, H = state.shape[0], state.shape[1]
    for n_, t in (("state", state), ("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                  ("o", o)):
        _contig(t, n_)
    if q.shape != (N, H, HEAD_DIM) or beta.shape != (N, H):
        raise ValueError("kda_decode: shape mismatch")
    f = torch.float32
    _check(LIB.kda_decode(_ptr(state, f, "state"), _ptr(q, f, "q"), _ptr(k, f, "k"),
                          _ptr(v, f, "v"), _ptr(g, f, "g"), _ptr(beta, f, "beta"),
                          _ptr(o, f, "o"), N, H, state.shape[-1], _stream(state)))


def kda_decode_k(state, q, k, v, g, beta, o, snapshots=()):
    """k rows per sequence walked in order: q, k, v, g, o [N,k,H,128]; beta
    [N,k,H]; snapshots: up to k tensors [N,H,128,128], snapshots[t] = state
    after row t."""
    N, krows, H = q.shape[0], q.shape[1], q.shape[2]
    for n_, t in (("state", state), ("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta),
                  ("o", o)):
        _contig(t, n_)
    if beta.shape != (N, krows, H) or state.shape[:2] != (N, H):
        raise ValueError("kda_decode_k: shape mismatch")
    f = torch.float32
    snaps = list(snapshots)
    for s in snaps:
        _contig(s, "snapshot")
        if s.shape != state.shape or s.dtype != f:
            raise ValueError("kda_decode_k: snapshot shape/dtype mismatch")
    arr = (_c.c_void_p * max(1, len(snaps)))(*[s.data_ptr() for s in snaps])
    _check(LIB.kda_decode_k(_ptr(state, f, "state"), _ptr(q, f, "q"), _ptr(k, f, "k"),
                            _ptr(v, f, "v"), _ptr(g, f, "g"), _ptr(beta, f, "beta"),
                            _ptr(o, f, "o"), N, krows, H, state.shape[-1],
                            _c.cast(arr, _c.c_void_p) if snaps else None, len(snaps),
                            _stream(state)))


def kda_prefill_workspace_size(rows, n_seqs, chunk, heads, dtype=torch.bfloat16):
    """Workspace bytes kda_prefill needs for `rows` token rows in total."""
    in_dtype = BF16 if dtype == torch.bfloat16 else F32
    return int(LIB.kda_prefill_workspace_size(int(rows), n_seqs, chunk, heads, HEAD_DIM, in_dtype))


def kda_prefill(state, q, k, v, g, beta, o, t, chunk, pad_fill=0.0, cu_seqlens=None,
                workspace=None):
    """Chunked prefill.  Without cu_seqlens: q, k, v, g [N, T_pad, H, 128]
    (or [T_pad, H, 128] for one sequence), beta [N, T_pad, H], t valid tokens
    per sequence; rows [t, T_pad) are the caller's padded tail (pad_fill),
    neither read into arithmetic nor written.  With
    cu_seqlens (device int32 [N+1]): packed rows [T, H, 128] and t = T.
    q, k and v may be strided views whose token rows are ``q.stride(-3)``
    elements apart (e.g. slices of one [T, 3*H*128] buffer)."""
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise TypeError("kda_prefill: inputs must be float32 or bfloat16")
    in_dtype = BF16 if dt == torch.bfloat16 else F32
    H = q.shape[-2]
    if q.shape[-1] != HEAD_DIM:
        raise ValueError("kda_prefill: head_dim must be 128")
    for n_, t_ in (("q", q), ("k", k), ("v", v)):
        if t_.dtype != dt or t_.stride(-1) != 1 or t_.stride(-2) != HEAD_DIM:
            raise ValueError("kda_prefill: %s must have unit channel stride and heads packed" % n_)
    stride = q.stride(-3)
    if k.stride(-3) != stride or v.stride(-3) != stride:
        raise ValueError("kda_prefill: q, k, v must share one token-row stride")
    for n_, t_ in (("g", g), ("beta", beta), ("o", o), ("state", state)):
        _contig(t_, n_)
    if g.dtype != dt or beta.dtype != dt:
        raise TypeError("kda_prefill: g and beta must have the inputs' dtype")
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.numel() - 1
        t_pad = t
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise TypeError("kda_prefill: cu_seqlens must be a CUDA int32 tensor")
        rows = q.shape[0]
    else:
        if q.dim() == 3:
            n_seqs, t_pad = 1, q.shape[0]
        else:
            n_seqs, t_pad = q.shape[0], q.shape[1]
            if q.dim() == 4 and q.stride(0) != t_pad * stride:
                raise ValueError("kda_prefill: sequences must be consecutive row blocks")
        rows = n_seqs * t_pad
    if g.numel() != rows * H * HEAD_DIM or beta.numel() != rows * H or o.numel() != rows * H * HEAD_DIM:
        raise ValueError("kda_prefill: g/beta/o sizes do not match the token rows")
    if state.numel() != n_seqs * H * HEAD_DIM * HEAD_DIM or state.dtype != torch.float32:
        raise ValueError("kda_prefill: state must be FP32 [N, H, 128, 128]")
    ws_need = kda_prefill_workspace_size(rows, n_seqs, chunk, H, dt)
    if ws_need and workspace is None:
        # The caller gave none: allocate one here, outside the library (which
        # never allocates).  Timed callers pass a preallocated buffer.
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=q.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(LIB.kda_prefill(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(o, torch.float32, "o"), int(t), int(t_pad), int(chunk),
                           float(pad_fill), H, HEAD_DIM, in_dtype, int(stride),
                           _ptr(cu_seqlens), n_seqs, ws_ptr, ws_bytes, _stream(state)))


def _row_view(x, rows, hd, name):
    """(pointer, token-row stride) of a BF16 [rows, >= hd] view with unit
    channel stride, or of any contiguous tensor of rows x hd values."""
    if x.dtype != torch.bfloat16 or not x.is_cuda:
        raise TypeError("%s must be a CUDA bfloat16 tensor" % name)
    if x.is_contiguous() and x.numel() == rows * hd:
        return x.data_ptr(), hd
    if x.dim() == 2 and x.shape[0] == rows and x.shape[1] >= hd and x.stride(1) == 1:
        return x.data_ptr(), x.stride(0)
    raise ValueError("%s must hold rows x heads*128 values (contiguous, or a 2-D row view)" % name)


def kda_prefill_o_norm(state, q, k, v, g, beta, gate, w, out, t, chunk=64, eps=1e-6,
                       cu_seqlens=None, workspace=None):
    """kda_prefill with the sigmoid-gated RMSNorm fused into its epilogue (BF16
    inputs, tensor-core path): writes out BF16 [rows, H*128] =
    rmsnorm(o) * w * sigmoid(gate) instead of the FP32 core output o.  gate
    and out: BF16 with rows x H*128 values (contiguous, or 2-D row views);
    w: BF16 [128].  The other arguments are kda_prefill's."""
    if q.dtype != torch.bfloat16:
        raise TypeError("kda_prefill_o_norm: inputs must be bfloat16")
    H = q.shape[-2]
    if q.shape[-1] != HEAD_DIM:
        raise ValueError("kda_prefill_o_norm: head_dim must be 128")
    for n_, t_ in (("q", q), ("k", k), ("v", v)):
        if t_.dtype != q.dtype or t_.stride(-1) != 1 or t_.stride(-2) != HEAD_DIM:
            raise ValueError("kda_prefill_o_norm: %s must have unit channel stride and heads "
                             "packed" % n_)
    stride = q.stride(-3)
    if k.stride(-3) != stride or v.stride(-3) != stride:
        raise ValueError("kda_prefill_o_norm: q, k, v must share one token-row stride")
    for n_, t_ in (("g", g), ("beta", beta), ("state", state), ("w", w)):
        _contig(t_, n_)
    if g.dtype != q.dtype or beta.dtype != q.dtype:
        raise TypeError("kda_prefill_o_norm: g and beta must have the inputs' dtype")
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.numel() - 1
        t_pad = t
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise TypeError("kda_prefill_o_norm: cu_seqlens must be a CUDA int32 tensor")
    else:
        if q.dim() == 3:
            n_seqs, t_pad = 1, q.shape[0]
        else:
            n_seqs, t_pad = q.shape[0], q.shape[1]
            if q.dim() == 4 and q.stride(0) != t_pad * stride:
                raise ValueError("kda_prefill_o_norm: sequences must be consecutive row blocks")
    rows = t if cu_seqlens is not None else n_seqs * t_pad
    if g.numel() != rows * H * HEAD_DIM or beta.numel() != rows * H:
        raise ValueError("kda_prefill_o_norm: g/beta sizes do not match the token rows")
    if state.numel() != n_seqs * H * HEAD_DIM * HEAD_DIM or state.dtype != torch.float32:
        raise ValueError("kda_prefill_o_norm: state must be FP32 [N, H, 128, 128]")
    if w.numel() != HEAD_DIM or w.dtype != torch.bfloat16:
        raise ValueError("kda_prefill_o_norm: w must be BF16 [128]")
    g_ptr, g_stride = _row_view(gate, rows, H * HEAD_DIM, "gate")
    o_ptr, o_stride = _row_view(out, rows, H * HEAD_DIM, "out")
    ws_need = kda_prefill_workspace_size(rows, n_seqs, chunk, H, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(ws_need, 1), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(LIB.kda_prefill_o_norm(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                  g_ptr, int(g_stride), _ptr(w), float(eps), o_ptr,
                                  int(o_stride), int(t), int(t_pad), int(chunk), H, HEAD_DIM,
                                  BF16, int(stride), _ptr(cu_seqlens), n_seqs,
                                  workspace.data_ptr(), ws_bytes, _stream(state)))


def kda_prefill_gated(state, q, k, v, g_raw, dt_bias, a_log, b_raw, o, t, gate_lower_bound,
                      cu_seqlens=None, workspace=None):
    """Tensor-core prefill (BF16 q, k, v; chunk 64) with the forget gate and
    beta formed in the prepare kernel from g_raw BF16 [rows, >= H*128],
    dt_bias FP32 [H*128], a_log FP32 [H] and b_raw BF16 [rows, >= H].
    Without cu_seqlens: q, k, v [N, T_pad, H, 128] (or [T_pad, H, 128]), t
    valid tokens per sequence, rows [t, T_pad) left as they are and never
    used.  With cu_seqlens (device int32 [N+1]): packed rows and t = T."""
    b16 = torch.bfloat16
    H = q.shape[-2]
    if q.shape[-1] != HEAD_DIM:
        raise ValueError("kda_prefill_gated: head_dim must be 128")
    for n_, t_ in (("q", q), ("k", k), ("v", v)):
        if t_.dtype != b16 or t_.stride(-1) != 1 or t_.stride(-2) != HEAD_DIM:
            raise ValueError("kda_prefill_gated: %s must be bfloat16 with unit channel stride "
                             "and heads packed" % n_)
    stride = q.stride(-3)
    if k.stride(-3) != stride or v.stride(-3) != stride:
        raise ValueError("kda_prefill_gated: q, k, v must share one token-row stride")
    for n_, t_ in (("dt_bias", dt_bias), ("a_log", a_log), ("o", o), ("state", state)):
        _contig(t_, n_)
    if g_raw.dim() != 2 or g_raw.stride(1) != 1 or b_raw.dim() != 2 or b_raw.stride(1) != 1:
        raise ValueError("kda_prefill_gated: g_raw and b_raw must be 2-D with unit channel stride")
    if cu_seqlens is not None:
        n_seqs = cu_seqlens.numel() - 1
        t_pad = t
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise TypeError("kda_prefill_gated: cu_seqlens must be a CUDA int32 tensor")
    elif q.dim() == 3:
        n_seqs, t_pad = 1, q.shape[0]
    else:
        n_seqs, t_pad = q.shape[0], q.shape[1]
        if q.stride(0) != t_pad * stride:
            raise ValueError("kda_prefill_gated: sequences must be consecutive row blocks")
    rows = t if cu_seqlens is not None else n_seqs * t_pad
    if (g_raw.shape[0] != rows or b_raw.shape[0] != rows or g_raw.shape[1] < H * HEAD_DIM
            or b_raw.shape[1] < H or dt_bias.numel() != H * HEAD_DIM or a_log.numel() != H
            or o.numel() != rows * H * HEAD_DIM):
        raise ValueError("kda_prefill_gated: shape mismatch")
    if state.numel() != n_seqs * H * HEAD_DIM * HEAD_DIM or state.dtype != torch.float32:
        raise ValueError("kda_prefill_gated: state must be FP32 [N, H, 128, 128]")
    if workspace is None:
        need = kda_prefill_workspace_size(rows, n_seqs, 64, H, b16)
        if need == 0:  # KDA_PREFILL_IMPL=simt makes the size query answer for the SIMT kernel
            raise KdaError(3, "kda_prefill_gated runs only on the tensor-core "
                           "kernels: unset KDA_PREFILL_IMPL=simt or pass a workspace")
        # allocated here, outside the library (which never allocates)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(LIB.kda_prefill_gated(
        _ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(g_raw, b16, "g_raw"), int(g_raw.stride(0)),
        _ptr(dt_bias, torch.float32, "dt_bias"), _ptr(a_log, torch.float32, "a_log"),
        float(gate_lower_bound), _ptr(b_raw, b16, "b_raw"), int(b_raw.stride(0)),
        _ptr(o, torch.float32, "o"), int(t), int(t_pad), H, HEAD_DIM, int(stride),
        _ptr(cu_seqlens), n_seqs, workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), _stream(state)))


def kda_conv_silu_l2(conv_state, x, w, out, cu_seqlens=None, n_seqs=None, l2_eps=1e-6):
    """Depthwise causal conv + SiLU + L2(q, k).  x, out BF16 [tokens, 3*H*128];
    w BF16 [3*H*128, K]; conv_state FP32 [N, 3*H*128, K] in place.  Without
    cu_seqlens x holds N sequences of tokens/N tokens each."""
    for n_, t_ in (("conv_state", conv_state), ("x", x), ("w", w), ("out", out)):
        _contig(t_, n_)
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("kda_conv_silu_l2: x, w, out must be bfloat16")
    conv_dim = x.shape[-1]
    if conv_dim % (3 * HEAD_DIM):
        raise ValueError("kda_conv_silu_l2: channels must be 3 * heads * 128")
    H = conv_dim // (3 * HEAD_DIM)
    K = w.shape[1]
    tokens = x.numel() // conv_dim
    if cu_seqlens is not None:
        N = cu_seqlens.numel() - 1
        t = tokens
    else:
        N = conv_state.shape[0] if n_seqs is None else n_seqs
        if tokens % N:
            raise ValueError("kda_conv_silu_l2: tokens not divisible by n_seqs")
        t = tokens // N
    if conv_state.shape != (N, conv_dim, K):
        raise ValueError("kda_conv_silu_l2: conv_state must be [N, conv_dim, K]")
    _check(LIB.kda_conv_silu_l2(_ptr(conv_state, torch.float32, "conv_state"), _ptr(x), _ptr(w),
                                _ptr(out), t, N, _ptr(cu_seqlens), K, float(l2_eps), H,
                                HEAD_DIM, _stream(x)))


def kda_conv_silu_l2_k(conv_state, x, w, out, snapshots=(), l2_eps=1e-6):
    """k rows per sequence through the conv front end: x, out BF16 [N, k,
    3*H*128]; conv_state FP32 [N, 3*H*128, K] in place; snapshots: up to k
    FP32 tensors shaped like conv_state, snapshots[t] = conv state after row t."""
    for n_, t_ in (("conv_state", conv_state), ("x", x), ("w", w), ("out", out)):
        _contig(t_, n_)
    if x.dtype != torch.bfloat16 or w.dtype != torch.bfloat16 or out.dtype != torch.bfloat16:
        raise TypeError("kda_conv_silu_l2_k: x, w, out must be bfloat16")
    N, krows, conv_dim = x.shape
    if conv_dim % (3 * HEAD_DIM) or conv_state.shape != (N, conv_dim, w.shape[1]):
        raise ValueError("kda_conv_silu_l2_k: shape mismatch")
    snaps = list(snapshots)
    for s_ in snaps:
        _contig(s_, "snapshot")
        if s_.shape != conv_state.shape or s_.dtype != torch.float32:
            raise ValueError("kda_conv_silu_l2_k: snapshot shape/dtype mismatch")
    arr = (_c.c_void_p * max(1, len(snaps)))(*[s_.data_ptr() for s_ in snaps])
    _check(LIB.kda_conv_silu_l2_k(_ptr(conv_state, torch.float32, "conv_state"), _ptr(x),
                                  _ptr(w), _ptr(out), N, krows, w.shape[1], float(l2_eps),
                                  conv_dim // (3 * HEAD_DIM), HEAD_DIM,
                                  _c.cast(arr, _c.c_void_p) if snaps else None, len(snaps),
                                  _stream(x)))


def kda_o_norm_gated(core, gate, w, out, eps=1e-6):
    """Sigmoid-gated RMSNorm: core FP32 [rows, H, 128] (or [rows, H*128]),
    gate and out BF16 [rows, H*128], w BF16 [128]."""
    for n_, t_ in (("core", core), ("gate", gate), ("w", w), ("out", out)):
        _contig(t_, n_)
    rows = core.shape[0]
    hd = core.numel() // max(rows, 1) if rows else gate.shape[-1]
    if hd % HEAD_DIM or gate.numel() != core.numel() or out.numel() != core.numel():
        raise ValueError("kda_o_norm_gated: core, gate and out must hold rows x H x 128 values")
    if w.numel() != HEAD_DIM:
        raise ValueError("kda_o_norm_gated: w must hold 128 values")
    b16 = torch.bfloat16
    _check(LIB.kda_o_norm_gated(_ptr(core, torch.float32, "core"), _ptr(gate, b16, "gate"),
                                _ptr(w, b16, "w"), _ptr(out, b16, "out"), int(rows),
                                hd // HEAD_DIM, HEAD_DIM, float(eps), _stream(core)))


def kda_gate(g_raw, dt_bias, a_log, b_raw, g_out, beta_out, gate_lower_bound):
    """Forget gate and beta: g_raw BF16 [rows, >= H*128] (row pitch a multiple
    of 8 channels), dt_bias FP32 [H*128], a_log FP32 [H], b_raw BF16
    [rows, >= H]; g_out [rows, H, 128] and beta_out [rows, H] in FP32 or BF16
    (both the same dtype)."""
    for n_, t_ in (("dt_bias", dt_bias), ("a_log", a_log), ("g_out", g_out),
                   ("beta_out", beta_out)):
        _contig(t_, n_)
    if g_raw.dim() != 2 or g_raw.stride(1) != 1 or b_raw.dim() != 2 or b_raw.stride(1) != 1:
        raise ValueError("kda_gate: g_raw and b_raw must be 2-D with unit channel stride")
    rows, H = g_out.shape[0], a_log.numel()
    if (g_out.numel() != rows * H * HEAD_DIM or beta_out.numel() != rows * H
            or dt_bias.numel() != H * HEAD_DIM or g_raw.shape[0] != rows
            or b_raw.shape[0] != rows or g_raw.shape[1] < H * HEAD_DIM or b_raw.shape[1] < H):
        raise ValueError("kda_gate: shape mismatch")
    if g_out.dtype != beta_out.dtype or g_out.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("kda_gate: g_out and beta_out must both be FP32 or both BF16")
    b16 = torch.bfloat16
    _check(LIB.kda_gate(_ptr(g_raw, b16, "g_raw"), int(g_raw.stride(0)),
                        _ptr(dt_bias, torch.float32, "dt_bias"), _ptr(a_log, torch.float32, "a_log"),
                        float(gate_lower_bound), _ptr(b_raw, b16, "b_raw"), int(b_raw.stride(0)),
                        _ptr(g_out), _ptr(beta_out), BF16 if g_out.dtype == b16 else F32,
                        int(rows), H, HEAD_DIM, _stream(g_out)))


def kda_sync_status(device=None):
    """Synchronise the current stream and raise if a device-side check failed."""
    s = torch.cuda.current_stream(device).cuda_stream
    _check(LIB.kda_sync_status(s))
