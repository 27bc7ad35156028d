"""The C ABI without a GPU: the library loads, exports every entry point
include/kda.h declares, and refuses bad arguments before touching the device."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._library_builder().build()
    L = ctypes.CDLL(path)
    L.kda_last_error.restype = ctypes.c_char_p
    return L


def test_header_declares_the_four_calls_and_helpers():
    fns = declared_functions()
    for name in ("kda_prefill", "kda_decode", "kda_decode_k", "kda_conv_silu_l2",
                 "kda_prefill_workspace_size", "kda_sync_status", "kda_last_error"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_every_declaration_is_documented():
    text = open(HEADER).read()
    for name in declared_functions():
        m = re.search(r"\n([a-z][a-z_0-9 ]*\**\s*)" + name + r"\(", text)
        assert m, name
        prev = text[:m.start()].rstrip()
        assert prev.endswith("*/"), "%s has no comment block above it" % name


V, I, F, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64, ctypes.c_size_t
BUF = ctypes.create_string_buffer(64)
P = ctypes.cast(ctypes.addressof(BUF) + (16 - ctypes.addressof(BUF) % 16) % 16, V)


def test_decode_refuses_bad_arguments(lib):
    f = lib.kda_decode
    f.argtypes = [V] * 7 + [I] * 3 + [U64]
    assert f(None, P, P, P, P, P, P, 1, 1, 128, 0) == 1
    assert b"null" in lib.kda_last_error()
    assert f(P, P, P, P, P, P, P, 1, 1, 64, 0) == 2
    assert f(P, P, P, P, P, P, P, 0, 1, 128, 0) == 1
    mis = ctypes.cast(P.value + 4, V)
    assert f(mis, P, P, P, P, P, P, 1, 1, 128, 0) == 1
    assert b"aligned" in lib.kda_last_error()


def test_decode_k_refuses_k_zero_and_k_above_limit(lib):
    f = lib.kda_decode_k
    f.argtypes = [V] * 7 + [I] * 4 + [V, I, U64]
    assert f(P, P, P, P, P, P, P, 1, 0, 1, 128, None, 0, 0) == 1
    assert b"k = 0" in lib.kda_last_error()
    assert f(P, P, P, P, P, P, P, 1, 9, 1, 128, None, 0, 0) == 1
    assert f(P, P, P, P, P, P, P, 1, 4, 1, 128, None, 5, 0) == 1   # n_snap > k
    assert f(P, P, P, P, P, P, P, 1, 4, 1, 128, None, 2, 0) == 1   # NULL snapshot list
    arr = (V * 1)(P.value)
    assert f(P, P, P, P, P, P, P, 1, 4, 1, 128, ctypes.cast(arr, V), 1, 0) == 1  # aliases state


def test_prefill_refuses_bad_arguments(lib):
    f = lib.kda_prefill
    f.argtypes = [V] * 7 + [I, I, I, F, I, I, I, ctypes.c_int64, V, I, V, SZ, U64]
    ok = dict(t=100, t_pad=128, chunk=64, heads=2, hd=128, dt=1, stride=256)

    def call(**kw):
        a = dict(ok, **kw)
        return f(P, P, P, P, P, P, P, a["t"], a["t_pad"], a["chunk"], 0.0, a["heads"], a["hd"],
                 a["dt"], a["stride"], None, 1, None, 0, 0)
    assert call(chunk=48) == 2
    assert call(chunk=256) == 2
    assert call(chunk=128) == 3        # a supported width: refused only for the workspace
    assert call(hd=64) == 2
    assert call(t=0) == 1
    assert call(t=200) == 1            # t > t_pad
    assert call(dt=7) == 1
    assert call(stride=100) == 1       # stride < heads * 128
    assert call(stride=260) == 1       # stride not a multiple of 16 bytes
    # packed sequences take no padding
    assert f(P, P, P, P, P, P, P, 100, 128, 64, 0.0, 2, 128, 1, 256, P, 1, None, 0, 0) == 1


def test_conv_refuses_bad_arguments(lib):
    f = lib.kda_conv_silu_l2
    f.argtypes = [V] * 4 + [I, I, V, I, F, I, I, U64]
    assert f(P, P, P, P, 4, 1, None, 5, 1e-6, 1, 128, 0) == 2      # conv_kernel > 4
    assert f(P, P, P, P, 4, 1, None, 0, 1e-6, 1, 128, 0) == 2
    assert f(P, P, P, P, 0, 1, None, 4, 1e-6, 1, 128, 0) == 1      # no tokens
    assert f(P, P, P, P, 4, 1, None, 4, -1.0, 1, 128, 0) == 1      # negative eps
    assert f(None, P, P, P, 4, 1, None, 4, 1e-6, 1, 128, 0) == 1


def test_fault_injection_hook_reports_launch_failure(lib, monkeypatch):
    """KDA_FAULT_INJECT=launch makes a valid call fail as a launch would,
    before anything reaches the device."""
    f = lib.kda_decode
    f.argtypes = [V] * 7 + [I] * 3 + [U64]
    monkeypatch.setenv("KDA_FAULT_INJECT", "launch")
    assert f(P, P, P, P, P, P, P, 1, 1, 128, 0) == 4
    assert b"injected" in lib.kda_last_error()


def test_workspace_size_is_queryable(lib):
    f = lib.kda_prefill_workspace_size
    f.restype = SZ
    f.argtypes = [ctypes.c_int64, I, I, I, I, I]
    big = f(8192, 1, 64, 32, 128, 1)          # BF16, chunk 64: tensor-core path
    # per (chunk, head): FP16 [Ktil; Qtil] 32 KiB, [T; P] 16 KiB, Khat^T 16 KiB, dec 512 B
    assert big >= (8192 // 64) * 32 * (32768 + 16384 + 16384 + 512)
    # FP32 inputs take the same path after FP16 copies of q, k, v (2 B each)
    # made in the workspace, 256-byte aligned after the rest
    f32 = f(8192, 1, 64, 32, 128, 0)
    assert f32 == ((big + 255) & ~255) + 3 * 8192 * 32 * 128 * 2
    # BF16 inputs take the tensor-core path (64-token steps) at every width
    assert f(8192, 1, 16, 32, 128, 1) == big and f(8192, 1, 128, 32, 128, 1) == big
    assert f(8192, 1, 64, 32, 64, 1) == 0     # invalid head_dim


def test_prefill_refuses_a_small_workspace(lib):
    f = lib.kda_prefill
    f.argtypes = [V] * 7 + [I, I, I, F, I, I, I, ctypes.c_int64, V, I, V, SZ, U64]
    assert f(P, P, P, P, P, P, P, 128, 128, 64, 0.0, 2, 128, 1, 256, None, 1, P, 64, 0) == 3
    assert b"workspace" in lib.kda_last_error()


def test_static_workspace_refuses_like_prefill(lib):
    """kda_prefill_static_ws checks its arguments as kda_prefill does, before
    its workspace limit, and returns the same status for the same bad call."""
    pf = lib.kda_prefill
    pf.argtypes = [V] * 7 + [I, I, I, F, I, I, I, ctypes.c_int64, V, I, V, SZ, U64]
    sf = lib.kda_prefill_static_ws
    sf.argtypes = [V] * 7 + [I, I, I, F, I, I, I, ctypes.c_int64, V, I, U64]
    cases = [dict(t=200, t_pad=128), dict(t=0), dict(chunk=48), dict(hd=64), dict(dt=7),
             dict(stride=100), dict(t=100, t_pad=128, cu=True), dict(t_pad=1 << 30, n=4)]
    for c in cases:
        a = dict(t=100, t_pad=128, chunk=64, heads=2, hd=128, dt=1, stride=256, cu=False, n=1)
        a.update(c)
        cu = P if a["cu"] else None
        want = pf(P, P, P, P, P, P, P, a["t"], a["t_pad"], a["chunk"], 0.0, a["heads"], a["hd"],
                  a["dt"], a["stride"], cu, a["n"], None, 0, 0)
        got = sf(P, P, P, P, P, P, P, a["t"], a["t_pad"], a["chunk"], 0.0, a["heads"], a["hd"],
                 a["dt"], a["stride"], cu, a["n"], 0)
        assert want in (1, 2) and got == want, (c, want, got)
        assert b"kda_prefill_static_ws" in lib.kda_last_error()


def test_o_norm_refuses_bad_arguments(lib):
    f = lib.kda_o_norm_gated
    f.argtypes = [V] * 4 + [ctypes.c_int64, I, I, F, U64]
    assert f(None, P, P, P, 4, 2, 128, 1e-6, 0) == 1
    assert f(None, None, None, None, 0, 2, 128, 1e-6, 0) == 0  # zero rows: nothing to touch
    assert f(P, P, P, P, 4, 2, 64, 1e-6, 0) == 2       # head_dim
    assert f(P, P, P, P, -1, 2, 128, 1e-6, 0) == 1     # rows
    assert f(P, P, P, P, 4, 0, 128, 1e-6, 0) == 1      # heads
    assert f(P, P, P, P, 4, 2, 128, -1.0, 0) == 1      # eps
    assert f(ctypes.c_void_p(P.value + 4), P, P, P, 4, 2, 128, 1e-6, 0) == 1  # core alignment
    assert b"kda_o_norm_gated" in lib.kda_last_error()


def test_gate_refuses_bad_arguments(lib):
    f = lib.kda_gate
    f.argtypes = [V, ctypes.c_int64, V, V, F, V, ctypes.c_int64, V, V, I, ctypes.c_int64, I, I,
                  U64]
    ok = (P, 256, P, P, -5.0, P, 2, P, P, 1, 4, 2, 128, 0)
    bad = lambda **kw: f(*[kw.get(k, v) for k, v in zip(
        ("g", "gs", "dt", "al", "lb", "b", "bs", "go", "bo", "dt_", "rows", "h", "hd", "s"), ok)])
    assert bad(hd=64) == 2                          # head_dim
    assert bad(rows=-1) == 1 and bad(h=0) == 1      # rows, heads
    assert bad(dt_=2) == 1                          # out_dtype
    assert bad(lb=0.0) == 1 and bad(lb=1.0) == 1    # the bound must be negative
    assert bad(gs=128) == 1 and bad(gs=260) == 1    # pitch below heads*128, not a multiple of 8
    assert bad(bs=1) == 1                           # b pitch below heads
    assert bad(g=None) == 1                         # null pointer
    assert bad(go=ctypes.c_void_p(P.value + 4)) == 1  # g_out alignment
    assert bad(rows=0, g=None, b=None, go=None, bo=None) == 0  # zero rows: nothing to touch
    assert b"kda_gate" in lib.kda_last_error()


def test_prefill_gated_refuses_bad_arguments(lib):
    f = lib.kda_prefill_gated
    f.argtypes = [V] * 5 + [ctypes.c_int64, V, V, F, V, ctypes.c_int64, V, I, I, I, I,
                            ctypes.c_int64, V, I, V, ctypes.c_size_t, U64]
    big = 1 << 40
    ok = (P, P, P, P, P, 512, P, P, -5.0, P, 4, P, 100, 128, 4, 128, 512, None, 1, P, big, 0)
    names = ("S", "q", "k", "v", "g", "gs", "dt", "al", "lb", "b", "bs", "o", "t", "tp", "h",
             "hd", "st", "cu", "n", "ws", "wsb", "s")
    bad = lambda **kw: f(*[kw.get(k, v) for k, v in zip(names, ok)])
    assert bad(hd=64) == 2                                   # head_dim
    assert bad(t=0) == 1 and bad(tp=99) == 1                 # 1 <= t <= t_pad
    assert bad(cu=P) == 1                                    # packed rows take no padding
    assert bad(h=0) == 1 and bad(n=0) == 1                   # heads, sequences
    assert bad(st=500) == 1 and bad(st=516) == 1             # q/k/v pitch
    assert bad(gs=500) == 1 and bad(gs=516) == 1             # g_raw pitch
    assert bad(bs=3) == 1                                    # b_raw pitch below heads
    assert bad(lb=0.0) == 1 and bad(lb=float("-inf")) == 1   # the bound: finite, negative
    assert bad(dt=None) == 1 and bad(b=None) == 1            # null pointers
    assert bad(g=ctypes.c_void_p(P.value + 2)) == 1          # g_raw alignment
    assert bad(wsb=1024) == 3 and bad(ws=None) == 3          # workspace too small / missing
    assert b"kda_prefill_gated" in lib.kda_last_error()


def test_prefill_o_norm_refuses_bad_arguments(lib):
    f = lib.kda_prefill_o_norm
    f.argtypes = [V] * 7 + [ctypes.c_int64, V, F, V, ctypes.c_int64, I, I, I, I, I, I,
                            ctypes.c_int64, V, I, V, ctypes.c_size_t, U64]
    big = 1 << 40
    ok = (P, P, P, P, P, P, P, 512, P, 1e-6, P, 512, 100, 128, 64, 4, 128, 1, 512, None, 1, P,
          big, 0)
    names = ("S", "q", "k", "v", "g", "b", "gate", "gs", "w", "eps", "out", "os", "t", "tp",
             "c", "h", "hd", "dt", "st", "cu", "n", "ws", "wsb", "s")
    bad = lambda **kw: f(*[kw.get(k, v) for k, v in zip(names, ok)])
    assert bad(hd=64) == 2 and bad(c=48) == 2                # head_dim, chunk width
    assert bad(dt=0) == 2                                    # FP32 inputs: no fused norm
    assert bad(t=0) == 1 and bad(tp=99) == 1                 # 1 <= t <= t_pad
    assert bad(cu=P) == 1                                    # packed rows take no padding
    assert bad(gate=None) == 1 and bad(w=None) == 1 and bad(out=None) == 1
    assert bad(gate=ctypes.c_void_p(P.value + 8)) == 1       # gate alignment (16 bytes)
    assert bad(out=ctypes.c_void_p(P.value + 8)) == 1        # out alignment (16 bytes)
    assert bad(w=ctypes.c_void_p(P.value + 4)) == 1          # w alignment (8 bytes)
    assert bad(gs=500) == 1 and bad(gs=516) == 1             # gate pitch
    assert bad(os=500) == 1 and bad(os=516) == 1             # out pitch
    assert bad(eps=-1.0) == 1 and bad(eps=float("inf")) == 1
    assert bad(wsb=1024) == 3 and bad(ws=None) == 3          # workspace too small / missing
    assert b"kda_prefill_o_norm" in lib.kda_last_error()


def test_conv_k_refuses_bad_arguments(lib):
    f = lib.kda_conv_silu_l2_k
    f.argtypes = [V] * 4 + [I, I, I, F, I, I, V, I, U64]
    assert f(P, P, P, P, 2, 0, 4, 1e-6, 1, 128, None, 0, 0) == 1      # k = 0
    assert f(P, P, P, P, 2, 9, 4, 1e-6, 1, 128, None, 0, 0) == 1      # k above KDA_MAX_K
    assert f(P, P, P, P, 2, 3, 4, 1e-6, 1, 128, None, 4, 0) == 1      # n_snap > k
    assert f(P, P, P, P, 2, 3, 4, 1e-6, 1, 128, None, 2, 0) == 1      # snapshots NULL
    assert f(P, P, P, P, 2, 3, 5, 1e-6, 1, 128, None, 0, 0) == 2      # conv_kernel
    assert b"kda_conv_silu_l2_k" in lib.kda_last_error()
