"""kda_prefill_static_ws, the prefill entry point that allocates nothing.

Callers that cannot allocate device memory themselves (a plugin handed only
input and output pointers by its host application, or a serving loop that
forbids cudaMalloc because it can synchronise the device) run the prefill
through this entry point; its workspace is a fixed array the library owns.
These tests call it through the C ABI and check it against kda_prefill with a
caller-owned workspace.  This file is collected last on purpose.
"""

import ctypes

import pytest
import torch

import kda_workloads as wl
from _util import kda

pytestmark = pytest.mark.gpu


def _static_fn(K):
    f = K.LIB.kda_prefill_static_ws
    c = ctypes
    f.argtypes = ([c.c_void_p] * 7 + [c.c_int, c.c_int, c.c_int, c.c_float, c.c_int, c.c_int,
                                      c.c_int, c.c_int64, c.c_void_p, c.c_int, c.c_uint64])
    f.restype = c.c_int
    return f


def _inputs(seed, T, H):
    d = wl.prefill(seed=seed, t=T, heads=H, dtype=torch.bfloat16)
    return {n: d[n].cuda() for n in ("q", "k", "v", "g", "beta", "state")}


def test_static_workspace_matches_caller_workspace_two_calls_in_a_row():
    K = kda()
    f = _static_fn(K)
    stream = torch.cuda.current_stream().cuda_stream
    for seed, T, H in ((1, 700, 4), (2, 300, 8)):
        d = _inputs(seed, T, H)
        S_ref = d["state"].clone()
        o_ref = torch.zeros((T, H, 128), device="cuda")
        ws = torch.empty(K.kda_prefill_workspace_size(T, 1, 64, H), dtype=torch.uint8,
                         device="cuda")
        K.kda_prefill(S_ref, d["q"], d["k"], d["v"], d["g"], d["beta"], o_ref, T, 64,
                      workspace=ws)
        S = d["state"].clone()
        o = torch.zeros((T, H, 128), device="cuda")
        st = f(S.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
               d["g"].data_ptr(), d["beta"].data_ptr(), o.data_ptr(), T, T, 64, 0.0, H, 128,
               1, H * 128, None, 1, stream)
        assert st == 0, K.LIB.kda_last_error().decode()
        K.kda_sync_status()
        # the same kernels on the same inputs: bit-identical to the call with
        # a caller workspace (a layout slip in the static array would show)
        assert torch.equal(o, o_ref)
        assert torch.equal(S, S_ref)


def test_static_workspace_refuses_a_call_beyond_its_size():
    K = kda()
    f = _static_fn(K)
    T, H = 8192, 32
    d = _inputs(3, 64, H)  # the refusal happens before any pointer is used
    S = d["state"].clone()
    st = f(S.data_ptr(), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
           d["g"].data_ptr(), d["beta"].data_ptr(), S.data_ptr(), T, T, 64, 0.0, H, 128, 1,
           H * 128, None, 1, torch.cuda.current_stream().cuda_stream)
    assert st == 3
    assert b"KDA_STATIC_WORKSPACE_BYTES" in K.LIB.kda_last_error()
    torch.cuda.synchronize()
    assert torch.equal(S, d["state"])
