"""kda_prefill_gated (the forget gate and beta formed inside the prepare
kernel from g_raw, dt_bias, a_log and b_raw) against the FP64 oracle: the
oracle's gate, then its token recurrence.  The fused grid and the two-kernel
path, packed sequences, strided views of wider projections, and rows past t
that never reach the arithmetic."""

import os

import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu


def reference(orc, d, rows, H):
    """The oracle's g and beta from the raw inputs of the first `rows` rows."""
    g, beta = orc.gate(d["g_raw"][:rows, :H * 128], d["dt_bias"], d["a_log"],
                       d["gate_lower_bound"], d["b_raw"][:rows, :H])
    return g, beta


def run(K, d, t, H, t_pad=None, cu=None, pad_value=None, state=None):
    t_pad = t_pad or t
    dev = {}
    for n in ("q", "k", "v"):
        dev[n] = wl.pad_rows(d[n][:t], t_pad, float("nan") if pad_value is None else pad_value
                             ).cuda()
    for n in ("g_raw", "b_raw"):
        dev[n] = wl.pad_rows(d[n][:t], t_pad, float("nan") if pad_value is None else pad_value
                             ).cuda()
    S = (d["state"] if state is None else state).clone().cuda()
    o = torch.full((t_pad, H, 128), 12345.0, device="cuda")
    K.kda_prefill_gated(S, dev["q"], dev["k"], dev["v"], dev["g_raw"], d["dt_bias"].cuda(),
                        d["a_log"].cuda(), dev["b_raw"], o, t, d["gate_lower_bound"],
                        cu_seqlens=cu)
    K.kda_sync_status()
    return o, S


@pytest.mark.parametrize("t", [1000, 130, 64, 1])
@pytest.mark.parametrize("impl", ["fused", "unfused"])
def test_gated_prefill_matches_oracle(orc, monkeypatch, t, impl):
    """One sequence of 32 heads (the fused grid's regime; KDA_PREFILL_IMPL=
    unfused pins the two kernels): every head and row against the oracle."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    H = 32
    d = wl.prefill_gated(seed=200 + t, t=t, heads=H)
    o, S = run(K, d, t, H)
    g, beta = reference(orc, d, t, H)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], g, beta, d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("impl", ["fused", "unfused"])
def test_gated_prefill_steep_lower_bound(orc, monkeypatch, impl):
    """gate_lower_bound -20: the gate reaches decays far steeper than the
    tensor-core blocks allow; those chunks take the exact products."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    H, t = 32, 200
    d = wl.prefill_gated(seed=17, t=t, heads=H)
    d["gate_lower_bound"] = -20.0
    o, S = run(K, d, t, H)
    g, beta = reference(orc, d, t, H)
    assert float(g.min()) < -10.0  # the steep path is exercised
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], g, beta, d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_gated_prefill_rows_past_t_unused(orc):
    """t = 1000 of 1024 rows: o[:t] and the final state are bit-identical
    whatever the rows past t hold (NaN or 0 in q, k, v, g_raw and b_raw),
    and rows past t of o are not written."""
    K = kda()
    H, t, t_pad = 32, 1000, 1024
    d = wl.prefill_gated(seed=7, t=t, heads=H)
    o_nan, S_nan = run(K, d, t, H, t_pad=t_pad, pad_value=float("nan"))
    o_zero, S_zero = run(K, d, t, H, t_pad=t_pad, pad_value=0.0)
    assert torch.equal(o_nan[:t], o_zero[:t]) and torch.equal(S_nan, S_zero)
    assert torch.all(o_nan[t:] == 12345.0)
    g, beta = reference(orc, d, t, H)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], g, beta, d["state"][0])
    assert rel_err(o_nan[:t], o_ref) < TOL_PREFILL


def test_gated_prefill_packed_strided(orc):
    """Three packed sequences of 4 heads (one of them empty, one shorter than
    a chunk) with q, k, v views of one [T, 3*H*128] buffer and g_raw / b_raw
    views of wider projections; each sequence starts from its own state."""
    K = kda()
    H = 4
    lengths = [300, 0, 45]
    T = sum(lengths)
    d = wl.prefill_gated(seed=31, t=T, heads=H, g_pitch_extra=64, b_pitch_extra=3)
    gen = torch.Generator().manual_seed(32)
    S0 = wl.state(gen, (len(lengths),), H, 0.02)
    qkv = torch.cat([d[n].reshape(T, H * 128) for n in ("q", "k", "v")], dim=1).cuda()
    q, k, v = (qkv[:, i * H * 128:(i + 1) * H * 128].view(T, H, 128) for i in range(3))
    g_raw, b_raw = d["g_raw"].cuda(), d["b_raw"].cuda()
    assert g_raw.stride(0) == H * 128 + 64 and b_raw.stride(0) == H + 3
    cu = torch.tensor([0, 300, 300, 345], dtype=torch.int32, device="cuda")
    S = S0.clone().cuda()
    o = torch.zeros((T, H, 128), device="cuda")
    K.kda_prefill_gated(S, q, k, v, g_raw[:, :H * 128], d["dt_bias"].cuda(), d["a_log"].cuda(),
                        b_raw[:, :H], o, T, d["gate_lower_bound"], cu_seqlens=cu)
    K.kda_sync_status()
    g, beta = reference(orc, d, T, H)
    start = 0
    for n, L in enumerate(lengths):
        if L == 0:
            assert torch.equal(S[n].cpu(), S0[n])  # an empty sequence leaves its state
            continue
        sl = slice(start, start + L)
        o_ref, S_ref = orc.prefill(d["q"][sl], d["k"][sl], d["v"][sl], g[sl], beta[sl], S0[n])
        assert rel_err(o[sl], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL
        start += L
