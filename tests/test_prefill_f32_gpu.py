"""kda_prefill with FP32 inputs on the tensor-core kernels: q, k and v are
rounded to FP16 copies in the workspace (11 significant bits, the precision
of the TF32 and FP16 operands they become), g and beta are read as FP32.
Checked against the FP64 oracle on the same FP32 inputs on the fused grid and
the two-kernel path, bit for bit between the two paths, for pad-fill
independence, packed batches, strided q/k/v rows, steep decays, scaled values
and state, and against the FP32 SIMT kernel."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu

H = 32  # one sequence of 32 heads: the fused grid's regime


def inputs(seed, t, g_low=-5.0, heads=H):
    gen = torch.Generator().manual_seed(seed)
    d = wl.core_inputs(gen, (t,), heads, torch.float32, g_low=g_low)
    d["state"] = wl.state(gen, (1,), heads, 0.02)
    return d


def run(K, d, t, t_pad=None, pad_fill=float("nan"), chunk=64):
    t_pad = t_pad or t
    heads = d["q"].shape[1]
    dev = {n: wl.pad_rows(d[n][:t], t_pad, pad_fill).cuda()
           for n in ("q", "k", "v", "g", "beta")}
    S = d["state"].clone().cuda()
    o = torch.full((t_pad, heads, 128), 12345.0, device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, chunk,
                  pad_fill=pad_fill)
    K.kda_sync_status()
    return o, S


def oracle(orc, d, t):
    return orc.prefill(d["q"][:t], d["k"][:t], d["v"][:t], d["g"][:t], d["beta"][:t],
                       d["state"][0])


@pytest.mark.parametrize("impl", ["fused", "unfused"])
@pytest.mark.parametrize("t,g_low", [(1000, -5.0), (777, -0.05), (64, -5.0), (9, -5.0),
                                     (130, -10.0), (130, -15.0), (200, -20.0)])
def test_f32_inputs_match_oracle(orc, monkeypatch, impl, t, g_low):
    """Whole and ragged chunk counts, the shortest sequence past the row
    walk, slow decay, and the 16-token blocks and exact products of steep
    decays, with g read in FP32."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    d = inputs(300 + t, t, g_low)
    o, S = run(K, d, t)
    o_ref, S_ref = oracle(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_f32_fused_and_two_kernel_paths_agree(monkeypatch):
    K = kda()
    d = inputs(31, 1000, g_low=-1.0)
    o_f, S_f = run(K, d, 1000)
    monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    o_u, S_u = run(K, d, 1000)
    assert torch.equal(o_f, o_u) and torch.equal(S_f, S_u)


@pytest.mark.parametrize("t,t_pad", [(1000, 1024), (100, 128)])
def test_f32_pad_fill_has_no_effect(t, t_pad):
    """Bit-identical o[:t] and state for pad_fill 0, NaN and 1e30 (FP16 inf
    once converted); rows [t, t_pad) of o are never written."""
    K = kda()
    d = inputs(5, t_pad)
    runs = [run(K, d, t, t_pad=t_pad, pad_fill=f) for f in (0.0, float("nan"), 1e30)]
    o0, S0 = runs[0]
    assert torch.isfinite(o0[:t]).all() and torch.isfinite(S0).all()
    for o, S in runs[1:]:
        assert torch.equal(o[:t], o0[:t])
        assert torch.equal(S, S0)
        assert (o[t:] == 12345.0).all()


def test_f32_packed_varlen_matches_per_sequence_oracle(orc):
    """Packed FP32 sequences (6 x 4 chains), with an empty one, a one-token
    one and lengths that are not whole chunks."""
    K = kda()
    lengths = [70, 0, 1, 64, 133, 9]
    heads = 4
    gen = torch.Generator().manual_seed(17)
    tot = sum(lengths)
    d = wl.core_inputs(gen, (tot,), heads, torch.float32)
    S0 = wl.state(gen, (len(lengths),), heads, 0.02)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    dev = {n: d[n].cuda() for n in d}
    S = S0.clone().cuda()
    o = torch.zeros((tot, heads, 128), device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, tot, 64,
                  cu_seqlens=cu.cuda())
    K.kda_sync_status()
    for n, L in enumerate(lengths):
        a, b = int(cu[n]), int(cu[n + 1])
        if L == 0:
            assert torch.equal(S[n].cpu(), S0[n])
            continue
        o_ref, S_ref = orc.prefill(d["q"][a:b], d["k"][a:b], d["v"][a:b], d["g"][a:b],
                                   d["beta"][a:b], S0[n])
        assert rel_err(o[a:b], o_ref) < TOL_PREFILL, n
        assert rel_err(S[n], S_ref) < TOL_PREFILL, n


def test_f32_strided_qkv_rows(orc):
    """q, k and v as column slices of one FP32 [T, 3 * heads * 128] buffer
    (the front end's layout): the conversion reads rows qkv_row_stride apart."""
    K = kda()
    t, heads = 300, 8
    d = inputs(41, t, heads=heads)
    hd = heads * 128
    qkv = torch.cat([d[n].reshape(t, hd) for n in ("q", "k", "v")], dim=1).cuda()
    q, k, v = (qkv[:, i * hd:(i + 1) * hd].view(t, heads, 128) for i in range(3))
    S = d["state"].clone().cuda()
    o = torch.empty((t, heads, 128), device="cuda")
    K.kda_prefill(S, q, k, v, d["g"].cuda(), d["beta"].cuda(), o, t, 64)
    K.kda_sync_status()
    o_ref, S_ref = oracle(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("v_scale,s_scale", [(1e-4, 1e-4), (1e3, 1e3), (1e-4, 1.0)])
def test_f32_scaled_values_and_state(orc, v_scale, s_scale):
    """The FP16 domain of the scan's operands (and now of the v copy): v and
    the initial state scaled by 1e-4 and 1e3."""
    K = kda()
    t = 300
    d = inputs(61, t)
    d["v"] = d["v"] * v_scale
    d["state"] = d["state"] * s_scale
    o, S = run(K, d, t)
    o_ref, S_ref = oracle(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_f32_tensor_core_and_simt_kernels_agree(orc, monkeypatch):
    """The SIMT kernel (KDA_PREFILL_IMPL=simt) keeps FP32 arithmetic
    throughout and tracks the oracle at 1e-5; the tensor-core path stays
    within the prefill tolerance of both."""
    K = kda()
    t, heads = 200, 4
    d = inputs(71, t, heads=heads)
    o_tc, S_tc = run(K, d, t)
    monkeypatch.setenv("KDA_PREFILL_IMPL", "simt")
    o_si, S_si = run(K, d, t)
    o_ref, S_ref = oracle(orc, d, t)
    assert rel_err(o_si, o_ref) < 1e-5 and rel_err(S_si[0], S_ref) < 1e-5
    assert rel_err(o_tc, o_ref) < TOL_PREFILL and rel_err(S_tc[0], S_ref) < TOL_PREFILL
    assert rel_err(o_tc, o_si.double().cpu().numpy()) < TOL_PREFILL
