"""kda_prefill through the fused prepare + scan grid (BF16, chunk 64, one
sequence of 32 heads: few enough (sequence, head) chains that the library
runs one cooperative grid in which the transposed scan consumes each chunk
as soon as another SM has prepared it), against the FP64 oracle, against the
two-kernel path (KDA_PREFILL_IMPL=unfused), and for pad-fill independence."""

import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu

H = 32  # 32 chains on one sequence: the fused grid's regime


def inputs(seed, t, g_low=-5.0):
    gen = torch.Generator().manual_seed(seed)
    d = wl.core_inputs(gen, (t,), H, torch.bfloat16, g_low=g_low)
    d["state"] = wl.state(gen, (1,), H, 0.02)
    return d


def run(K, d, t, t_pad=None, pad_fill=float("nan"), cu=False, workspace=None):
    """Rows [t, t_pad) hold pad_fill (the caller's tail; NaN by default)."""
    t_pad = t_pad or t
    dev = {n: wl.pad_rows(d[n][:t], t_pad, pad_fill).cuda()
           for n in ("q", "k", "v", "g", "beta")}
    S = d["state"].clone().cuda()
    o = torch.full((t_pad, H, 128), 12345.0, device="cuda")
    if cu:
        cuv = torch.tensor([0, t], dtype=torch.int32, device="cuda")
        K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 64,
                      cu_seqlens=cuv, workspace=workspace)
    else:
        K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 64,
                      pad_fill=pad_fill, workspace=workspace)
    K.kda_sync_status()
    return o, S


def oracle_all_heads(orc, d, t):
    return orc.prefill(d["q"][:t], d["k"][:t], d["v"][:t], d["g"][:t], d["beta"][:t],
                       d["state"][0])


@pytest.mark.parametrize("t,g_low", [(1000, -5.0), (777, -0.05), (64, -5.0), (1, -5.0),
                                     (130, -10.0), (130, -15.0), (200, -20.0)])
def test_fused_grid_matches_oracle(orc, t, g_low):
    """Every head and output row: whole and ragged chunk counts, one-chunk
    sequences (one token: the row walk), slow decay (the state carries across
    every chunk), and steep decays: down to -10 the 16-token tensor-core
    blocks, beyond it the exact per-pair products."""
    K = kda()
    d = inputs(100 + t, t, g_low)
    o, S = run(K, d, t)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_fused_packed_single_sequence_matches_oracle(orc):
    """The packed form (cu_seqlens = [0, t]) takes the fused grid as well."""
    K = kda()
    t = 517
    d = inputs(7, t)
    o, S = run(K, d, t, cu=True)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("t", [640, 1000])
def test_fused_and_two_kernel_paths_agree(orc, monkeypatch, t):
    """The fused grid and prepare followed by the scan kernel run the same
    prepare and scan arithmetic, only scheduled differently: their results are
    identical bit for bit, and within the tolerance of the oracle."""
    K = kda()
    d = inputs(13, t, g_low=-1.0)
    o_f, S_f = run(K, d, t)
    monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    o_u, S_u = run(K, d, t)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o_f, o_ref) < TOL_PREFILL
    assert rel_err(S_f[0], S_ref) < TOL_PREFILL
    assert torch.equal(o_f, o_u) and torch.equal(S_f, S_u)


def test_fused_pad_fill_has_no_effect():
    """Bit-identical o[:t] and state for pad_fill 0, NaN and 1e30 on the fused
    grid; rows [t, t_pad) of o are never written."""
    K = kda()
    t, t_pad = 1000, 1024
    d = inputs(3, t_pad)
    runs = [run(K, d, t, t_pad=t_pad, pad_fill=f) for f in (0.0, float("nan"), 1e30)]
    o0, S0 = runs[0]
    assert torch.isfinite(o0[:t]).all() and torch.isfinite(S0).all()
    for o, S in runs[1:]:
        assert torch.equal(o[:t], o0[:t])
        assert torch.equal(S, S0)
        assert (o[t:] == 12345.0).all()


def test_fused_stale_workspace_and_repeated_calls(orc):
    """The grid's ready flags are cleared by every call: a workspace whose
    bytes are all 0xFF (every flag set) still gives the oracle's result, and
    two calls on the same workspace give the same bits whichever SM prepared
    which chunk."""
    K = kda()
    t = 900
    d = inputs(5, t)
    need = K.kda_prefill_workspace_size(t, 1, 64, H)
    ws = torch.full((need,), 255, dtype=torch.uint8, device="cuda")
    o1, S1 = run(K, d, t, workspace=ws)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o1, o_ref) < TOL_PREFILL
    assert rel_err(S1[0], S_ref) < TOL_PREFILL
    o2, S2 = run(K, d, t, workspace=ws)
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


@pytest.mark.parametrize("packed", [True, False])
def test_fused_grid_two_sequences(orc, packed):
    """Two sequences of 16 heads (32 chains: the fused grid) whose chunk
    counts are not multiples of four, so the second sequence's chunks start
    inside a group of four ready flags; packed and uniform forms."""
    K = kda()
    Hs = 16
    lengths = [300, 517] if packed else [517, 517]
    gen = torch.Generator().manual_seed(77 + int(packed))
    tot = sum(lengths)
    d = wl.core_inputs(gen, (tot,), Hs, torch.bfloat16)
    S0 = wl.state(gen, (2,), Hs, 0.02)
    S = S0.clone().cuda()
    dev = {n: d[n].cuda() for n in d}
    o = torch.zeros((tot, Hs, 128), device="cuda")
    if packed:
        cu = torch.tensor([0, lengths[0], tot], dtype=torch.int32, device="cuda")
        K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, tot, 64,
                      cu_seqlens=cu)
    else:
        t = lengths[0]
        view = {n: dev[n].view((2, t) + tuple(dev[n].shape[1:])) for n in dev}
        K.kda_prefill(S, view["q"], view["k"], view["v"], view["g"], view["beta"],
                      o.view(2, t, Hs, 128), t, 64)
    K.kda_sync_status()
    a = 0
    for n, L in enumerate(lengths):
        b = a + L
        o_ref, S_ref = orc.prefill(d["q"][a:b], d["k"][a:b], d["v"][a:b], d["g"][a:b],
                                   d["beta"][a:b], S0[n])
        assert rel_err(o[a:b], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL
        a = b


@pytest.mark.parametrize("impl", ["fused", "unfused"])
def test_steep_decay_matches_oracle_on_both_paths(orc, monkeypatch, impl):
    """g in [-20, 0]: every chunk is steeper than the tensor-core blocks allow
    and takes the exact products, on the fused grid and on the two kernels."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    t = 300
    d = inputs(77, t, g_low=-20.0)
    o, S = run(K, d, t)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_bounded_ready_wait_runs_out_and_reports(orc, monkeypatch):
    """The chains' wait on a ready flag is bounded.  KDA_FAULT_INJECT=ready_wait
    makes the prepare CTAs release no flag and cuts the wait to a few
    milliseconds: every chain gives up, the kernel still returns, and
    kda_sync_status reports KDA_ERR_DEVICE with the timeout text.  No chain
    writes its state or o, and the next call on the same context is correct."""
    K = kda()
    t = 256
    d = inputs(21, t)
    dev = {n: d[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    S = d["state"].clone().cuda()
    o = torch.full((t, H, 128), 12345.0, device="cuda")
    monkeypatch.setenv("KDA_FAULT_INJECT", "ready_wait")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 64)
    with pytest.raises(K.KdaError) as err:
        K.kda_sync_status()
    assert err.value.status == 5  # KDA_ERR_DEVICE
    assert "a bounded wait timed out" in str(err.value)
    assert torch.equal(S.cpu(), d["state"])
    assert (o == 12345.0).all()
    monkeypatch.delenv("KDA_FAULT_INJECT")
    K.kda_sync_status()  # the status word was cleared by the read above
    o2, S2 = run(K, d, t)
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    assert rel_err(o2, o_ref) < TOL_PREFILL
    assert rel_err(S2[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("impl", ["fused", "unfused"])
@pytest.mark.parametrize("t", [1, 5, 8])
def test_short_sequences_on_the_tensor_core_kernels(orc, monkeypatch, impl, t):
    """Sequences of at most 8 tokens on the tensor-core kernels: q, k, v as
    slices of one wider buffer (a contiguous short sequence takes the row
    walk instead).  One ragged chunk of t rows against the oracle."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    d = inputs(500 + t, t)
    hd = H * 128
    qkv = torch.cat([d[n].reshape(t, hd) for n in ("q", "k", "v")], dim=1).cuda()
    # as_strided keeps the row stride of a one-row view (a plain view may not)
    q, k, v = (torch.as_strided(qkv, (t, H, 128), (3 * hd, 128, 1), i * hd) for i in range(3))
    S = d["state"].clone().cuda()
    o = torch.empty((t, H, 128), device="cuda")
    assert q.stride(0) == 3 * hd
    K.kda_prefill(S, q, k, v, d["g"].cuda(), d["beta"].cuda(), o, t, 64)
    K.kda_sync_status()
    o_ref, S_ref = oracle_all_heads(orc, d, t)
    e_o, e_s = rel_err(o, o_ref), rel_err(S[0], S_ref)
    assert e_o < TOL_PREFILL and e_s < TOL_PREFILL
    assert e_s > 1e-6  # the FP16 scan operands' rounding: not the FP32 row walk
