"""kda_prefill against the FP64 oracle (token recurrence), pad-fill
independence bit for bit (prefill_with_pad_fill: positions at or past t are
ignored in-kernel), packed variable-length batches, and the full-size prefill
workload on sampled heads."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu


def run_prefill(K, d, t, chunk, pad_fill=float("nan"), t_pad=None):
    """d holds host tensors [T, H, D] / [T, H]; pads to t_pad rows with
    pad_fill (NaN by default, to prove the kernels never read them) and runs
    one sequence."""
    T = d["q"].shape[0]
    t_pad = t_pad or T
    dev = {n: wl.pad_rows(d[n][:t], t_pad, pad_fill).cuda()
           for n in ("q", "k", "v", "g", "beta")}
    S = d["state"].clone().cuda()
    o = torch.full((t_pad,) + tuple(d["q"].shape[1:]), 12345.0, device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, chunk,
                  pad_fill=pad_fill)
    torch.cuda.synchronize()
    return o, S, dev


def test_tiny_config_matches_oracle(orc):
    """1 sequence, T=64, 2 heads, chunk 16, FP32, zero initial state."""
    K = kda()
    d = wl.tiny()
    o, S, _ = run_prefill(K, d, 64, 16)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("chunk,t", [(16, 77), (32, 100), (64, 200), (64, 64), (64, 1),
                                     (16, 16), (64, 129), (128, 300), (128, 77), (128, 128)])
def test_prefill_matches_oracle(orc, dtype, chunk, t):
    """Every chunk width the boundary accepts, whole and ragged last chunks,
    on the tensor-core kernels (64-token steps whatever the width; FP32
    inputs through their FP16 copies) or, for FP32 with t <= 8, the row
    walk."""
    K = kda()
    d = wl.prefill(seed=t + chunk, t=t, heads=3, chunk=chunk, dtype=dtype)
    o, S, _ = run_prefill(K, d, t, chunk)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("t,t_pad", [(8155, 8192), (8191, 8192), (100, 128), (1, 64)])
def test_pad_fill_has_no_effect(t, t_pad):
    """o[:t] and the final state are bit-identical for pad_fill 0, NaN and 1e30,
    and rows [t, t_pad) of o are never written."""
    K = kda()
    H = 4 if t_pad > 1000 else 2
    d = wl.prefill(seed=t, t=t_pad, heads=H, chunk=64, dtype=torch.bfloat16)
    runs = [run_prefill(K, d, t, 64, pad_fill=f, t_pad=t_pad)
            for f in (0.0, float("nan"), 1e30)]
    o0, S0, dev0 = runs[0]
    assert torch.isfinite(o0[:t]).all() and torch.isfinite(S0).all()
    for o, S, dev in runs[1:]:
        assert torch.equal(o[:t], o0[:t])
        assert torch.equal(S, S0)
        assert (o[t:] == 12345.0).all()
    # the caller's tails are left as they were (the library never writes them)
    assert torch.isnan(runs[1][2]["q"][t:].float()).all()
    assert (runs[2][2]["g"][t:].float() > 1e29).all()
    assert (dev0["beta"][t:].float() == 0).all()


def test_padded_run_equals_unpadded_run():
    K = kda()
    d = wl.prefill(seed=5, t=150, heads=2, chunk=64, dtype=torch.float32)
    o_a, S_a, _ = run_prefill(K, d, 150, 64, t_pad=150)
    o_b, S_b, _ = run_prefill(K, d, 150, 64, pad_fill=float("nan"), t_pad=192)
    assert torch.equal(o_a, o_b[:150]) and torch.equal(S_a, S_b)


def test_packed_varlen_matches_per_sequence_oracle(orc):
    """Packed sequences with cu_seqlens, including an empty one and lengths
    that are not whole chunks."""
    K = kda()
    lengths = [70, 0, 1, 64, 133]
    H = 2
    gen = torch.Generator().manual_seed(11)
    tot = sum(lengths)
    d = wl.core_inputs(gen, (tot,), H, torch.bfloat16)
    S0 = wl.state(gen, (len(lengths),), H, 0.02)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    dev = {n: d[n].cuda() for n in d}
    S = S0.clone().cuda()
    o = torch.zeros((tot, H, 128), device="cuda")
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
        assert rel_err(o[a:b], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("n_seqs", [128, 129])
def test_many_packed_sequences_match_per_sequence_oracle(orc, n_seqs):
    """Packed batches on both sides of prepare's shared-memory chunk map (it
    holds up to 128 sequences; larger batches search the map in device
    memory), with empty, one-token and whole-chunk sequences: hundreds of
    (sequence, head) chains on the two-kernel path."""
    K = kda()
    H = 2
    gen = torch.Generator().manual_seed(40 + n_seqs)
    lengths = torch.randint(0, 150, (n_seqs,), generator=gen).tolist()
    lengths[3], lengths[17], lengths[64], lengths[-1] = 0, 1, 64, 128
    tot = sum(lengths)
    d = wl.core_inputs(gen, (tot,), H, torch.bfloat16)
    S0 = wl.state(gen, (n_seqs,), H, 0.02)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    dev = {n: d[n].cuda() for n in d}
    S = S0.clone().cuda()
    o = torch.zeros((tot, H, 128), device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, tot, 64,
                  cu_seqlens=cu.cuda())
    K.kda_sync_status()
    S, o = S.cpu(), o.cpu()
    for n, L in enumerate(lengths):
        a, b = int(cu[n]), int(cu[n + 1])
        if L == 0:
            assert torch.equal(S[n], S0[n])
            continue
        o_ref, S_ref = orc.prefill(d["q"][a:b], d["k"][a:b], d["v"][a:b], d["g"][a:b],
                                   d["beta"][a:b], S0[n])
        assert rel_err(o[a:b], o_ref) < TOL_PREFILL, n
        assert rel_err(S[n], S_ref) < TOL_PREFILL, n


def test_uniform_batch_of_many_chains_matches_oracle(orc):
    """Three sequences of 32 heads (96 chains): more chains than the fused grid
    takes, fewer than the SMs, so prepare runs on every SM and then every chain
    in one wave."""
    K = kda()
    N, t, H = 3, 200, 32
    gen = torch.Generator().manual_seed(21)
    d = wl.core_inputs(gen, (N, t), H, torch.bfloat16)
    S0 = wl.state(gen, (N,), H, 0.02)
    dev = {n: d[n].cuda() for n in d}
    S = S0.clone().cuda()
    o = torch.zeros((N, t, H, 128), device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 64)
    K.kda_sync_status()
    for n in range(N):
        o_ref, S_ref = orc.prefill(d["q"][n], d["k"][n], d["v"][n], d["g"][n], d["beta"][n],
                                   S0[n])
        assert rel_err(o[n], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL


def test_malformed_cu_seqlens_is_reported_by_sync_status():
    K = kda()
    H = 1
    d = wl.core_inputs(torch.Generator().manual_seed(1), (32,), H, torch.float32)
    dev = {n: d[n].cuda() for n in d}
    S = torch.zeros((2, H, 128, 128), device="cuda")
    o = torch.zeros((32, H, 128), device="cuda")
    bad = torch.tensor([0, 40, 32], dtype=torch.int32, device="cuda")  # decreasing
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, 32, 16,
                  cu_seqlens=bad)
    with pytest.raises(K.KdaError) as ei:
        K.kda_sync_status()
    assert ei.value.status == 5
    K.kda_sync_status()  # the word was cleared


def test_batched_uniform_sequences(orc):
    K = kda()
    N, Tp, t, H = 3, 96, 90, 2
    gen = torch.Generator().manual_seed(2)
    d = wl.core_inputs(gen, (N, Tp), H, torch.bfloat16)
    S0 = wl.state(gen, (N,), H, 0.02)
    dev = {n: d[n].clone().cuda() for n in d}
    S = S0.clone().cuda()
    o = torch.zeros((N, Tp, H, 128), device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 32,
                  pad_fill=float("nan"))
    for n in range(N):
        o_ref, S_ref = orc.prefill(d["q"][n, :t], d["k"][n, :t], d["v"][n, :t], d["g"][n, :t],
                                   d["beta"][n, :t], S0[n])
        assert rel_err(o[n, :t], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL


def test_full_size_prefill_sampled_heads(orc):
    """The prefill workload (T=8192, 32 heads, chunk 64, BF16 inputs, state
    ~N(0, 0.02)) in the benchmark's launch configuration; 3 heads checked
    against the oracle, all heads for finiteness."""
    K = kda()
    d = wl.prefill()
    o, S, _ = run_prefill(K, d, 8192, 64)
    assert torch.isfinite(o).all() and torch.isfinite(S).all()
    for h in (0, 13, 31):
        o_ref, S_ref = orc.prefill(d["q"][:, h:h + 1], d["k"][:, h:h + 1], d["v"][:, h:h + 1],
                                   d["g"][:, h:h + 1], d["beta"][:, h:h + 1],
                                   d["state"][0, h:h + 1])
        assert rel_err(o[:, h:h + 1], o_ref) < TOL_PREFILL, h
        assert rel_err(S[0, h:h + 1], S_ref) < TOL_PREFILL, h


@pytest.mark.parametrize("impl,tol", [("simt", 1e-5), ("tc", TOL_PREFILL)])
def test_chained_prefills_equal_one_prefill(monkeypatch, impl, tol):
    """Two prefill calls carrying the state equal one call over both halves
    (within rounding: the chunk boundaries differ), on the FP32 SIMT kernel
    and on the tensor-core path."""
    if impl == "simt":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "simt")
    K = kda()
    d = wl.prefill(seed=9, t=200, heads=2, chunk=64, dtype=torch.float32)
    o_all, S_all, _ = run_prefill(K, d, 200, 64)
    first = {n: d[n][:100] for n in ("q", "k", "v", "g", "beta")}
    first["state"] = d["state"]
    o1, S1, _ = run_prefill(K, first, 100, 64)
    second = {n: d[n][100:] for n in ("q", "k", "v", "g", "beta")}
    second["state"] = S1.cpu()
    o2, S2, _ = run_prefill(K, second, 100, 64)
    assert rel_err(torch.cat([o1, o2]), o_all.cpu().double().numpy()) < tol
    assert rel_err(S2, S_all.cpu().double().numpy()) < tol


def test_tensor_core_and_simt_kernels_agree(orc, monkeypatch):
    """BF16 inputs with chunk 64 run on the tensor-core kernel; the FP32 SIMT
    kernel (pinned with KDA_PREFILL_IMPL=simt) computes the same method; both
    stay within the prefill tolerance of the oracle and of each other."""
    K = kda()
    d = wl.prefill(seed=21, t=300, heads=4, chunk=64, dtype=torch.bfloat16)
    o_tc, S_tc, _ = run_prefill(K, d, 300, 64)
    monkeypatch.setenv("KDA_PREFILL_IMPL", "simt")
    o_si, S_si, _ = run_prefill(K, d, 300, 64)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    assert rel_err(o_si, o_ref) < 1e-5 and rel_err(S_si[0], S_ref) < 1e-5
    assert rel_err(o_tc, o_ref) < TOL_PREFILL and rel_err(S_tc[0], S_ref) < TOL_PREFILL
    assert rel_err(o_tc, o_si.double().cpu().numpy()) < TOL_PREFILL


@pytest.mark.parametrize("g_low", [-0.05, -10.0, -30.0])
def test_prefill_long_memory_and_strong_decay(orc, g_low):
    """Slow decay (g in [-0.05, 0]: the state carries across all 16 chunks, so
    rounding in the carried state accumulates), the steepest decay of the
    tensor-core blocks (g in [-10, 0]) and one beyond it (exact products)."""
    K = kda()
    gen = torch.Generator().manual_seed(31)
    T, H = 1024, 2
    d = wl.core_inputs(gen, (T,), H, torch.bfloat16, g_low=g_low)
    d["state"] = wl.state(gen, (1,), H, 0.02)
    o, S, _ = run_prefill(K, d, T, 64)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


def test_prefill_mixes_wide_and_narrow_decay_blocks(orc):
    """Chunks whose decays all stay above -5.1 take 32-token A/P blocks, the
    others 16-token blocks; one sequence with both kinds of chunk (single
    steep decays of -9 and -5.5 in two of its chunks) matches the oracle."""
    K = kda()
    gen = torch.Generator().manual_seed(41)
    T, H = 320, 2
    d = wl.core_inputs(gen, (T,), H, torch.bfloat16)
    d["g"][70, 0, 5] = -9.0
    d["g"][200, 1, 100] = -5.5
    d["g"][260, 0, 7] = -5.1
    d["state"] = wl.state(gen, (1,), H, 0.02)
    o, S, _ = run_prefill(K, d, T, 64)
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    assert rel_err(o, o_ref) < TOL_PREFILL
    assert rel_err(S[0], S_ref) < TOL_PREFILL


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("t,t_pad", [(1, 1), (5, 8), (8, 8)])
def test_short_prefill_takes_the_row_walk(orc, dtype, t, t_pad):
    """Sequences of t <= 8 tokens (uniform form) run decode_k's row walk, BF16
    inputs widened exactly: oracle parity per sequence at the FP32 tolerance,
    padded rows ignored, and the same bits as an explicit kda_decode_k over
    the same (widened) rows."""
    from _util import TOL_DECODE
    K = kda()
    gen = torch.Generator().manual_seed(60 + t)
    N, H = 3, 2
    d = wl.core_inputs(gen, (N, t_pad), H, dtype)
    S0 = wl.state(gen, (N,), H, 0.02)
    dev = {}
    for n in ("q", "k", "v", "g", "beta"):
        x = d[n].clone()
        x[:, t:] = float("nan")
        dev[n] = x.cuda()
    S = S0.clone().cuda()
    o = torch.full((N, t_pad, H, 128), 12345.0, device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 16,
                  pad_fill=0.0)
    torch.cuda.synchronize()
    assert torch.all(o[:, t:] == 12345.0)  # padding rows are not written
    for n in range(N):
        o_ref, S_ref = orc.prefill(d["q"][n, :t], d["k"][n, :t], d["v"][n, :t], d["g"][n, :t],
                                   d["beta"][n, :t], S0[n])
        assert rel_err(o[n, :t], o_ref) < TOL_DECODE
        assert rel_err(S[n], S_ref) < TOL_DECODE
    if t == t_pad:
        S2 = S0.clone().cuda()
        o2 = torch.empty_like(o)
        K.kda_decode_k(S2, *(d[n].float().cuda().contiguous()
                             for n in ("q", "k", "v", "g", "beta")), o2)
        torch.cuda.synchronize()
        assert torch.equal(S2, S) and torch.equal(o2, o)
