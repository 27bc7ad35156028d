"""kda_prefill_o_norm: the sigmoid-gated RMSNorm fused into the tensor-core
prefill's epilogue (BF16 output, no FP32 core output written).

Two checks per case:
  - against the oracle's norm of this library's own FP32 core output
    (kda_prefill on the same inputs: the fused path reads the same O values
    from TMEM), within one BF16 ulp: the epilogue itself;
  - against the FP64 oracle end to end (oracle core, then oracle norm),
    within the prefill tolerance carried through the normalisation plus one
    BF16 ulp (the bound is derived in check())."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda

pytestmark = pytest.mark.gpu

EPS = 1e-6


def bf16_ulp(x):
    """The spacing of BF16 numbers at |x| (8 significand bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def norm_inputs(gen, rows, H):
    gate = torch.randn((rows, H * 128), generator=gen, dtype=torch.float64).to(torch.bfloat16)
    w = (1.0 + 0.1 * torch.randn(128, generator=gen, dtype=torch.float64)).to(torch.bfloat16)
    return gate, w


def check(out, o_gpu, o_ref, gate, w, orc):
    rows, H = o_ref.shape[0], o_ref.shape[1]
    got = out.float().cpu().double().numpy().reshape(rows, H, 128)
    assert np.all(np.isfinite(got))
    # the epilogue: the oracle's norm of this library's FP32 core output
    ref_own = orc.o_norm_gated(o_gpu.cpu(), gate, w, EPS)
    err_own = np.abs(got - ref_own)
    assert np.all(err_own <= 1.01 * bf16_ulp(ref_own) + 1e-7), err_own.max()
    # end to end: the oracle's core, then its norm.  The core's bound is
    # normwise, |do| <= TOL_PREFILL * max|o| over the whole output; through
    # o_j / r (r the row's RMS) it becomes |d(o_j / r)| <= max|do| / r *
    # (1 + |o_j| / r), times |w_j sigmoid(gate_j)|, plus one BF16 ulp.
    ref = orc.o_norm_gated(o_ref, gate, w, EPS)
    o64 = np.asarray(o_ref, dtype=np.float64)
    r = np.sqrt((o64 ** 2).mean(axis=2, keepdims=True) + EPS)
    ws = (w.double().numpy()[None, None, :] /
          (1.0 + np.exp(-gate.double().numpy().reshape(o64.shape))))
    err = np.abs(got - ref)
    bound = (TOL_PREFILL * np.abs(o64).max() / r * (1.0 + np.abs(o64) / r) * np.abs(ws)
             + bf16_ulp(ref))
    worst = (err / bound).max()
    print("o_norm fused: worst err / bound %.3f" % worst)
    assert worst <= 1.0


@pytest.mark.parametrize("impl", ["fused", "unfused"])
@pytest.mark.parametrize("t", [1, 64, 300, 1000])
def test_prefill_o_norm_matches_oracle(orc, monkeypatch, impl, t):
    """One sequence of 32 heads (the fused grid; KDA_PREFILL_IMPL=unfused pins
    the two kernels): one-token, one-chunk, ragged and long sequences."""
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    H = 32
    gen = torch.Generator().manual_seed(400 + t)
    d = wl.core_inputs(gen, (t,), H, torch.bfloat16)
    S0 = wl.state(gen, (1,), H, 0.02)
    gate, w = norm_inputs(gen, t, H)
    dev = {n: d[n].cuda() for n in d}
    # this library's FP32 core output, for the epilogue check; q, k, v as
    # slices of one wider buffer keep this call on the tensor-core kernels for
    # every t (a short contiguous sequence would take the row walk)
    hd = H * 128
    qkv = torch.cat([dev[n].reshape(t, hd) for n in ("q", "k", "v")], dim=1)
    qs, ks, vs = (torch.as_strided(qkv, (t, H, 128), (3 * hd, 128, 1), i * hd)
                  for i in range(3))
    S1 = S0.clone().cuda()
    o_gpu = torch.empty((t, H, 128), device="cuda")
    K.kda_prefill(S1, qs, ks, vs, dev["g"], dev["beta"], o_gpu, t, 64)
    S2 = S0.clone().cuda()
    out = torch.full((t, H * 128), 7.0, dtype=torch.bfloat16, device="cuda")
    K.kda_prefill_o_norm(S2, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], gate.cuda(),
                         w.cuda(), out, t, 64, eps=EPS)
    K.kda_sync_status()
    assert torch.equal(S1, S2)  # the same chain: the same state, bit for bit
    o_ref, _ = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], S0[0])
    check(out, o_gpu, o_ref, gate, w, orc)


@pytest.mark.parametrize("packed", [True, False])
def test_prefill_o_norm_two_sequences(orc, packed):
    """Two sequences of 16 heads, packed (cu_seqlens) with ragged lengths, or
    uniform with a padded tail whose output rows stay untouched; gate and out
    as row views of wider buffers."""
    K = kda()
    H = 16
    lengths = [300, 517] if packed else [517, 517]
    t_pad = 600 if not packed else None
    gen = torch.Generator().manual_seed(11 + int(packed))
    tot = sum(lengths)
    d = wl.core_inputs(gen, (tot,), H, torch.bfloat16)
    S0 = wl.state(gen, (2,), H, 0.02)
    gate, w = norm_inputs(gen, tot, H)
    if packed:
        rows = tot
        dev = {n: d[n].cuda() for n in d}
        gate_rows = gate
    else:
        rows = 2 * t_pad
        dev = {}
        for n, x in d.items():
            xp = torch.zeros((2, t_pad) + tuple(x.shape[1:]), dtype=x.dtype)
            xp[0, :517] = x[:517]
            xp[1, :517] = x[517:]
            dev[n] = xp.cuda()
        gate_rows = torch.zeros((rows, H * 128), dtype=torch.bfloat16)
        gate_rows[:517] = gate[:517]
        gate_rows[t_pad:t_pad + 517] = gate[517:]
    wide_g = torch.zeros((rows, H * 128 + 64), dtype=torch.bfloat16, device="cuda")
    wide_g[:, :H * 128] = gate_rows.cuda()
    wide_o = torch.full((rows, H * 128 + 64), 7.0, dtype=torch.bfloat16, device="cuda")
    S1 = S0.clone().cuda()
    S2 = S0.clone().cuda()
    o_gpu = torch.empty((rows, H, 128), device="cuda")
    if packed:
        cu = torch.tensor([0, lengths[0], tot], dtype=torch.int32, device="cuda")
        K.kda_prefill(S1, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o_gpu, tot, 64,
                      cu_seqlens=cu)
        K.kda_prefill_o_norm(S2, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                             wide_g[:, :H * 128], w.cuda(), wide_o[:, :H * 128], tot, 64,
                             eps=EPS, cu_seqlens=cu)
    else:
        K.kda_prefill(S1, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                      o_gpu.view(2, t_pad, H, 128), 517, 64)
        K.kda_prefill_o_norm(S2, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"],
                             wide_g[:, :H * 128], w.cuda(), wide_o[:, :H * 128], 517, 64,
                             eps=EPS)
    K.kda_sync_status()
    assert torch.equal(S1, S2)
    assert (wide_o[:, H * 128:] == 7.0).all()  # nothing past the heads' channels
    a = 0
    for n, L in enumerate(lengths):
        r0 = a if packed else n * t_pad
        o_ref, _ = orc.prefill(d["q"][a:a + L], d["k"][a:a + L], d["v"][a:a + L],
                               d["g"][a:a + L], d["beta"][a:a + L], S0[n])
        check(wide_o[r0:r0 + L, :H * 128], o_gpu[r0:r0 + L], o_ref, gate[a:a + L], w, orc)
        if not packed:  # padded rows are not written
            assert (wide_o[r0 + L:r0 + t_pad] == 7.0).all()
        a += L
