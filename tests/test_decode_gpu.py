"""kda_decode and kda_decode_k against the FP64 oracle, and decode_k against
serial decodes bit for bit (Glm5NextKdaLayer::decode_k: "matches k serial
decode calls bit for bit")."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import TOL_DECODE, kda, rel_err

pytestmark = pytest.mark.gpu


def _dev(d):
    return {k_: (v_.cuda() if isinstance(v_, torch.Tensor) else v_) for k_, v_ in d.items()}


@pytest.mark.parametrize("N,H", [(1, 1), (3, 2), (5, 7)])
def test_decode_single_step_matches_oracle(orc, N, H):
    K = kda()
    d = wl.decode_steps(seed=N * 10 + H, n_seqs=N, heads=H, steps=1)
    g = _dev(d)
    S = g["state"].clone()
    o = torch.empty((N, H, 128), device="cuda")
    K.kda_decode(S, g["q"][0], g["k"][0], g["v"][0], g["g"][0], g["beta"][0], o)
    o_ref, S_ref = orc.recurrent(d["q"][0][:, None], d["k"][0][:, None], d["v"][0][:, None],
                                 d["g"][0][:, None], d["beta"][0][:, None], d["state"])
    assert rel_err(o, o_ref[:, 0]) < TOL_DECODE
    assert rel_err(S, S_ref) < TOL_DECODE


def test_decode_100_chained_steps_full_size_sampled(orc):
    """The decode workload: 64 sequences x 32 heads, state ~N(0, 0.02), 100
    chained steps in place; o checked at every step and the final state on a
    sample of 8 sequences (all heads), the rest checked for finiteness."""
    K = kda()
    d = wl.decode_steps()
    g = _dev(d)
    S = g["state"].clone()
    steps = d["q"].shape[0]
    o_all = torch.empty((steps, 64, 32, 128), device="cuda")
    for t in range(steps):
        K.kda_decode(S, g["q"][t], g["k"][t], g["v"][t], g["g"][t], g["beta"][t], o_all[t])
    torch.cuda.synchronize()
    sample = [0, 9, 17, 30, 33, 47, 58, 63]
    tr = lambda x: x[:, sample].transpose(0, 1).contiguous()  # [steps,N,...] -> [N,steps,...]
    o_ref, S_ref = orc.recurrent(tr(d["q"]), tr(d["k"]), tr(d["v"]), tr(d["g"]),
                                 tr(d["beta"]), d["state"][sample])
    o_gpu = o_all[:, sample].transpose(0, 1).cpu()
    for t in range(steps):
        assert rel_err(o_gpu[:, t], o_ref[:, t]) < TOL_DECODE, t
    assert rel_err(S[sample].cpu(), S_ref) < TOL_DECODE
    assert torch.isfinite(S).all() and torch.isfinite(o_all).all()


@pytest.mark.parametrize("krows,n_snap", [(1, 1), (4, 4), (4, 2), (8, 0), (8, 8), (3, 3)])
def test_decode_k_bit_identical_to_serial_decodes(krows, n_snap):
    K = kda()
    N, H = 6, 3
    d = _dev(wl.decode_k(seed=krows * 7 + n_snap, n_seqs=N, krows=krows, heads=H))
    S_k = d["state"].clone()
    o_k = torch.empty((N, krows, H, 128), device="cuda")
    snaps = [torch.full_like(S_k, float("nan")) for _ in range(n_snap)]
    K.kda_decode_k(S_k, d["q"], d["k"], d["v"], d["g"], d["beta"], o_k, snaps)
    S_s = d["state"].clone()
    for t in range(krows):
        o_t = torch.empty((N, H, 128), device="cuda")
        K.kda_decode(S_s, d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                     d["v"][:, t].contiguous(), d["g"][:, t].contiguous(),
                     d["beta"][:, t].contiguous(), o_t)
        assert torch.equal(o_t, o_k[:, t]), "row %d output differs" % t
        if t < n_snap:
            assert torch.equal(snaps[t], S_s), "snapshot %d differs" % t
    assert torch.equal(S_k, S_s)


def test_decode_k_full_size_matches_oracle_sampled(orc):
    """The speculative-verify workload: 128 sequences x k=4 rows x 32 heads,
    a snapshot after each row; sampled sequences against the oracle."""
    K = kda()
    d = wl.decode_k()
    g = _dev(d)
    S = g["state"].clone()
    o = torch.empty((128, 4, 32, 128), device="cuda")
    snaps = [torch.empty_like(S) for _ in range(4)]
    K.kda_decode_k(S, g["q"], g["k"], g["v"], g["g"], g["beta"], o, snaps)
    torch.cuda.synchronize()
    sample = [0, 5, 64, 127]
    o_ref, S_ref, snap_ref = orc.recurrent(d["q"][sample], d["k"][sample], d["v"][sample],
                                           d["g"][sample], d["beta"][sample],
                                           d["state"][sample], snapshots=True)
    assert rel_err(o[sample].cpu(), o_ref) < TOL_DECODE
    assert rel_err(S[sample].cpu(), S_ref) < TOL_DECODE
    for t in range(4):
        assert rel_err(snaps[t][sample].cpu(), snap_ref[t]) < TOL_DECODE
    assert torch.equal(snaps[3], S)


def test_decode_k_leaves_unrequested_snapshots_untouched():
    K = kda()
    d = _dev(wl.decode_k(seed=3, n_seqs=2, krows=4, heads=2))
    S = d["state"].clone()
    o = torch.empty((2, 4, 2, 128), device="cuda")
    snaps = [torch.full_like(S, 7.0) for _ in range(2)]
    guard = torch.full_like(S, 7.0)
    K.kda_decode_k(S, d["q"], d["k"], d["v"], d["g"], d["beta"], o, snaps)
    torch.cuda.synchronize()
    assert torch.equal(guard, torch.full_like(S, 7.0))
    assert not torch.equal(snaps[1], guard)


def test_decode_rejects_bad_calls_without_launching():
    K = kda()
    S = torch.zeros((1, 1, 128, 128), device="cuda")
    x = torch.zeros((1, 1, 4, 1, 128), device="cuda")[0]
    b = torch.zeros((1, 4, 1), device="cuda")
    o = torch.zeros((1, 4, 1, 128), device="cuda")
    with pytest.raises(K.KdaError):
        K.kda_decode_k(S, x, x, x, x, b, o, [torch.zeros_like(S)] * 5)
    q9 = torch.zeros((1, 9, 1, 128), device="cuda")
    with pytest.raises(K.KdaError):
        K.kda_decode_k(S, q9, q9, q9, q9, torch.zeros((1, 9, 1), device="cuda"), q9.clone())
