"""Input range of the tensor-core prefill.  The scan multiplies FP16 operands
(the state, X = V - Ktil S, U = T X; FP32 accumulation), so values far below
or above 1 meet FP16's subnormal floor (2^-24) and its largest finite value
(65504).  These tests scale v and the initial state together and apart by
1e-4 and 1e3, on the fused grid and on the two-kernel path, against the FP64
oracle on the same inputs."""

import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu

H = 32


def scaled_inputs(seed, t, v_scale, s_scale, g_low):
    gen = torch.Generator().manual_seed(seed)
    d = wl.core_inputs(gen, (t,), H, torch.float64, g_low=g_low)
    d["v"] = d["v"] * v_scale
    d = {n: x.to(torch.bfloat16) for n, x in d.items()}
    d["state"] = wl.state(gen, (1,), H, 0.02 * s_scale)
    return d


@pytest.mark.parametrize("impl", ["fused", "unfused"])
@pytest.mark.parametrize("v_scale,s_scale", [(1e-4, 1.0), (1.0, 1e-4), (1e-4, 1e-4),
                                             (1e3, 1.0), (1.0, 1e3), (1e3, 1e3)])
@pytest.mark.parametrize("g_low", [-5.0, -0.05])
def test_scaled_values_and_state(orc, monkeypatch, impl, v_scale, s_scale, g_low):
    if impl == "unfused":
        monkeypatch.setenv("KDA_PREFILL_IMPL", "unfused")
    K = kda()
    t = 300
    d = scaled_inputs(900 + int(v_scale < 1) + 2 * int(s_scale < 1), t, v_scale, s_scale, g_low)
    dev = {n: d[n].cuda() for n in ("q", "k", "v", "g", "beta")}
    S = d["state"].clone().cuda()
    o = torch.empty((t, H, 128), device="cuda")
    K.kda_prefill(S, dev["q"], dev["k"], dev["v"], dev["g"], dev["beta"], o, t, 64)
    K.kda_sync_status()
    o_ref, S_ref = orc.prefill(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"][0])
    e_o, e_s = rel_err(o, o_ref), rel_err(S[0], S_ref)
    print("range v x%g S0 x%g g>=%g %s: o %.3g state %.3g" % (v_scale, s_scale, g_low, impl,
                                                              e_o, e_s))
    assert e_o < TOL_PREFILL and e_s < TOL_PREFILL
