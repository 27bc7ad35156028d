"""Front end + core: kda_conv_silu_l2 then kda_prefill reading q, k, v as
strided views of the conv output, on packed variable-length sequences.  Each
stage is compared on its own (the core against the oracle on the GPU's own
conv output), as the pages ask: stage by stage."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import TOL_PREFILL, kda, rel_err

pytestmark = pytest.mark.gpu


def test_conv_then_core_varlen(orc):
    K = kda()
    d = wl.frontend(lengths=[300, 64, 1, 777], heads=4)
    H = 4
    hd = H * 128
    cu = d["cu_seqlens"]
    tot = int(cu[-1])
    x = d["x"].cuda()
    out = torch.empty_like(x)
    cst = d["conv_state"].clone().cuda()
    cu_d = cu.cuda()
    K.kda_conv_silu_l2(cst, x, d["w"].cuda(), out, cu_seqlens=cu_d)
    q = out[:, :hd].view(tot, H, 128)
    k = out[:, hd:2 * hd].view(tot, H, 128)
    v = out[:, 2 * hd:].view(tot, H, 128)
    S = d["state"].clone().cuda()
    o = torch.zeros((tot, H, 128), device="cuda")
    K.kda_prefill(S, q, k, v, d["g"].cuda(), d["beta"].cuda(), o, tot, 64, cu_seqlens=cu_d)
    K.kda_sync_status()
    conv_host = out.cpu()
    for n in range(4):
        a, b = int(cu[n]), int(cu[n + 1])
        qs = conv_host[a:b, :hd].view(b - a, H, 128)
        ks = conv_host[a:b, hd:2 * hd].view(b - a, H, 128)
        vs = conv_host[a:b, 2 * hd:].view(b - a, H, 128)
        o_ref, S_ref = orc.prefill(qs, ks, vs, d["g"][a:b], d["beta"][a:b], d["state"][n])
        assert rel_err(o[a:b], o_ref) < TOL_PREFILL
        assert rel_err(S[n], S_ref) < TOL_PREFILL
