"""kda_gate (the forget gate and beta before the core) against the FP64
oracle: FP32 and BF16 outputs, a strided g_raw / b_raw (views of wider
projections), and a prefill-sized problem on sampled rows; the gate feeds the
prefill like a caller's g and beta."""

import numpy as np
import pytest
import torch

from _util import kda, rel_err

pytestmark = pytest.mark.gpu

LB = -5.0


def inputs(seed, rows, H, pitch_extra=0):
    gen = torch.Generator().manual_seed(seed)
    g_raw = torch.randn((rows, H * 128 + pitch_extra), generator=gen).to(torch.bfloat16)
    dt = (torch.randn(H * 128, generator=gen) * 0.5).float()
    al = (torch.randn(H, generator=gen) * 0.5).float()
    b = torch.randn((rows, H + 3), generator=gen).to(torch.bfloat16)
    return g_raw, dt, al, b


def run(K, g_raw, dt, al, b, H, dtype):
    rows = g_raw.shape[0]
    g = torch.empty((rows, H, 128), dtype=dtype, device="cuda")
    beta = torch.empty((rows, H), dtype=dtype, device="cuda")
    K.kda_gate(g_raw.cuda(), dt.cuda(), al.cuda(), b.cuda(), g, beta, LB)
    torch.cuda.synchronize()
    return g, beta


def ref(orc, g_raw, dt, al, b, H):
    return orc.gate(g_raw[:, :H * 128], dt, al, LB, b[:, :H])


# (40000, 3): every thread walks several steps of 4 rows and the grid is
# rounded to whole rows of 48 groups; (5, 7): a grid of 7 CTAs, mostly idle.
@pytest.mark.parametrize("rows,H,extra", [(1, 1, 0), (37, 4, 0), (300, 2, 64), (5, 7, 8),
                                          (40000, 3, 8)])
def test_gate_fp32_matches_oracle(orc, rows, H, extra):
    K = kda()
    g_raw, dt, al, b = inputs(rows + H, rows, H, extra)
    g, beta = run(K, g_raw, dt, al, b, H, torch.float32)
    g_ref, b_ref = ref(orc, g_raw, dt, al, b, H)
    # the hardware exponential and reciprocal: a few ulp, normwise under 1e-5
    assert rel_err(g, g_ref) < 1e-5 and rel_err(beta, b_ref) < 1e-5
    gh = g.double().cpu().numpy()
    assert np.all(gh <= 0) and np.all(gh >= LB)


def test_gate_bf16_within_one_ulp(orc):
    K = kda()
    rows, H = 200, 3
    g_raw, dt, al, b = inputs(9, rows, H)
    g, beta = run(K, g_raw, dt, al, b, H, torch.bfloat16)
    g_ref, b_ref = ref(orc, g_raw, dt, al, b, H)
    for x, r in ((g, g_ref), (beta, b_ref)):
        x = x.double().cpu().numpy()
        ulp = np.abs(r) * 2.0 ** -7  # one BF16 ulp at the value (8 significand bits)
        assert np.all(np.abs(x - r) <= ulp + 1e-6)


def test_gate_prefill_sized_sampled_rows(orc):
    """8192 rows x 32 heads (the prefill workload's g and beta), BF16 out; the
    oracle on every 97th row."""
    K = kda()
    rows, H = 8192, 32
    g_raw, dt, al, b = inputs(11, rows, H)
    g, beta = run(K, g_raw, dt, al, b, H, torch.bfloat16)
    idx = torch.arange(0, rows, 97)
    g_ref, b_ref = ref(orc, g_raw[idx], dt, al, b[idx], H)
    assert rel_err(g[idx.cuda()], g_ref) < 8e-3
    assert rel_err(beta[idx.cuda()], b_ref) < 8e-3
