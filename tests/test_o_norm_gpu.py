"""kda_o_norm_gated (sigmoid-gated RMSNorm of the core output) against the
FP64 oracle, at small sizes and on the prefill workload's output shape."""

import numpy as np
import pytest
import torch

import kda_workloads as wl
from _util import kda

pytestmark = pytest.mark.gpu


def bf16_close(out, ref):
    """|gpu - ref| <= 1 BF16 ulp of ref (+ a tiny absolute floor): the kernel
    computes in FP32 and rounds once to BF16."""
    x = out.float().cpu().double().numpy()
    ref = np.asarray(ref)
    ulp = np.maximum(np.abs(ref), 1e-30) * 2.0 ** -7
    bad = np.abs(x - ref) > ulp + 1e-6
    assert not bad.any(), "max excess %g" % float((np.abs(x - ref) - ulp).max())


def _inputs(seed, rows, H):
    gen = torch.Generator().manual_seed(seed)
    core = torch.randn((rows, H, 128), generator=gen) * 3.0
    gate = torch.randn((rows, H * 128), generator=gen).to(torch.bfloat16)
    w = (1.0 + 0.5 * torch.randn(128, generator=gen)).to(torch.bfloat16)
    return core, gate, w


@pytest.mark.parametrize("rows,H", [(1, 1), (77, 3), (300, 8)])
def test_o_norm_matches_oracle(orc, rows, H):
    K = kda()
    core, gate, w = _inputs(rows * 10 + H, rows, H)
    out = torch.empty((rows, H * 128), dtype=torch.bfloat16, device="cuda")
    K.kda_o_norm_gated(core.cuda(), gate.cuda(), w.cuda(), out, eps=1e-6)
    ref = orc.o_norm_gated(core, gate, w, eps=1e-6)
    bf16_close(out.reshape(rows, H, 128), ref)


def test_o_norm_zero_rows_and_zero_head():
    K = kda()
    core, gate, w = _inputs(5, 4, 2)
    core[2, 1] = 0.0  # an all-zero head: 0 / sqrt(eps) = 0
    out = torch.full((4, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    K.kda_o_norm_gated(core.cuda(), gate.cuda(), w.cuda(), out, eps=1e-6)
    assert torch.equal(out[2, 128:].float().cpu(), torch.zeros(128))
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    K.kda_o_norm_gated(torch.empty((0, 2, 128), device="cuda"), empty, w.cuda(), empty)


def test_o_norm_prefill_output_shape_sampled(orc):
    """The prefill workload's output shape (8192 tokens x 32 heads), checked
    on sampled rows."""
    K = kda()
    T, H = 8192, 32
    core, gate, w = _inputs(11, T, H)
    out = torch.empty((T, H * 128), dtype=torch.bfloat16, device="cuda")
    K.kda_o_norm_gated(core.cuda(), gate.cuda(), w.cuda(), out, eps=1e-6)
    rows = torch.randint(0, T, (64,), generator=torch.Generator().manual_seed(3))
    ref = orc.o_norm_gated(core[rows], gate[rows], w, eps=1e-6)
    bf16_close(out[rows.cuda()].reshape(64, H, 128), ref)
