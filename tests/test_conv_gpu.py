"""kda_conv_silu_l2 against the FP64 oracle (rounded to BF16), decode-style
streaming against one prefill call, and the conv state update."""

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


@pytest.mark.parametrize("K_,lengths", [(4, [37, 1, 0, 100]), (3, [5]), (1, [64, 64]),
                                        (2, [2, 3])])
def test_conv_varlen_matches_oracle(orc, K_, lengths):
    K = kda()
    H = 2
    ch = 3 * H * 128
    gen = torch.Generator().manual_seed(len(lengths) * 10 + K_)
    tot = sum(lengths)
    x = torch.randn((tot, ch), generator=gen).to(torch.bfloat16)
    w = (torch.randn((ch, K_), generator=gen) * 0.5).to(torch.bfloat16)
    st = torch.randn((len(lengths), ch, K_), generator=gen)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    out = torch.empty_like(x).cuda()
    st_d = st.clone().cuda()
    K.kda_conv_silu_l2(st_d, x.cuda(), w.cuda(), out, cu_seqlens=cu.cuda())
    K.kda_sync_status()
    ref, st_ref = orc.conv_silu_l2(x, w, st, cu.numpy(), H)
    bf16_close(out, ref)
    np.testing.assert_array_equal(st_d.cpu().double().numpy(), st_ref)


@pytest.mark.parametrize("K_,T", [(4, 8), (4, 20), (3, 8), (1, 5)])
def test_conv_decode_stream_equals_prefill(K_, T):
    """T single-token calls for 5 sequences at once (decode, the short-rows
    kernel) give the same bits as one T-token prefill call per sequence, in
    the uniform form (short-rows kernel for T <= 8) and in the varlen form
    (the token-span kernel)."""
    K = kda()
    H, N = 1, 5
    ch = 3 * H * 128
    gen = torch.Generator().manual_seed(3 + T + K_)
    x = torch.randn((N, T, ch), generator=gen).to(torch.bfloat16).cuda()
    w = (torch.randn((ch, K_), generator=gen) * 0.5).to(torch.bfloat16).cuda()
    st0 = torch.randn((N, ch, K_), generator=gen).cuda()
    out_p = torch.empty_like(x)
    st_p = st0.clone()
    K.kda_conv_silu_l2(st_p, x.reshape(N * T, ch), w, out_p.reshape(N * T, ch), n_seqs=N)
    out_v = torch.empty_like(x)
    st_v = st0.clone()
    cu = torch.arange(0, N * T + 1, T, dtype=torch.int32, device="cuda")
    K.kda_conv_silu_l2(st_v, x.reshape(N * T, ch), w, out_v.reshape(N * T, ch), cu_seqlens=cu)
    K.kda_sync_status()
    assert torch.equal(out_v, out_p)
    assert torch.equal(st_v, st_p)
    st_d = st0.clone()
    for t in range(T):
        o1 = torch.empty((N, ch), dtype=torch.bfloat16, device="cuda")
        K.kda_conv_silu_l2(st_d, x[:, t].contiguous(), w, o1, n_seqs=N)
        assert torch.equal(o1, out_p[:, t])
    assert torch.equal(st_d, st_p)


def test_conv_frontend_workload_sampled(orc):
    """The front-end workload's conv (16 sequences, lengths 512..8192, 12288
    channels, K=4): all outputs against the oracle on 3 sequences."""
    K = kda()
    d = wl.frontend()
    cu = d["cu_seqlens"]
    out = torch.empty_like(d["x"]).cuda()
    st = d["conv_state"].clone().cuda()
    K.kda_conv_silu_l2(st, d["x"].cuda(), d["w"].cuda(), out, cu_seqlens=cu.cuda())
    K.kda_sync_status()
    for n in (0, 7, 15):
        a, b = int(cu[n]), int(cu[n + 1])
        ref, st_ref = orc.conv_silu_l2(d["x"][a:b], d["w"], d["conv_state"][n:n + 1],
                                       [0, b - a], 32)
        bf16_close(out[a:b], ref)
        np.testing.assert_array_equal(st[n].cpu().double().numpy(), st_ref[0])


@pytest.mark.parametrize("K_,krows,n_snap", [(4, 4, 4), (4, 6, 3), (3, 1, 1), (2, 8, 0)])
def test_conv_k_rows_equal_serial_calls_with_snapshots(orc, K_, krows, n_snap):
    """kda_conv_silu_l2_k over k rows gives the bits of k single-token calls,
    and snapshots[t] the conv state after row t; the oracle agrees."""
    K = kda()
    H, N = 1, 5
    ch = 3 * H * 128
    gen = torch.Generator().manual_seed(70 + krows)
    x = torch.randn((N, krows, ch), generator=gen).to(torch.bfloat16).cuda()
    w = (torch.randn((ch, K_), generator=gen) * 0.5).to(torch.bfloat16).cuda()
    st0 = torch.randn((N, ch, K_), generator=gen).cuda()
    st_k = st0.clone()
    out_k = torch.empty_like(x)
    snaps = [torch.full_like(st0, float("nan")) for _ in range(n_snap)]
    K.kda_conv_silu_l2_k(st_k, x, w, out_k, snaps)
    st_s = st0.clone()
    for t in range(krows):
        o1 = torch.empty((N, ch), dtype=torch.bfloat16, device="cuda")
        K.kda_conv_silu_l2(st_s, x[:, t].contiguous(), w, o1, n_seqs=N)
        assert torch.equal(o1, out_k[:, t])
        if t < n_snap:
            assert torch.equal(snaps[t], st_s)
    assert torch.equal(st_k, st_s)
    xc = x.reshape(N * krows, ch).cpu()
    cu = [krows * n for n in range(N + 1)]
    ref, st_ref = orc.conv_silu_l2(xc, w.cpu(), st0.cpu(), cu, H)
    bf16_close(out_k.reshape(N * krows, ch).cpu(), ref)
    np.testing.assert_array_equal(st_k.cpu().double().numpy(), st_ref)
