"""Pins for the FP64 oracle: closed forms, special cases, hand-worked examples,
brute-force invariants and library-routine cross-checks.  No GPU.

Each test names the property of the method it holds the oracle to; the
method is the gated delta-rule token step of the GLM-5.3-Flash KDA block
(Glm5NextKdaLayer::decode / decode_k / prefill), its chunked form
(Glm5NextKdaKernels::chunk_prepare / chunk_scan) and the conv + SiLU + L2 front
end of the block pipeline (glm5next_kda module index).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import kda_workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rng(seed=0):
    return np.random.default_rng(seed)


def rand_inputs(r, N, T, H, D, g_low=-5.0):
    def unit(shape):
        x = r.standard_normal(shape)
        return x / np.linalg.norm(x, axis=-1, keepdims=True)
    q = unit((N, T, H, D))
    k = unit((N, T, H, D))
    v = r.standard_normal((N, T, H, D))
    g = r.uniform(g_low, 0.0, (N, T, H, D))
    beta = 1.0 / (1.0 + np.exp(-r.standard_normal((N, T, H))))
    return q, k, v, g, beta


# ----------------------------------------------------------------- hand-worked

def test_hand_d2_golden(orc):
    cases = json.load(open(os.path.join(GOLDEN, "hand_d2.json")))["cases"]
    for c in cases:
        D = c["D"]
        vec = lambda n: np.array(c[n], dtype=np.float64).reshape(1, 1, 1, D)
        o, S = orc.recurrent(vec("q"), vec("k"), vec("v"), vec("g"),
                             np.array(c["beta"]).reshape(1, 1, 1),
                             np.array(c["S0"]).reshape(1, 1, D, D))
        scale = 1.0 / math.sqrt(D)
        np.testing.assert_allclose(S[0, 0], np.array(c["S1"]), rtol=0, atol=1e-14,
                                   err_msg=c["name"])
        np.testing.assert_allclose(o[0, 0, 0] / scale, np.array(c["o_over_scale"]),
                                   rtol=0, atol=1e-14, err_msg=c["name"])


def test_hand_d1_three_tokens_golden(orc):
    c = json.load(open(os.path.join(GOLDEN, "hand_d1_three_tokens.json")))
    T = len(c["g"])
    col = lambda n: np.array(c[n], dtype=np.float64).reshape(1, T, 1, 1)
    o, S, snaps = orc.recurrent(col("q"), col("k"), col("v"), col("g"),
                                np.array(c["beta"]).reshape(1, T, 1),
                                np.array(c["S0"]).reshape(1, 1, 1, 1), snapshots=True)
    np.testing.assert_allclose(o.reshape(T), c["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(snaps.reshape(T), c["S_after"], rtol=0, atol=1e-14)
    assert abs(S.item() - c["S_after"][-1]) < 1e-14


# ----------------------------------------------------------------- closed forms

@pytest.mark.parametrize("D", [8, 128])
def test_one_token_from_zero_state(orc, D):
    """From S = 0, one token gives S = beta k v^T and o = scale beta (q.k) v."""
    r = rng(1)
    q, k, v, g, beta = rand_inputs(r, 1, 1, 3, D)
    o, S = orc.recurrent(q, k, v, g, beta, np.zeros((1, 3, D, D)))
    scale = 1.0 / math.sqrt(D)
    for h in range(3):
        kk, vv, qq, b = k[0, 0, h], v[0, 0, h], q[0, 0, h], beta[0, 0, h]
        np.testing.assert_allclose(S[0, h], b * np.outer(kk, vv), atol=1e-14)
        np.testing.assert_allclose(o[0, 0, h], scale * b * qq.dot(kk) * vv, atol=1e-14)


def test_beta_one_unit_k_recovers_v(orc):
    """With beta = 1 and |k| = 1, right after the update S^T k = v, at every
    token and for any decay: the residual is taken on the decayed state."""
    r = rng(2)
    D, T, H = 128, 12, 2
    q, k, v, g, _ = rand_inputs(r, 1, T, H, D)
    beta = np.ones((1, T, H))
    S0 = r.standard_normal((1, H, D, D)) * 0.3
    _, _, snaps = orc.recurrent(q, k, v, g, beta, S0, snapshots=True)
    for t in range(T):
        for h in range(H):
            np.testing.assert_allclose(snaps[t, 0, h].T @ k[0, t, h], v[0, t, h], atol=1e-12)


def test_g0_beta0_state_unchanged_and_readout(orc):
    """g = 0, beta = 0: an empty update; o_t = scale * S0^T q_t."""
    r = rng(3)
    D, T, H = 128, 5, 2
    q, k, v, _, _ = rand_inputs(r, 1, T, H, D)
    g = np.zeros_like(q)
    beta = np.zeros((1, T, H))
    S0 = r.standard_normal((1, H, D, D))
    o, S = orc.recurrent(q, k, v, g, beta, S0)
    np.testing.assert_array_equal(S, S0)
    scale = 1.0 / math.sqrt(D)
    for t in range(T):
        for h in range(H):
            np.testing.assert_allclose(o[0, t, h], scale * S0[0, h].T @ q[0, t, h], atol=1e-12)


def test_beta0_pure_decay_closed_form(orc):
    """beta = 0: S_t = diag(exp(Gamma_t)) S0 with Gamma_t the running sum of g;
    decay scales rows (key channels), never columns."""
    r = rng(4)
    D, T, H = 128, 7, 2
    q, k, v, g, _ = rand_inputs(r, 1, T, H, D)
    beta = np.zeros((1, T, H))
    S0 = r.standard_normal((1, H, D, D))
    o, S, snaps = orc.recurrent(q, k, v, g, beta, S0, snapshots=True)
    gam = np.cumsum(g[0], axis=0)  # [T, H, D]
    scale = 1.0 / math.sqrt(D)
    for t in range(T):
        for h in range(H):
            expect = np.exp(gam[t, h])[:, None] * S0[0, h]
            np.testing.assert_allclose(snaps[t, 0, h], expect, rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(o[0, t, h], scale * expect.T @ q[0, t, h],
                                       rtol=1e-12, atol=1e-14)


def test_delta_rule_overwrites_basis_row(orc):
    """g = 0, beta = 1, k = e_i: row i of S becomes v, other rows untouched."""
    r = rng(5)
    D = 16
    S0 = r.standard_normal((1, 1, D, D))
    for i in (0, 7, 15):
        k = np.zeros((1, 1, 1, D))
        k[..., i] = 1.0
        v = r.standard_normal((1, 1, 1, D))
        q = r.standard_normal((1, 1, 1, D))
        _, S = orc.recurrent(q, k, v, np.zeros_like(q), np.ones((1, 1, 1)), S0)
        expect = S0[0, 0].copy()
        expect[i] = v[0, 0, 0]
        np.testing.assert_allclose(S[0, 0], expect, atol=1e-15)


def test_readout_uses_updated_state(orc):
    """o_t reads the state after token t's update: with S0 = 0 and q = k the
    first output is scale * beta * |k|^2 * v, not zero."""
    r = rng(6)
    D = 32
    _, k, v, g, beta = rand_inputs(r, 1, 1, 1, D)
    o, _ = orc.recurrent(k, k, v, g, beta, np.zeros((1, 1, D, D)))
    np.testing.assert_allclose(o[0, 0, 0], beta[0, 0, 0] / math.sqrt(D) * v[0, 0, 0],
                               atol=1e-14)


def test_default_scale_is_inverse_sqrt_head_dim(orc):
    assert orc.q_scale(128) == pytest.approx(1.0 / math.sqrt(128), rel=0, abs=1e-17)


# ---------------------------------------------------------------- invariants

def test_sequences_and_heads_are_independent(orc):
    """Permuting sequences or heads permutes the results the same way."""
    r = rng(7)
    q, k, v, g, beta = rand_inputs(r, 3, 6, 2, 32)
    S0 = r.standard_normal((3, 2, 32, 32))
    o, S = orc.recurrent(q, k, v, g, beta, S0)
    pn, ph = [2, 0, 1], [1, 0]
    o2, S2 = orc.recurrent(q[pn][:, :, ph], k[pn][:, :, ph], v[pn][:, :, ph],
                           g[pn][:, :, ph], beta[pn][:, :, ph], S0[pn][:, ph])
    np.testing.assert_array_equal(o2, o[pn][:, :, ph])
    np.testing.assert_array_equal(S2, S[pn][:, ph])


def test_causality(orc):
    """Perturbing token t' leaves every output before t' unchanged."""
    r = rng(8)
    T = 20
    q, k, v, g, beta = rand_inputs(r, 1, T, 2, 64)
    S0 = r.standard_normal((1, 2, 64, 64)) * 0.1
    o, _ = orc.recurrent(q, k, v, g, beta, S0)
    for tp in (0, 7, 19):
        v2, g2 = v.copy(), g.copy()
        v2[0, tp] += 1.0
        g2[0, tp] -= 0.5
        o2, _ = orc.recurrent(q, k, v2, g2, beta, S0)
        np.testing.assert_array_equal(o2[0, :tp], o[0, :tp])
        assert np.abs(o2[0, tp] - o[0, tp]).max() > 1e-6


def test_split_run_equals_whole_run(orc):
    """The state carries everything: running T tokens in two calls equals one call."""
    r = rng(9)
    q, k, v, g, beta = rand_inputs(r, 2, 15, 2, 32)
    S0 = r.standard_normal((2, 2, 32, 32)) * 0.1
    o, S = orc.recurrent(q, k, v, g, beta, S0)
    oa, Sa = orc.recurrent(q[:, :6], k[:, :6], v[:, :6], g[:, :6], beta[:, :6], S0)
    ob, Sb = orc.recurrent(q[:, 6:], k[:, 6:], v[:, 6:], g[:, 6:], beta[:, 6:], Sa)
    np.testing.assert_allclose(np.concatenate([oa, ob], axis=1), o, atol=1e-14)
    np.testing.assert_allclose(Sb, S, atol=1e-14)


# ---------------------------------------------------------- chunked form

@pytest.mark.parametrize("C,T", [(1, 9), (16, 50), (64, 100), (64, 64), (16, 16)])
def test_chunked_equals_recurrent(orc, C, T):
    """chunk_prepare + chunk_scan reproduce the token recurrence (the two forms
    agree up to rounding), including a partial last chunk."""
    r = rng(10 + C)
    H, D = 2, 128
    q, k, v, g, beta = rand_inputs(r, 1, T, H, D)
    S0 = r.standard_normal((H, D, D)) * 0.02
    o_ref, S_ref = orc.prefill(q[0], k[0], v[0], g[0], beta[0], S0)
    o_ch, S_ch = orc.chunked(q[0], k[0], v[0], g[0], beta[0], S0, C)
    assert np.abs(o_ch - o_ref).max() / np.abs(o_ref).max() < 1e-12
    assert np.abs(S_ch - S_ref).max() / np.abs(S_ref).max() < 1e-12


def test_prepare_stages_against_library_routines(orc):
    """Gamma is numpy's cumsum; T is numpy's inverse of (I + A); A is strictly
    lower and P lower triangular; W = T Ktil and Ut = T V by matmul."""
    r = rng(11)
    L, D = 40, 128
    q, k, v, g, beta = (a[0, :, 0] for a in rand_inputs(r, 1, L, 1, D))
    p = orc.chunk_prepare(q, k, v, g, beta)
    np.testing.assert_allclose(p["Gamma"], np.cumsum(g, axis=0), rtol=1e-14, atol=1e-12)
    Tinv = np.linalg.inv(np.eye(L) + p["A"])
    np.testing.assert_allclose(p["T"], Tinv, atol=1e-12)
    assert np.all(np.triu(p["A"]) == 0.0)
    assert np.all(np.triu(p["P"], 1) == 0.0)
    ktil = np.exp(p["Gamma"]) * k
    np.testing.assert_allclose(p["W"], Tinv @ ktil, atol=1e-12)
    np.testing.assert_allclose(p["Ut"], Tinv @ v, atol=1e-12)
    np.testing.assert_allclose(p["dec"], np.exp(p["Gamma"][-1]), rtol=1e-14)


def test_prepare_residuals_match_recurrence(orc):
    """From a zero state the chunk's residuals U = T V must equal the u_t the
    token recurrence forms, recovered from its successive states as
    u_t = (S_t - diag(exp g_t) S_{t-1})^T k_t / (beta_t |k_t|^2)."""
    r = rng(12)
    L, D = 24, 64
    q, k, v, g, beta = rand_inputs(r, 1, L, 1, D)
    _, _, snaps = orc.recurrent(q, k, v, g, beta, np.zeros((1, 1, D, D)), snapshots=True)
    prev = np.zeros((D, D))
    u_rec = np.zeros((L, D))
    for t in range(L):
        cur = snaps[t, 0, 0]
        kt = k[0, t, 0]
        u_rec[t] = (cur - np.exp(g[0, t, 0])[:, None] * prev).T @ kt / (beta[0, t, 0] * kt @ kt)
        prev = cur
    p = orc.chunk_prepare(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0])
    np.testing.assert_allclose(p["Ut"], u_rec, atol=1e-10)


def test_scan_from_prepared_chunks_matches(orc):
    """Driving chunk_scan by hand over prepared chunks equals the recurrence."""
    r = rng(13)
    T, C, D = 37, 16, 64
    q, k, v, g, beta = rand_inputs(r, 1, T, 1, D)
    S0 = r.standard_normal((D, D)) * 0.05
    o_ref, S_ref = orc.prefill(q[0], k[0], v[0], g[0], beta[0], S0[None])
    S = S0.copy()
    outs = []
    for c0 in range(0, T, C):
        sl = slice(c0, min(T, c0 + C))
        p = orc.chunk_prepare(q[0, sl, 0], k[0, sl, 0], v[0, sl, 0], g[0, sl, 0],
                              beta[0, sl, 0])
        o, S = orc.chunk_scan(p, beta[0, sl, 0], S)
        outs.append(o)
    np.testing.assert_allclose(np.concatenate(outs), o_ref[:, 0], atol=1e-12)
    np.testing.assert_allclose(S, S_ref[0], atol=1e-12)


# ------------------------------------------------------------- conv front end

def _conv_inputs(r, lengths, H, D, K):
    ch = 3 * H * D
    total = sum(lengths)
    x = r.standard_normal((total, ch))
    w = r.standard_normal((ch, K)) * 0.5
    st = r.standard_normal((len(lengths), ch, K))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return x, w, st, cu


def test_conv_against_torch_conv1d(orc):
    """Depthwise causal conv + SiLU equals torch's grouped conv1d with the
    history prepended, then F.silu; q and k heads then scaled by
    1/sqrt(sum y^2 + eps); v channels as they are."""
    r = rng(20)
    H, D, K, eps = 2, 16, 4, 1e-6
    lengths = [9, 1, 5]
    x, w, st, cu = _conv_inputs(r, lengths, H, D, K)
    out, st_new = orc.conv_silu_l2(x, w, st, cu, H, D, eps)
    ch = 3 * H * D
    for n, L in enumerate(lengths):
        xs = x[cu[n]:cu[n + 1]]
        hist = st[n][:, 1:].T  # slots 1..K-1 are the K-1 most recent inputs
        full = torch.tensor(np.concatenate([hist, xs], axis=0).T[None])  # [1, ch, K-1+L]
        y = torch.nn.functional.conv1d(full, torch.tensor(w)[:, None, :], groups=ch)[0].T
        y = torch.nn.functional.silu(y).numpy()
        ref = y.copy()
        for grp in range(2 * H):
            blk = y[:, grp * D:(grp + 1) * D]
            ref[:, grp * D:(grp + 1) * D] = blk / np.sqrt((blk ** 2).sum(1, keepdims=True) + eps)
        np.testing.assert_allclose(out[cu[n]:cu[n + 1]], ref, rtol=1e-12, atol=1e-13)
        seq_all = np.concatenate([st[n].T, xs], axis=0)  # K old slots then the new inputs
        np.testing.assert_array_equal(st_new[n], seq_all[-K:].T)


def test_conv_impulse_response_pins_tap_order(orc):
    """A unit impulse at token 0 on one v channel, zero state: output at token
    j is SiLU(w[c, K-1-j]), so tap K-1 multiplies the current token."""
    H, D, K = 1, 8, 4
    ch = 3 * H * D
    c = 2 * H * D + 3
    T = 6
    x = np.zeros((T, ch))
    x[0, c] = 1.0
    w = np.zeros((ch, K))
    w[c] = [0.5, -1.0, 2.0, 3.0]
    out, _ = orc.conv_silu_l2(x, w, np.zeros((1, ch, K)), [0, T], H, D)
    silu = lambda z: z / (1 + math.exp(-z))
    expect = [silu(w[c, K - 1 - j]) if j < K else 0.0 for j in range(T)]
    np.testing.assert_allclose(out[:, c], expect, atol=1e-15)


def test_conv_k1_unit_weight_is_silu_then_l2(orc):
    r = rng(21)
    H, D, eps = 1, 32, 1e-6
    x, _, _, cu = _conv_inputs(r, [7], H, D, 1)
    w = np.ones((3 * H * D, 1))
    out, _ = orc.conv_silu_l2(x, w, np.zeros((1, 3 * H * D, 1)), cu, H, D, eps)
    y = torch.nn.functional.silu(torch.tensor(x)).numpy()
    qk = y[:, :2 * D].reshape(7, 2, D)
    qk = qk / np.sqrt((qk ** 2).sum(-1, keepdims=True) + eps)
    np.testing.assert_allclose(out[:, :2 * D], qk.reshape(7, 2 * D), rtol=1e-13)
    np.testing.assert_allclose(out[:, 2 * D:], y[:, 2 * D:], rtol=1e-13)


def test_conv_streaming_equals_prefill(orc):
    """Decoding tokens one at a time (state carried) equals one prefill call."""
    r = rng(22)
    H, D, K = 1, 16, 3
    x, w, st, cu = _conv_inputs(r, [8], H, D, K)
    out, st_end = orc.conv_silu_l2(x, w, st, cu, H, D)
    s = st.copy()
    for t in range(8):
        o1, s = orc.conv_silu_l2(x[t:t + 1], w, s, [0, 1], H, D)
        np.testing.assert_allclose(o1[0], out[t], rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(s, st_end)


# ------------------------------------------------------------ gated RMSNorm

def _onorm_inputs(r, rows, H, D):
    core = r.standard_normal((rows, H, D)) * 3.0
    gate = r.standard_normal((rows, H * D))
    w = r.standard_normal(D)
    return core, gate, w


def test_o_norm_unit_rms_when_gate_open(orc):
    """w = 1, sigmoid(gate) = 1, eps = 0: every (token, head) comes out with
    mean square exactly 1 -- the norm runs over the head's channels."""
    r = rng(31)
    core, _, _ = _onorm_inputs(r, 5, 3, 16)
    out = orc.o_norm_gated(core, np.full((5, 48), 60.0), np.ones(16), eps=0.0)
    np.testing.assert_allclose((out * out).mean(-1), 1.0, rtol=1e-12)


def test_o_norm_scale_invariant_and_odd(orc):
    r = rng(32)
    core, gate, w = _onorm_inputs(r, 4, 2, 8)
    base = orc.o_norm_gated(core, gate, w, eps=0.0)
    np.testing.assert_allclose(orc.o_norm_gated(core * 7.5, gate, w, eps=0.0), base, rtol=1e-12)
    np.testing.assert_allclose(orc.o_norm_gated(-core, gate, w, eps=0.0), -base, rtol=1e-12)


def test_o_norm_gate_is_a_sigmoid(orc):
    """gate 0 halves the open-gate output; gate -g scales by 1 - sigmoid(g)."""
    r = rng(33)
    core, gate, w = _onorm_inputs(r, 3, 2, 8)
    open_ = orc.o_norm_gated(core, np.full(gate.shape, 60.0), w)
    np.testing.assert_allclose(orc.o_norm_gated(core, np.zeros(gate.shape), w), 0.5 * open_,
                               rtol=1e-12)
    pos = orc.o_norm_gated(core, gate, w)
    neg = orc.o_norm_gated(core, -gate, w)
    np.testing.assert_allclose(pos + neg, open_, rtol=1e-12, atol=1e-15)


def test_o_norm_weight_per_channel(orc):
    r = rng(34)
    core, gate, w = _onorm_inputs(r, 3, 4, 8)
    one = orc.o_norm_gated(core, gate, np.ones(8))
    np.testing.assert_allclose(orc.o_norm_gated(core, gate, w), one * w, rtol=1e-12)


def test_o_norm_eps_closed_form(orc):
    """A head whose channels all equal a: out = a / sqrt(a^2 + eps)."""
    a, eps = 0.01, 1e-4
    core = np.full((1, 1, 16), a)
    out = orc.o_norm_gated(core, np.full((1, 16), 60.0), np.ones(16), eps=eps)
    np.testing.assert_allclose(out, a / math.sqrt(a * a + eps), rtol=1e-12)


def test_o_norm_heads_and_rows_independent(orc):
    r = rng(35)
    core, gate, w = _onorm_inputs(r, 4, 3, 8)
    out = orc.o_norm_gated(core, gate, w)
    perm = [2, 0, 1]
    g3 = gate.reshape(4, 3, 8)
    out_p = orc.o_norm_gated(core[:, perm], g3[:, perm].reshape(4, 24), w)
    np.testing.assert_allclose(out_p, out[:, perm], rtol=1e-13)
    np.testing.assert_allclose(orc.o_norm_gated(core[1:2], gate[1:2], w), out[1:2], rtol=1e-13)


# ------------------------------------------------------------ input recipe

def test_workload_inputs_follow_recipe():
    d = wl.tiny()
    q, k = d["q"].double(), d["k"].double()
    n2 = (q * q).sum(-1)
    assert torch.allclose(n2, torch.ones_like(n2), atol=1e-5)
    assert torch.allclose((k * k).sum(-1), torch.ones_like(n2), atol=1e-5)
    assert d["g"].min() >= -5.0 and d["g"].max() <= 0.0
    assert d["beta"].min() > 0.0 and d["beta"].max() < 1.0
    assert d["state"].abs().max() == 0.0
    d2 = wl.tiny()
    for n in ("q", "k", "v", "g", "beta"):
        assert torch.equal(d[n], d2[n])


# ---------------------------------------------------------------- forget gate and beta
# The formula is a reading (the pages give its inputs and its bound, not the
# expression): g = lb * sigmoid(exp(a_log[h]) * (g_raw + dt_bias[c])),
# beta = sigmoid(b).  These pins fix everything but that choice: the closed
# form at a zero argument, the limits, the range, the monotonicity, and which
# parameter broadcasts over which axis.

def _gate_inputs(seed, rows=5, H=3, D=8):
    rng = np.random.default_rng(seed)
    return (rng.normal(size=(rows, H * D)), rng.normal(size=H * D) * 0.5,
            rng.normal(size=H) * 0.5, rng.normal(size=(rows, H)))


def test_gate_zero_argument_is_half_the_bound(orc):
    g_raw, dt, al, b = _gate_inputs(1)
    g, _ = orc.gate(-np.broadcast_to(dt, g_raw.shape), dt, al, -5.0, b)
    assert np.allclose(g, -2.5, rtol=0, atol=1e-15)


def test_gate_hand_value(orc):
    """a_log = 0 (rate 1) and g_raw + dt_bias = 1: g = lb / (1 + e^-1)."""
    g, beta = orc.gate(np.ones((1, 4)), np.zeros(4), np.zeros(1), -4.0, np.zeros((1, 1)))
    assert np.allclose(g, -4.0 * 0.7310585786300049, rtol=0, atol=1e-15)
    assert beta[0, 0] == 0.5


def test_gate_limits_and_range(orc):
    g_raw, dt, al, b = _gate_inputs(2)
    lb = -7.0
    g, _ = orc.gate(g_raw, dt, al, lb, b)
    assert np.all(g < 0) and np.all(g > lb)
    big = np.full_like(g_raw, 1e4)
    g_hi, _ = orc.gate(big, dt, al, lb, b)        # the strongest decay: the bound
    g_lo, _ = orc.gate(-big, dt, al, lb, b)       # no decay: zero
    assert np.allclose(g_hi, lb, rtol=0, atol=1e-12)
    assert np.allclose(g_lo, 0.0, rtol=0, atol=1e-12)
    g_slow, _ = orc.gate(g_raw, dt, np.full_like(al, -60.0), lb, b)  # rate -> 0
    assert np.allclose(g_slow, lb / 2, rtol=0, atol=1e-12)


def test_gate_is_monotone_in_the_projection(orc):
    g_raw, dt, al, b = _gate_inputs(3)
    g1, _ = orc.gate(g_raw, dt, al, -5.0, b)
    g2, _ = orc.gate(g_raw + 0.1, dt, al, -5.0, b)
    assert np.all(g2 < g1)  # a larger projection decays faster (lb < 0)


def test_gate_broadcasts_bias_per_channel_and_rate_per_head(orc):
    g_raw, dt, al, b = _gate_inputs(4, rows=4, H=3, D=8)
    g0, _ = orc.gate(g_raw, dt, al, -5.0, b)
    dt2 = dt.copy()
    dt2[8 + 5] += 1.0                      # channel 5 of head 1
    g1, _ = orc.gate(g_raw, dt2, al, -5.0, b)
    changed = np.argwhere(np.abs(g1 - g0) > 0)
    assert set(map(tuple, changed[:, 1:])) == {(1, 5)}
    al2 = al.copy()
    al2[2] += 0.5                          # head 2
    g2, _ = orc.gate(g_raw, dt, al2, -5.0, b)
    diff = np.abs(g2 - g0) > 0
    assert diff[:, 2].all() and not diff[:, :2].any()


def test_beta_is_the_logistic_function(orc):
    _, _, _, b = _gate_inputs(5)
    _, beta = orc.gate(np.zeros((5, 24)), np.zeros(24), np.zeros(3), -5.0, b)
    _, beta_neg = orc.gate(np.zeros((5, 24)), np.zeros(24), np.zeros(3), -5.0, -b)
    assert np.allclose(beta + beta_neg, 1.0, rtol=0, atol=1e-15)
    assert np.allclose(beta, 1.0 / (1.0 + np.exp(-b)), rtol=1e-15, atol=0)
