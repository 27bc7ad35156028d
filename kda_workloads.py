"""Seeded synthetic inputs for the KDA core workloads.

This module only draws random tensors; it holds none of the method's
arithmetic (no decay, no delta-rule update, no convolution).  Both the CUDA
path and the CPU oracle consume the exact host tensors produced here, so the
two sides see bit-identical inputs.

Recipe (from the five workload descriptions this library is measured on):

* q, k: N(0, 1) per channel, then each (token, head) vector is scaled to unit
  length as ``x / sqrt(sum x^2 + 1e-6)`` in float64 before rounding to the
  input dtype.  This is how the workloads draw a random *direction*; the core
  itself consumes q and k as given.
* v: N(0, 1).
* g (log-decay): uniform in [-5, 0] per (token, head, key channel).
* beta: sigmoid(N(0, 1)) per (token, head).
* initial state: zero, or N(0, 0.02) (standard deviation 0.02) where stated.
* conv front end: x ~ N(0, 1) BF16 over q|k|v channels, depthwise weights
  ~ N(0, 0.5) BF16, zero conv state.

Draw order within one call is q, k, v, g, beta, then the state, from one
``torch.Generator`` seeded by the caller (seed 0 for every named workload).
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

HEAD_DIM = 128
UNIT_EPS = 1e-6


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _unit_directions(gen: torch.Generator, shape, dtype) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float64)
    x = x / torch.sqrt((x * x).sum(dim=-1, keepdim=True) + UNIT_EPS)
    return x.to(dtype)


def core_inputs(gen: torch.Generator, lead: tuple, heads: int, dtype=torch.float32,
                head_dim: int = HEAD_DIM, g_low: float = -5.0) -> dict:
    """q, k, v, g of shape lead+(heads, head_dim) and beta of lead+(heads,)."""
    shp = tuple(lead) + (heads, head_dim)
    q = _unit_directions(gen, shp, dtype)
    k = _unit_directions(gen, shp, dtype)
    v = torch.randn(shp, generator=gen, dtype=torch.float64).to(dtype)
    g = (torch.rand(shp, generator=gen, dtype=torch.float64) * (-g_low) + g_low).to(dtype)
    beta = torch.sigmoid(torch.randn(tuple(lead) + (heads,), generator=gen,
                                     dtype=torch.float64)).to(dtype)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta}


def state(gen: torch.Generator, lead: tuple, heads: int, std: float,
          head_dim: int = HEAD_DIM) -> torch.Tensor:
    shp = tuple(lead) + (heads, head_dim, head_dim)
    if std == 0.0:
        return torch.zeros(shp, dtype=torch.float32)
    return (torch.randn(shp, generator=gen, dtype=torch.float64) * std).to(torch.float32)


def pad_rows(x: torch.Tensor, t_pad: int, fill: float = 0.0) -> torch.Tensor:
    """Extend dim 0 to ``t_pad`` rows filled with ``fill`` (harness padding)."""
    t = x.shape[0]
    if t_pad == t:
        return x
    out = torch.full((t_pad,) + tuple(x.shape[1:]), fill, dtype=x.dtype)
    out[:t] = x
    return out


# ---------------------------------------------------------------- workloads

@dataclass(frozen=True)
class Workload:
    name: str
    description: str


TINY = Workload("kda_tiny_T64_H2_C16_f32",
                "1 sequence, T=64, heads=2, head_dim=128, chunk=16, FP32, zero state")
DECODE = Workload("kda_decode_N64_H32_f32_x100",
                  "64 sequences x 1 token, heads=32, FP32 state [64,32,128,128] "
                  "~N(0,0.02), 100 chained steps")
PREFILL = Workload("kda_prefill_T8192_H32_C64_bf16",
                   "1 sequence, T=8192, heads=32, chunk=64, BF16 q/k/v/g/beta, "
                   "FP32 state ~N(0,0.02) and FP32 o")
DECODE_K = Workload("kda_decode_k_N128_k4_H32_f32",
                    "128 sequences x k=4 rows, heads=32, FP32, snapshot after each row")
FRONTEND = Workload("kda_conv_core_16seq_512to8192_H32_C64_bf16",
                    "16 sequences, lengths U{512..8192}, conv K=4 over 3x4096 BF16 "
                    "channels, then the chunked core")


def tiny(seed: int = 0, t: int = 64, heads: int = 2, dtype=torch.float32) -> dict:
    gen = _gen(seed)
    d = core_inputs(gen, (t,), heads, dtype)
    d["state"] = state(gen, (1,), heads, 0.0)
    d["chunk"] = 16
    return d


def decode_steps(seed: int = 0, n_seqs: int = 64, heads: int = 32, steps: int = 100,
                 state_std: float = 0.02) -> dict:
    """Initial state then ``steps`` fresh single-token inputs, [steps, N, H, D]."""
    gen = _gen(seed)
    s0 = state(gen, (n_seqs,), heads, state_std)
    d = core_inputs(gen, (steps, n_seqs), heads, torch.float32)
    d["state"] = s0
    return d


def prefill(seed: int = 0, t: int = 8192, heads: int = 32, chunk: int = 64,
            dtype=torch.bfloat16, state_std: float = 0.02) -> dict:
    gen = _gen(seed)
    d = core_inputs(gen, (t,), heads, dtype)
    d["state"] = state(gen, (1,), heads, state_std)
    d["chunk"] = chunk
    return d


def decode_k(seed: int = 0, n_seqs: int = 128, krows: int = 4, heads: int = 32,
             state_std: float = 0.02) -> dict:
    gen = _gen(seed)
    d = core_inputs(gen, (n_seqs, krows), heads, torch.float32)
    d["state"] = state(gen, (n_seqs,), heads, state_std)
    return d


def seq_lengths(gen: torch.Generator, n: int, lo: int, hi: int) -> list:
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def frontend(seed: int = 0, n_seqs: int = 16, lo: int = 512, hi: int = 8192,
             heads: int = 32, conv_kernel: int = 4, lengths=None) -> dict:
    """Packed varlen batch: x [sum T, 3*H*D] BF16, w [3*H*D, K] BF16, zero conv
    state, g [sum T, H, D] and beta [sum T, H] (BF16), zero per-sequence state."""
    gen = _gen(seed)
    if lengths is None:
        lengths = seq_lengths(gen, n_seqs, lo, hi)
    n_seqs = len(lengths)
    total = int(sum(lengths))
    ch = 3 * heads * HEAD_DIM
    # x is the largest draw (sum T x 12288 values): FP32 draws, rounded to BF16.
    x = torch.randn((total, ch), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    w = (torch.randn((ch, conv_kernel), generator=gen, dtype=torch.float64) * 0.5
         ).to(torch.bfloat16)
    g = (torch.rand((total, heads, HEAD_DIM), generator=gen, dtype=torch.float32) * 5.0
         - 5.0).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((total, heads), generator=gen, dtype=torch.float64)
                         ).to(torch.bfloat16)
    cu = [0]
    for L in lengths:
        cu.append(cu[-1] + L)
    return {
        "lengths": lengths, "cu_seqlens": torch.tensor(cu, dtype=torch.int32),
        "x": x, "w": w, "g": g, "beta": beta,
        "conv_state": torch.zeros((n_seqs, ch, conv_kernel), dtype=torch.float32),
        "state": torch.zeros((n_seqs, heads, HEAD_DIM, HEAD_DIM), dtype=torch.float32),
        "chunk": 64, "conv_kernel": conv_kernel, "l2_eps": 1e-6,
    }



def gate_inputs(gen: torch.Generator, rows: int, heads: int, g_pitch_extra: int = 0,
                b_pitch_extra: int = 0) -> dict:
    """Raw inputs of the forget gate and beta: the gate projection g_raw BF16
    [rows, H*D + g_pitch_extra] ~N(0, 1), dt_bias FP32 [H*D] ~N(0, 0.25),
    a_log FP32 [H] ~N(0, 0.25), the b_proj output b_raw BF16
    [rows, H + b_pitch_extra] ~N(0, 1), and gate_lower_bound -5."""
    g_raw = torch.randn((rows, heads * HEAD_DIM + g_pitch_extra), generator=gen,
                        dtype=torch.float32).to(torch.bfloat16)
    dt_bias = torch.randn(heads * HEAD_DIM, generator=gen, dtype=torch.float32) * 0.5
    a_log = torch.randn(heads, generator=gen, dtype=torch.float32) * 0.5
    b_raw = torch.randn((rows, heads + b_pitch_extra), generator=gen,
                        dtype=torch.float32).to(torch.bfloat16)
    return {"g_raw": g_raw, "dt_bias": dt_bias, "a_log": a_log, "b_raw": b_raw,
            "gate_lower_bound": -5.0}


def prefill_gated(seed: int = 0, t: int = 8192, heads: int = 32, g_pitch_extra: int = 0,
                  b_pitch_extra: int = 0, state_std: float = 0.02) -> dict:
    """The prefill workload with raw gate inputs in place of g and beta: q, k,
    v BF16 [t, H, D] as in prefill(), then the gate_inputs() draws, then the
    state."""
    gen = _gen(seed)
    d = core_inputs(gen, (t,), heads, torch.bfloat16)
    del d["g"], d["beta"]
    d.update(gate_inputs(gen, t, heads, g_pitch_extra, b_pitch_extra))
    d["state"] = state(gen, (1,), heads, state_std)
    return d
