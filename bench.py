"""Benchmark of the KDA core on one GB300 (or N independent replicas).

One step = one kda_prefill of the chunked-prefill workload: 1 sequence of
8192 tokens, 32 heads, head_dim 128, chunk 64, BF16 q/k/v/g/beta, FP32 state
and output, inputs resident in HBM (400 MB per step, larger than the 129 MB
L2, so no flush is needed between steps).  The state carries from step to
step, as one long prefill would.  The same run also times the decode
workload (64 sequences x 32 heads, 100 chained steps) and the decode_k
workload (128 sequences x k=4 rows, 4 snapshots) and reports their state
GB/s against the HBM peak.

Prints ONE JSON line on rank 0.  `--impl reference` times the FP64 CPU oracle
instead (a bounded sample of the same workload per step).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import kda_workloads as wl  # noqa: E402

METRIC = "KDA prefill tokens/s and decode state GB/s (% of HBM peak), 1xGB300"
T_PREFILL, H, D, CHUNK = 8192, 32, 128, 64
# Algorithmic bytes of one prefill launch: q, k, v, g BF16 [8192, 32, 128],
# beta BF16 [8192, 32], o FP32 [8192, 32, 128], state FP32 read + write.
PREFILL_BYTES = 4 * T_PREFILL * H * D * 2 + T_PREFILL * H * 2 + T_PREFILL * H * D * 4 \
    + 2 * H * D * D * 4
# Multiply-adds x 2 of the chunked form per token-head: 6 D^2 + 5 C D + C^2 / 3.
PREFILL_FLOPS = T_PREFILL * H * (6 * D * D + 5 * CHUNK * D + CHUNK * CHUNK / 3)
DECODE_N, DECODE_STEPS = 64, 100
DECODE_BYTES = 2 * DECODE_N * H * D * D * 4 + 4 * DECODE_N * H * D * 4 + DECODE_N * H * 4
DK_N, DK_K = 128, 4
CONV_K = 4
DK_BYTES = (2 + DK_K) * DK_N * H * D * D * 4 + 4 * DK_N * DK_K * H * D * 4 + DK_N * DK_K * H * 4
ONORM_BYTES = T_PREFILL * 32 * 128 * (4 + 2 + 2) + 128 * 2  # core FP32, gate and out BF16, w
# the forget gate and beta of a prefill-sized problem (8192 rows x 32 heads):
# BF16 g_raw in and BF16 g out per channel, BF16 b in and BF16 beta out per head,
# dt_bias and a_log once
GATE_BYTES = T_PREFILL * H * D * (2 + 2) + T_PREFILL * H * (2 + 2) + H * D * 4 + H * 4
SHORT_T = 4
SHORT_BYTES = 2 * DECODE_N * H * D * D * 4 + 5 * DECODE_N * SHORT_T * H * D * 4 + DECODE_N * SHORT_T * H * 4
CONVK_BYTES = (DK_N * DK_K * 3 * H * D * 2 * 2 + 3 * H * D * CONV_K * 2
               + (2 + DK_K) * DK_N * 3 * H * D * CONV_K * 4)  # x, out, w, state R/W, snapshots
TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense TF32 : BF16 tensor ratio of the part


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        m = json.load(open(path))
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")
                  if k in m})
        p["source"] = "measured"
    return p


def kernel_source_sha() -> str:
    """Hash of the sources the prefill kernels are built from."""
    h = hashlib.sha256()
    for name in ("prefill_tc.cu", "prefill.cu", "sm103_tc.h", "kda_common.h", "tma_map.h",
                 "f32x2.h"):
        h.update(open(os.path.join(ROOT, "gated_delta_rule_prepare_gb300", "csrc", name),
                      "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """Per-launch DRAM bytes of the prefill kernel from the committed ncu
    summary, valid only while the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "prefill_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    if rec.get("source_sha") != kernel_source_sha():
        return None
    return rec.get("traffic_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                rows.append({"sm": float(f[1]), "max": float(f[2]), "util": float(f[4]),
                             "hw": f[6], "hwt": f[7], "swt": f[8], "pcap": f[9]})
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        load = [r for r in rows if r["util"] > 0] or rows
        reasons = set()
        for r in load:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples_under_load": len(load)}


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------- GPU arm

def hbm_frac(gbs: float, peak: float):
    """The fraction of the measured HBM copy peak, or None above 1: a figure
    over the copy peak means part of the traffic came from L2 and is not an
    HBM number."""
    f = gbs / peak
    return f if f <= 1.0 else None

def time_launches(fn, n: int, stream):
    """Runs fn() n times back to back between one pair of events on `stream`;
    returns (the per-call ms as a list of n equal values, the total ms).
    Per-call event pairs would overlap: with programmatic dependent launch a
    call's first kernel may be scheduled while the previous call's last kernel
    still drains, so only the span of the whole sequence is a clean measure."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    total = e0.elapsed_time(e1)
    return [total / n] * n, total


def run_gpu(args):
    import gated_delta_rule_prepare_gb300 as K

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    pk = peaks()
    stream = torch.cuda.current_stream(dev)

    # ---------------- prefill workload (the step)
    d = wl.prefill()
    q, k, v, g, beta = (d[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
    S = d["state"].to(dev)
    o = torch.empty((T_PREFILL, H, D), device=dev)
    ws = torch.empty(K.kda_prefill_workspace_size(T_PREFILL, 1, CHUNK, H), dtype=torch.uint8,
                     device=dev)

    def prefill():
        K.kda_prefill(S, q, k, v, g, beta, o, T_PREFILL, CHUNK, workspace=ws)

    for _ in range(args.warmup):
        prefill()
    K.kda_sync_status()

    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        per, total_ms = time_launches(prefill, args.steps, stream)
        torch.cuda.synchronize()
        barrier(world)
        wall = time.perf_counter() - t0
        K.kda_sync_status()
        ms_step = max_over_ranks(total_ms / args.steps, world, dev)

        # ---------------- decode workload: 100 chained steps
        # Two batches of 64 sequences (two state sets of 128 MiB) take turns,
        # as two micro-batches of a serving loop would: each step's state was
        # last touched two steps ago, with the other 128 MiB set in between,
        # so the L2 (129 MB) cannot hold it from one step to its next.  The
        # single-set figure (state partly L2-resident) is reported beside it.
        dd = wl.decode_steps()
        dS_sets = [dd["state"].to(dev), dd["state"].to(dev)]
        dq, dk, dv, dg, db = (dd[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
        do = torch.empty((DECODE_N, H, D), device=dev)
        step = [0]
        sets_used = [2]

        def decode():
            t = step[0] % DECODE_STEPS
            K.kda_decode(dS_sets[step[0] % sets_used[0]], dq[t], dk[t], dv[t], dg[t], db[t], do)
            step[0] += 1

        for _ in range(5):
            decode()
        # The chain of 100 steps is the unit: one event pair around it, so the
        # launches follow each other as in a serving loop; reported per step.
        def decode_chain():
            per = []
            for _ in range(3):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                for _ in range(DECODE_STEPS):
                    decode()
                e1.record(stream)
                torch.cuda.synchronize()
                per.append(e0.elapsed_time(e1) / DECODE_STEPS)
            return [statistics.median(per)]

        dec_per = decode_chain()
        sets_used[0] = 1
        for _ in range(5):
            decode()
        dec1_per = decode_chain()
        del dq, dk, dv, dg, db, dS_sets

        # ---------------- decode_k workload
        kd = wl.decode_k()
        kS = kd["state"].to(dev)
        kin = {n: kd[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        ko = torch.empty((DK_N, DK_K, H, D), device=dev)
        snaps = [torch.empty_like(kS) for _ in range(DK_K)]

        def decode_k():
            K.kda_decode_k(kS, kin["q"], kin["k"], kin["v"], kin["g"], kin["beta"], ko, snaps)

        for _ in range(3):
            decode_k()
        dk_per, _ = time_launches(decode_k, 20, stream)
        del kS, snaps, kin

        # ---------------- short FP32 prefill (t = 4): decode_k's row walk vs the
        # SIMT chunk kernel it replaces (pinned through KDA_PREFILL_IMPL=simt)
        sgen = torch.Generator(device="cpu").manual_seed(0)
        sd = wl.core_inputs(sgen, (DECODE_N, SHORT_T), H, torch.float32)
        s_in = {n: sd[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
        s_S = wl.state(sgen, (DECODE_N,), H, 0.02).to(dev)
        s_o = torch.empty((DECODE_N, SHORT_T, H, D), device=dev)

        def short_prefill():
            K.kda_prefill(s_S, s_in["q"], s_in["k"], s_in["v"], s_in["g"], s_in["beta"], s_o,
                          SHORT_T, 16)

        short_us = {}
        for mode in ("row_walk", "simt"):
            if mode == "simt":
                os.environ["KDA_PREFILL_IMPL"] = "simt"
            for _ in range(3):
                short_prefill()
            sp_per, _ = time_launches(short_prefill, 20, stream)
            short_us[mode] = statistics.mean(sp_per) * 1e3
            os.environ.pop("KDA_PREFILL_IMPL", None)
        del s_in, s_S, s_o

        # ---------------- k-row conv with snapshots (decode_k's front end)
        cgen = torch.Generator(device="cpu").manual_seed(0)
        ck_x = torch.randn((DK_N, DK_K, 3 * H * D), generator=cgen).to(torch.bfloat16).to(dev)
        ck_w = (torch.randn((3 * H * D, CONV_K), generator=cgen) * 0.5).to(torch.bfloat16).to(dev)
        ck_st = torch.zeros((DK_N, 3 * H * D, CONV_K), device=dev)
        ck_o = torch.empty_like(ck_x)
        ck_snaps = [torch.empty_like(ck_st) for _ in range(DK_K)]

        def conv_k():
            K.kda_conv_silu_l2_k(ck_st, ck_x, ck_w, ck_o, ck_snaps)

        for _ in range(3):
            conv_k()
        ck_per, _ = time_launches(conv_k, 20, stream)
        del ck_x, ck_st, ck_o, ck_snaps

        # ---------------- gated RMSNorm of a prefill-sized core output
        ngen = torch.Generator(device="cpu").manual_seed(0)
        # Two input/output sets, alternated (537 MB touched per pair of
        # launches), so no launch finds its inputs in L2.
        n_sets = [(torch.randn((T_PREFILL, H, D), generator=ngen).to(dev),
                   torch.randn((T_PREFILL, H * D), generator=ngen).to(torch.bfloat16).to(dev),
                   torch.empty((T_PREFILL, H * D), dtype=torch.bfloat16, device=dev))
                  for _ in range(2)]
        n_w = torch.ones(D, dtype=torch.bfloat16, device=dev)
        n_turn = [0]

        def o_norm():
            n_core, n_gate, n_out = n_sets[n_turn[0]]
            n_turn[0] ^= 1
            K.kda_o_norm_gated(n_core, n_gate, n_w, n_out)

        for _ in range(3):
            o_norm()
        on_per, _ = time_launches(o_norm, 20, stream)

        # ---------------- the prefill step with the gated RMSNorm fused into its
        # epilogue (BF16 out, no FP32 o), against the step followed by o_norm
        pn_gate, pn_w, pn_out = n_sets[0][1], n_w, n_sets[0][2]

        def prefill_o_norm():
            K.kda_prefill_o_norm(S, q, k, v, g, beta, pn_gate, pn_w, pn_out, T_PREFILL, CHUNK,
                                 workspace=ws)

        for _ in range(3):
            prefill_o_norm()
        K.kda_sync_status()
        pn_per, _ = time_launches(prefill_o_norm, 20, stream)
        del n_sets

        # ---------------- forget gate and beta of a prefill-sized problem
        # Two input/output sets, alternated: consecutive launches touch 270 MB,
        # more than L2 holds, so no launch finds its inputs cached.
        g_sets = []
        for _ in range(2):
            g_sets.append((
                torch.randn((T_PREFILL, H * D), generator=ngen).to(torch.bfloat16).to(dev),
                torch.randn((T_PREFILL, H), generator=ngen).to(torch.bfloat16).to(dev),
                torch.empty((T_PREFILL, H, D), dtype=torch.bfloat16, device=dev),
                torch.empty((T_PREFILL, H), dtype=torch.bfloat16, device=dev)))
        g_dt = (torch.randn(H * D, generator=ngen) * 0.5).to(dev)
        g_al = (torch.randn(H, generator=ngen) * 0.5).to(dev)
        g_turn = [0]

        def gate():
            g_raw, g_b, g_out, g_beta = g_sets[g_turn[0]]
            g_turn[0] ^= 1
            K.kda_gate(g_raw, g_dt, g_al, g_b, g_out, g_beta, -5.0)

        for _ in range(3):
            gate()
        gate_per, _ = time_launches(gate, 20, stream)
        del g_sets

        # ---------------- the prefill step with the forget gate and beta formed
        # inside prepare from their raw inputs (the step's q, k, v and state)
        pgen = torch.Generator(device="cpu").manual_seed(1)
        gi = wl.gate_inputs(pgen, T_PREFILL, H)
        pg_in = {n: gi[n].to(dev) for n in ("g_raw", "dt_bias", "a_log", "b_raw")}

        def prefill_gated():
            K.kda_prefill_gated(S, q, k, v, pg_in["g_raw"], pg_in["dt_bias"], pg_in["a_log"],
                                pg_in["b_raw"], o, T_PREFILL, gi["gate_lower_bound"],
                                workspace=ws)

        for _ in range(3):
            prefill_gated()
        K.kda_sync_status()
        pg_per, _ = time_launches(prefill_gated, 20, stream)
        del pg_in

        # ---------------- the prefill step with FP32 inputs (the step's values
        # widened): FP16 copies of q, k and v made in the workspace, then the
        # same prepare and scan kernels
        f_in = [x_.float() for x_ in (q, k, v, g, beta)]
        f_ws = torch.empty(K.kda_prefill_workspace_size(T_PREFILL, 1, CHUNK, H, torch.float32),
                           dtype=torch.uint8, device=dev)

        def prefill_f32():
            K.kda_prefill(S, *f_in, o, T_PREFILL, CHUNK, workspace=f_ws)

        for _ in range(3):
            prefill_f32()
        K.kda_sync_status()
        pf_per, _ = time_launches(prefill_f32, 20, stream)
        del f_in, f_ws

        # ---------------- front end + core: 16 packed sequences, conv then prefill
        fe = wl.frontend()
        cu = fe["cu_seqlens"].to(dev)
        tot = int(fe["cu_seqlens"][-1])
        x = fe["x"].to(dev)
        wconv = fe["w"].to(dev)
        cst = fe["conv_state"].to(dev)
        xo = torch.empty_like(x)
        fg, fb = fe["g"].to(dev), fe["beta"].to(dev)
        fS = fe["state"].to(dev)
        fo = torch.empty((tot, H, D), device=dev)
        fws = torch.empty(K.kda_prefill_workspace_size(tot, len(fe["lengths"]), CHUNK, H),
                          dtype=torch.uint8, device=dev)
        hd = H * D

        def conv():
            K.kda_conv_silu_l2(cst, x, wconv, xo, cu_seqlens=cu)

        def core():
            K.kda_prefill(fS, xo[:, :hd].view(tot, H, D), xo[:, hd:2 * hd].view(tot, H, D),
                          xo[:, 2 * hd:].view(tot, H, D), fg, fb, fo, tot, CHUNK, cu_seqlens=cu,
                          workspace=fws)

        for _ in range(3):
            conv()
            core()
        conv_per, _ = time_launches(conv, 10, stream)
        core_per, _ = time_launches(core, 3, stream)
        K.kda_sync_status()
        n_fe = len(fe["lengths"])
        conv_bytes = tot * 3 * hd * 2 * 2 + 3 * hd * CONV_K * 2 + 2 * n_fe * 3 * hd * CONV_K * 4
        del x, xo, fg, fb, fS, fo, cst, fws
    clocks = clk.summary()

    # ---------------- end to end through the public API, host buffers
    host = {n: d[n].pin_memory() for n in ("q", "k", "v", "g", "beta")}
    o_host = torch.empty((T_PREFILL, H, D), dtype=torch.float32).pin_memory()
    S_host = torch.empty_like(S, device="cpu").pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o_host.numel() * 4 + S_host.numel() * 4

    # Steps are pipelined as a serving loop would run them: step i + 1's
    # inputs go up on one copy stream while step i computes, and step i - 1's
    # o and state come down on another; inputs and outputs are double-buffered
    # and the state is snapshotted on the device after each step, so no copy
    # reads a buffer a later step is writing.  Every step's copies stay inside
    # the timed region.
    comp = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    names = ("q", "k", "v", "g", "beta")
    dbuf = [dict(zip(names, (q, k, v, g, beta))),
            {n: torch.empty_like(t) for n, t in zip(names, (q, k, v, g, beta))}]
    obuf = [o, torch.empty_like(o)]
    sbuf = [torch.empty_like(S), torch.empty_like(S)]
    ev_in = [torch.cuda.Event(), torch.cuda.Event()]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]
    ev_out = [torch.cuda.Event(), torch.cuda.Event()]
    for b_ in range(2):  # nothing in flight yet
        for e_ in (ev_done[b_], ev_out[b_]):
            e_.record(comp)

    def e2e_run(n_steps):
        for i in range(n_steps):
            b_ = i & 1
            with torch.cuda.stream(s_in):  # inputs of step i (buffer free after step i - 2)
                s_in.wait_event(ev_done[b_])
                for n_ in names:
                    dbuf[b_][n_].copy_(host[n_], non_blocking=True)
                ev_in[b_].record(s_in)
            comp.wait_event(ev_in[b_])
            comp.wait_event(ev_out[b_])  # step i - 2's outputs have left this buffer
            x_ = dbuf[b_]
            K.kda_prefill(S, x_["q"], x_["k"], x_["v"], x_["g"], x_["beta"], obuf[b_], T_PREFILL,
                          CHUNK, workspace=ws)
            sbuf[b_].copy_(S, non_blocking=True)
            ev_done[b_].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[b_])
                o_host.copy_(obuf[b_], non_blocking=True)
                S_host.copy_(sbuf[b_], non_blocking=True)
                ev_out[b_].record(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    e_steps = max(3, min(args.steps, 20))
    barrier(world)
    t0 = time.perf_counter()
    e2e_run(e_steps)
    torch.cuda.synchronize()
    e_wall = max_over_ranks(time.perf_counter() - t0, world, dev)

    # ---------------- report
    avg_launch_s = ms_step / 1e3  # the span of the timed calls / K (see time_launches)
    achieved = PREFILL_BYTES / avg_launch_s / 1e9
    tf32_peak = pk["bf16_tflops"] * TF32_OVER_BF16
    t_bytes = PREFILL_BYTES / (pk["hbm_gbs"] * 1e9)
    t_flops = PREFILL_FLOPS / (tf32_peak * 1e12)
    bound = "hbm" if t_bytes >= t_flops else "tensor"
    dec_s = statistics.mean(dec_per) / 1e3
    dec1_s = statistics.mean(dec1_per) / 1e3
    dk_s = statistics.mean(dk_per) / 1e3
    value = world * T_PREFILL / (ms_step / 1e3)
    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 in; tf32 (A, P) and fp16 (scan) tensor-core operands; "
                 "fp32 accumulate, T solve and state",
        "data": "synthetic",
        "config": {
            "workload": wl.PREFILL.name,
            "description": wl.PREFILL.description,
            "seq_len": T_PREFILL, "heads": H, "head_dim": D, "chunk": CHUNK,
            "global_batch": world, "in_dtype": "bf16", "out_dtype": "f32 (o), f32 (state)",
            "l2": "inputs larger than L2 (400 MB per step), no flush",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {
            "bound": bound,
            "achieved": achieved if bound == "hbm" else PREFILL_FLOPS / avg_launch_s / 1e12,
            "peak": pk["hbm_gbs"] if bound == "hbm" else tf32_peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": (achieved / pk["hbm_gbs"]) if bound == "hbm"
            else (PREFILL_FLOPS / avg_launch_s / 1e12) / tf32_peak,
            "traffic": traffic_from_profile(),
            "kernel": "prefill (kda_prefill: chunk_map_kernel + prefill_fused_kernel, the "
                      "cooperative prepare + transposed-scan grid)",
            "algorithmic_bytes": PREFILL_BYTES, "algorithmic_flops": PREFILL_FLOPS,
            "avg_launch_us": avg_launch_s * 1e6,
            "peak_source": pk["source"] + " (hbm_gbs)",
            "time_floor_us": {"bytes": t_bytes * 1e6, "tf32_flops": t_flops * 1e6},
        },
        "e2e": {
            "value": world * T_PREFILL * e_steps / e_wall, "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "pinned host q/k/v/g/beta -> kda_prefill -> o and state to host; "
                    "copies on two copy streams overlap the neighbouring steps' compute",
        },
        # per prefill call: the chunk map and the fused prepare + scan grid
        "gpu_launches": 2 * args.steps,
        "clocks": clocks,
        "decode": {
            "workload": wl.DECODE.name, "value": DECODE_BYTES / dec_s / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": DECODE_BYTES / dec_s / 1e9 / pk["hbm_gbs"],
            "us_per_step": dec_s * 1e6, "algorithmic_bytes": DECODE_BYTES,
            "steps": DECODE_STEPS,
            "l2": "two state sets of 128 MiB alternated step by step (256 MiB), no flush",
            "single_state_set": {
                "value": DECODE_BYTES / dec1_s / 1e9, "unit": "GB/s",
                "us_per_step": dec1_s * 1e6,
                "l2": "one 128 MiB state set, partly L2-resident between steps"},
        },
        "decode_k": {
            "workload": wl.DECODE_K.name, "value": DK_BYTES / dk_s / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": DK_BYTES / dk_s / 1e9 / pk["hbm_gbs"],
            "us_per_call": dk_s * 1e6, "algorithmic_bytes": DK_BYTES,
        },
        "short_prefill": {
            "workload": "FP32 prefill, 64 sequences x 4 tokens x 32 heads (decode_k's row walk)",
            "value": SHORT_BYTES / short_us["row_walk"] / 1e3, "unit": "GB/s",
            "frac_of_hbm_peak": SHORT_BYTES / short_us["row_walk"] / 1e3 / pk["hbm_gbs"],
            "us_per_call": short_us["row_walk"], "simt_chunk_kernel_us": short_us["simt"],
            "algorithmic_bytes": SHORT_BYTES,
        },
        "conv_k": {
            "workload": "k-row conv + SiLU + L2, 128 sequences x 4 rows x 12288 channels, 4 snapshots",
            "value": CONVK_BYTES / (statistics.mean(ck_per) / 1e3) / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": CONVK_BYTES / (statistics.mean(ck_per) / 1e3) / 1e9
            / pk["hbm_gbs"],
            "us_per_call": statistics.mean(ck_per) * 1e3, "algorithmic_bytes": CONVK_BYTES,
            "gpu_launches_per_call": 2,
        },
        "o_norm": {
            "workload": "sigmoid-gated RMSNorm of a prefill-sized core output (8192 x 32 x 128)",
            "value": ONORM_BYTES / (statistics.mean(on_per) / 1e3) / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": hbm_frac(ONORM_BYTES / (statistics.mean(on_per) / 1e3) / 1e9,
                                         pk["hbm_gbs"]),
            "us_per_call": statistics.mean(on_per) * 1e3, "algorithmic_bytes": ONORM_BYTES,
            "l2": "two input/output sets alternated (537 MB touched per pair of launches), "
                  "no flush",
        },
        "prefill_o_norm": {
            "workload": "the prefill step (8192 x 32 heads, BF16) with the sigmoid-gated "
                        "RMSNorm fused into the scan's epilogue: BF16 out, no FP32 o",
            "value": T_PREFILL / (statistics.mean(pn_per) / 1e3), "unit": "tokens/s",
            "us_per_call": statistics.mean(pn_per) * 1e3,
            "prefill_then_o_norm_us": (ms_step + statistics.mean(on_per)) * 1e3,
        },
        "prefill_gated": {
            "workload": "the prefill step (8192 x 32 heads, BF16) with g and beta formed in "
                        "prepare from g_raw, dt_bias, a_log and b_raw",
            "value": T_PREFILL / (statistics.mean(pg_per) / 1e3), "unit": "tokens/s",
            "us_per_call": statistics.mean(pg_per) * 1e3,
            "gate_then_prefill_us": (statistics.mean(gate_per) + ms_step) * 1e3,
        },
        "prefill_f32": {
            "workload": "the prefill step (8192 x 32 heads) with FP32 q, k, v, g, beta: FP16 "
                        "copies of q, k, v, then the tensor-core kernels",
            "value": T_PREFILL / (statistics.mean(pf_per) / 1e3), "unit": "tokens/s",
            "us_per_call": statistics.mean(pf_per) * 1e3, "gpu_launches_per_call": 3,
        },
        "gate": {
            "workload": "forget gate and beta of a prefill-sized problem (8192 x 32 x 128, BF16)",
            "value": GATE_BYTES / (statistics.mean(gate_per) / 1e3) / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": GATE_BYTES / (statistics.mean(gate_per) / 1e3) / 1e9
            / pk["hbm_gbs"],
            "us_per_call": statistics.mean(gate_per) * 1e3, "algorithmic_bytes": GATE_BYTES,
            "l2": "two input/output sets alternated (270 MB touched per pair of launches), no flush",
        },
        "conv": {
            "workload": wl.FRONTEND.name + " (conv + SiLU + L2 stage)",
            "value": conv_bytes / (statistics.mean(conv_per) / 1e3) / 1e9, "unit": "GB/s",
            "frac_of_hbm_peak": conv_bytes / (statistics.mean(conv_per) / 1e3) / 1e9
            / pk["hbm_gbs"],
            "us_per_call": statistics.mean(conv_per) * 1e3, "algorithmic_bytes": conv_bytes,
            "tokens": tot, "gpu_launches_per_call": 2,
        },
        "frontend": {
            "workload": wl.FRONTEND.name, "lengths": fe["lengths"],
            "value": tot / ((statistics.mean(conv_per) + statistics.mean(core_per)) / 1e3),
            "unit": "tokens/s", "conv_us": statistics.mean(conv_per) * 1e3,
            "core_us": statistics.mean(core_per) * 1e3,
        },
        "wall_s_timed_region": wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_prefill(seconds=args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out))


# ------------------------------------------------------------ oracle (CPU)

def _oracle_prefill_sample(d, tokens):
    import oracle
    t0 = time.perf_counter()
    oracle.prefill(d["q"][:tokens], d["k"][:tokens], d["v"][:tokens], d["g"][:tokens],
                   d["beta"][:tokens], d["state"][0])
    return time.perf_counter() - t0


def cpu_baseline_prefill(seconds: float = 15.0):
    """The FP64 oracle on the host cores, on a bounded sample of the prefill
    workload: the first `tokens` tokens of the sequence, all 32 heads."""
    import oracle
    d = wl.prefill()
    tokens = 64
    dt = _oracle_prefill_sample(d, tokens)
    tokens = int(min(T_PREFILL, max(64, tokens * seconds / max(dt, 1e-3) / 2)))
    dt = _oracle_prefill_sample(d, tokens)
    return {"value": tokens / dt, "unit": "tokens/s", "cores": oracle.threads(),
            "kind": "oracle",
            "sample": "first %d tokens of the 8192-token sequence, all 32 heads, FP64, %.1f s"
                      % (tokens, dt)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    d = wl.prefill()
    tokens = 64   # one chunk of the sequence, all heads, per step
    for _ in range(args.warmup):
        _oracle_prefill_sample(d, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_prefill_sample(d, tokens)
    wall = time.perf_counter() - t0
    value = tokens * args.steps / wall
    sample = "per step: the first %d tokens of the 8192-token prefill workload, all 32 heads, " \
             "FP64 oracle on the host cores" % tokens
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": wall / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.PREFILL.name, "description": wl.PREFILL.description,
                   "seq_len": T_PREFILL, "heads": H, "head_dim": D, "chunk": CHUNK},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def run_case(args):
    """One kernel alone on a chosen size, for ncu captures: W + K launches."""
    import gated_delta_rule_prepare_gb300 as K
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(dev)
    if args.case == "prefill":
        d = wl.prefill(t=args.seq_len)
        q, k, v, g, beta = (d[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
        S = d["state"].to(dev)
        o = torch.empty((args.seq_len, H, D), device=dev)
        ws = torch.empty(K.kda_prefill_workspace_size(args.seq_len, 1, CHUNK, H),
                         dtype=torch.uint8, device=dev)
        fn = lambda: K.kda_prefill(S, q, k, v, g, beta, o, args.seq_len, CHUNK, workspace=ws)
        nbytes = 4 * args.seq_len * H * D * 2 + args.seq_len * H * 2 + args.seq_len * H * D * 4 \
            + 2 * H * D * D * 4
    elif args.case == "prefill_f32":
        d = wl.prefill(t=args.seq_len)
        q, k, v, g, beta = (d[n].float().to(dev) for n in ("q", "k", "v", "g", "beta"))
        S = d["state"].to(dev)
        o = torch.empty((args.seq_len, H, D), device=dev)
        ws = torch.empty(K.kda_prefill_workspace_size(args.seq_len, 1, CHUNK, H, torch.float32),
                         dtype=torch.uint8, device=dev)
        fn = lambda: K.kda_prefill(S, q, k, v, g, beta, o, args.seq_len, CHUNK, workspace=ws)
        nbytes = 5 * args.seq_len * H * D * 4 + args.seq_len * H * 4 + 2 * H * D * D * 4
    elif args.case == "prefill_o_norm":
        d = wl.prefill(t=args.seq_len)
        q, k, v, g, beta = (d[n].to(dev) for n in ("q", "k", "v", "g", "beta"))
        S = d["state"].to(dev)
        ngen = torch.Generator(device="cpu").manual_seed(3)
        n_gate = torch.randn((args.seq_len, H * D), generator=ngen).to(torch.bfloat16).to(dev)
        n_w = torch.ones(D, dtype=torch.bfloat16, device=dev)
        n_out = torch.empty((args.seq_len, H * D), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(K.kda_prefill_workspace_size(args.seq_len, 1, CHUNK, H),
                         dtype=torch.uint8, device=dev)
        fn = lambda: K.kda_prefill_o_norm(S, q, k, v, g, beta, n_gate, n_w, n_out, args.seq_len,
                                          CHUNK, workspace=ws)
        nbytes = 4 * args.seq_len * H * D * 2 + args.seq_len * H * 2 + 2 * args.seq_len * H * D * 2 \
            + 2 * H * D * D * 4 + D * 2
    elif args.case == "prefill_gated":
        d = wl.prefill_gated(t=args.seq_len)
        q, k, v = (d[n].to(dev) for n in ("q", "k", "v"))
        gin = {n: d[n].to(dev) for n in ("g_raw", "dt_bias", "a_log", "b_raw")}
        S = d["state"].to(dev)
        o = torch.empty((args.seq_len, H, D), device=dev)
        ws = torch.empty(K.kda_prefill_workspace_size(args.seq_len, 1, CHUNK, H),
                         dtype=torch.uint8, device=dev)
        fn = lambda: K.kda_prefill_gated(S, q, k, v, gin["g_raw"], gin["dt_bias"], gin["a_log"],
                                         gin["b_raw"], o, args.seq_len, d["gate_lower_bound"],
                                         workspace=ws)
        nbytes = 4 * args.seq_len * H * D * 2 + args.seq_len * H * 2 + args.seq_len * H * D * 4 \
            + 2 * H * D * D * 4 + H * D * 4 + H * 4
    elif args.case == "gate":
        ggen = torch.Generator(device="cpu").manual_seed(0)
        sets = [(torch.randn((args.seq_len, H * D), generator=ggen).to(torch.bfloat16).to(dev),
                 torch.randn((args.seq_len, H), generator=ggen).to(torch.bfloat16).to(dev),
                 torch.empty((args.seq_len, H, D), dtype=torch.bfloat16, device=dev),
                 torch.empty((args.seq_len, H), dtype=torch.bfloat16, device=dev))
                for _ in range(2)]  # alternated, so no launch finds its inputs in L2
        g_dt = (torch.randn(H * D, generator=ggen) * 0.5).to(dev)
        g_al = (torch.randn(H, generator=ggen) * 0.5).to(dev)
        turn = [0]

        def fn():
            g_raw, g_b, g_out, g_beta = sets[turn[0]]
            turn[0] ^= 1
            K.kda_gate(g_raw, g_dt, g_al, g_b, g_out, g_beta, -5.0)
        nbytes = args.seq_len * H * (D * 4 + 4) + H * D * 4 + H * 4
    elif args.case == "decode":
        # two state sets alternated, as in the full run (256 MiB, beyond L2)
        dd = wl.decode_steps(steps=1)
        S_sets = [dd["state"].to(dev), dd["state"].to(dev)]
        ins = [dd[n][0].to(dev) for n in ("q", "k", "v", "g", "beta")]
        o = torch.empty((DECODE_N, H, D), device=dev)
        turn = [0]

        def fn():
            K.kda_decode(S_sets[turn[0]], *ins, o)
            turn[0] ^= 1
        nbytes = DECODE_BYTES
    elif args.case == "conv":
        fe = wl.frontend(lengths=[args.seq_len])
        cu = fe["cu_seqlens"].to(dev)
        x = fe["x"].to(dev)
        wconv = fe["w"].to(dev)
        cst = fe["conv_state"].to(dev)
        xo = torch.empty_like(x)
        fn = lambda: K.kda_conv_silu_l2(cst, x, wconv, xo, cu_seqlens=cu)
        nbytes = args.seq_len * 3 * H * D * 2 * 2 + 3 * H * D * CONV_K * 2 + 2 * 3 * H * D * CONV_K * 4
    else:
        kd = wl.decode_k()
        S = kd["state"].to(dev)
        ins = [kd[n].to(dev) for n in ("q", "k", "v", "g", "beta")]
        o = torch.empty((DK_N, DK_K, H, D), device=dev)
        snaps = [torch.empty_like(S) for _ in range(DK_K)]
        fn = lambda: K.kda_decode_k(S, *ins, o, snaps)
        nbytes = DK_BYTES
    for _ in range(args.warmup):
        fn()
    per, _ = time_launches(fn, args.steps, stream)
    K.kda_sync_status()
    us = statistics.mean(per) * 1e3
    print(json.dumps({"case": args.case, "seq_len": args.seq_len, "launches": args.steps,
                      "avg_launch_us": us, "algorithmic_bytes": nbytes,
                      "GBps": nbytes / us / 1e3}))


def spawn_replicas(n: int) -> int:
    """`python bench.py --gpus N` without a launcher: re-runs this command as N
    ranks (one process per GPU) under torch.distributed.run, as the multi-GPU
    launch does, and returns its exit code."""
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           "--nproc-per-node", str(n), "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__)] + sys.argv[1:]
    return subprocess.call(cmd)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    choices=["prefill", "prefill_f32", "prefill_gated", "prefill_o_norm",
                             "decode", "decode_k", "conv", "gate"],
                    help="time one kernel alone (for profiler captures)")
    ap.add_argument("--seq-len", type=int, default=T_PREFILL)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    _, world, _ = dist_env()
    if args.gpus != world and not args.case:
        if "RANK" in os.environ or args.gpus < 1:
            ap.error("--gpus %d does not match WORLD_SIZE=%d" % (args.gpus, world))
        sys.exit(spawn_replicas(args.gpus))
    if args.case:
        run_case(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
