#!/usr/bin/env python3
"""Benchmark of the fused draft-block select-and-verify step (DFlash 2) on GB300.

One step = one dfs_select_verify call over one batch of the throughput workload
(B=32 requests, block L=8, V=151936, d=5120, r=256, bf16, Zipf-shaped drafter rows):
LM head + top-16, gate, pair scores, path, verification. Metric: draft blocks/s (one block
= one request's L-position block), plus the fraction of the HBM roofline set by the bytes
of W_vocab and the target logits.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 it runs under torch.distributed.run, one process per GPU; every rank is an
independent replica with its own batch (weak scaling), rank 0 prints one JSON line.
--impl reference times the fp64 CPU oracle on this host's cores on a bounded sample of
the same workload.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
sys.path.insert(1, os.path.join(ROOT, "tests"))  # the planted-target checks of the loop leg

METRIC = "draft blocks/s for select+verify at B=32,L=8,V=151936; % of HBM roofline"
UNIT = "blocks/s"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    # defaults: our arm times 2000 steps (about 0.6 s at the bench workload, long enough for
    # the clock samples to see the kernels under load); the oracle arm 50 one-request steps
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="throughput_B32_L8_V151936_d5120_zipf")
    ap.add_argument("--path-mode", choices=["greedy", "viterbi"], default="greedy")
    ap.add_argument("--sampling-temperature", type=float, default=0.6)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU time budget of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def lmhead_source_hash() -> str:
    h = hashlib.sha256()
    for name in ("lmhead_tc.cu", "common.cuh", "rowstat.cuh"):
        with open(os.path.join(ROOT, "draft_speculative_decoding_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per LM-head launch from the committed ncu summary, if it was taken on
    the kernel source as it is now."""
    p = os.path.join(ROOT, "profiles", "lmhead_ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("source_hash") != lmhead_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons every 50 ms; the summary keeps only the
    samples whose own timestamp falls inside the marked (timed) window."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_uuid: str | None):
        self.rows = []
        self.proc = None
        self.thread = None
        self.window = [None, None]
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if gpu_uuid:
            cmd += ["-i", gpu_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def mark_start(self):
        self.window[0] = datetime.datetime.now()

    def mark_end(self):
        self.window[1] = datetime.datetime.now()

    @staticmethod
    def _when(ts: str):
        try:
            return datetime.datetime.strptime(ts, "%Y/%m/%d %H:%M:%S.%f")
        except ValueError:
            return None

    def in_window(self, t0, t1):
        return [r for r in list(self.rows) if (w := self._when(r[0])) is not None and t0 <= w <= t1]

    def stop(self, t0=None, t1=None):
        """Stops sampling; summarises the samples taken between t0 and t1 (default: the
        marked window)."""
        if self.proc is None:
            return None
        time.sleep(0.15)  # let the sample that covers the window's end arrive
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        t0 = self.window[0] if t0 is None else t0
        t1 = self.window[1] if t1 is None else t1
        rows = self.rows
        if t0 is not None and t1 is not None:
            rows = self.in_window(t0, t1)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_median": statistics.median(pw) if pw else None,
                "samples": len(rows)}


# ------------------------------------------------------------------- our implementation
def run_ours(args):
    import numpy as np
    import torch

    from draft_speculative_decoding_gb300 import binding, replicas
    from draft_speculative_decoding_gb300 import build as dfs_build
    from draft_speculative_decoding_gb300 import workloads as wl

    rank, world, local = replicas.init()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        dfs_build.build()
    replicas.barrier()
    binding.load()

    spec = wl.WORKLOADS[args.workload]
    data = wl.generate(spec.with_(seed=spec.seed + 1000 * rank), dev)
    nrot = 3  # rotate target-logit / hidden buffers so no step rereads an L2-resident copy
    Zs = [data["Z"]] + [wl.fresh_targets(data, 100 + i) for i in range(1, nrot)]
    hs = [data["h"]] + [data["h"].clone() for _ in range(1, nrot)]
    dims = binding.make_dims(spec.B, spec.L, spec.V, spec.d, spec.r, binding.DFS_BF16,
                             binding.DFS_BF16)
    ws = binding.alloc_workspace(dims)
    P = spec.L - 1
    outs = (torch.empty(spec.B, P, dtype=torch.int32, device=dev),
            torch.empty(spec.B, spec.L, dtype=torch.int32, device=dev),
            torch.empty(spec.B, dtype=torch.int32, device=dev))
    mode = binding.DFS_PATH_GREEDY if args.path_mode == "greedy" else binding.DFS_PATH_VITERBI
    stream = torch.cuda.current_stream()

    def step(i, T, h=None, Z=None, x0=None, path_mode=None):
        binding.dfs_select_verify(dims, hs[i % nrot] if h is None else h, data["W"], data["Wg"],
                                  data["A"], data["Bt"], data["x0"] if x0 is None else x0,
                                  Zs[i % nrot] if Z is None else Z,
                                  mode if path_mode is None else path_mode, T, spec.seed + i, ws,
                                  outputs=outs, stream=stream)

    def timed(T, K, W, trace=False, clocks=None, path_mode=None):
        for i in range(W):
            step(i, T, path_mode=path_mode)
        torch.cuda.synchronize()
        replicas.barrier()
        torch.cuda.synchronize()
        tr = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)] if trace else None
        for ev in (tr or []):
            ev[0].record(stream)
            ev[1].record(stream)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        n0 = binding.dfs_launch_count()
        if clocks is not None:
            clocks.mark_start()
        e0.record(stream)
        for i in range(K):
            if trace:
                binding.dfs_set_trace_events(*tr[i])
            step(W + i, T, path_mode=path_mode)
        e1.record(stream)
        n1 = binding.dfs_launch_count()
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.mark_end()
        binding.dfs_set_trace_events(None, None)
        replicas.barrier()
        ms = e0.elapsed_time(e1) / K
        lm = [a.elapsed_time(b) for a, b in tr] if trace else None
        return ms, lm, n1 - n0

    def per_call(T, K, W, path_mode=None):
        """Per-call durations: events around each call. The event between two calls stops
        the second launching early (no programmatic overlap), so each call pays its own
        launch; used for the spread, not the headline."""
        for i in range(W):
            step(i, T, path_mode=path_mode)
        torch.cuda.synchronize()
        replicas.barrier()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for i in range(K):
            evs[i][0].record(stream)
            step(W + i, T, path_mode=path_mode)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        replicas.barrier()
        return [a.elapsed_time(b) for a, b in evs]

    def spread(xs):
        q = sorted(xs)

        def pct(f):  # nearest rank
            return q[min(len(q) - 1, max(0, math.ceil(f * len(q)) - 1))]
        return {"median_ms": round(statistics.median(q), 4), "p10_ms": round(pct(0.1), 4),
                "p90_ms": round(pct(0.9), 4), "n": len(q)}

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        uuid = None
    clocks = ClockSampler(uuid)
    ms_greedy, _, launches = timed(0.0, args.steps, args.warmup, clocks=clocks)
    # The sampler reports every 50 ms. When the timed region held fewer than 10 samples, the
    # same greedy steps keep running, untimed, for 0.6 s right after it, and the clock record
    # comes from those samples (said so in the record).
    t_win = clocks.window[:]
    clk_note = "samples taken inside the timed region"
    if clocks.proc is not None and len(clocks.in_window(*t_win)) < 10:
        t_probe0 = datetime.datetime.now()
        i = 0
        while (datetime.datetime.now() - t_probe0).total_seconds() < 0.6:
            for _ in range(20):
                step(args.warmup + args.steps + i, 0.0)
                i += 1
            torch.cuda.synchronize()
        t_win = [t_probe0, datetime.datetime.now()]
        clk_note = (f"the timed region ({ms_greedy * args.steps:.1f} ms) is shorter than 10 "
                    f"sampler periods: samples taken over {i} more of the same greedy steps "
                    f"run untimed right after it")
    clk = clocks.stop(*t_win)
    if clk is not None:
        clk["window"] = clk_note
        if clk.get("sm_mhz"):
            clk["sm_kcycles_per_step"] = round(ms_greedy * clk["sm_mhz"], 1)
    # the dominant kernel's own duration, from events recorded around it on its stream (a
    # separate pass: an event between two kernels stops the second launching early)
    _, lm_list, _ = timed(0.0, args.steps, 1, trace=True)
    lm_ms = statistics.mean(lm_list)
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    accept = outs[2].float().mean().item()
    ms_samp, _, _ = timed(args.sampling_temperature, max(10, args.steps // 2), args.warmup)
    accept_samp = outs[2].float().mean().item()
    # the sampled traversal (each successor drawn from the scores) verified against its own
    # proposal
    ms_prop, _, _ = timed(args.sampling_temperature, max(10, args.steps // 2), args.warmup,
                          path_mode=binding.DFS_PATH_SAMPLE)
    accept_prop = outs[2].float().mean().item()
    # the joint path draw (the whole path from the distribution the scores define over the
    # lattice) verified against its own conditionals
    ms_joint, _, _ = timed(args.sampling_temperature, max(10, args.steps // 2), args.warmup,
                           path_mode=binding.DFS_PATH_SAMPLE_JOINT)
    accept_joint = outs[2].float().mean().item()
    # the other path mode at both temperatures (the headline's is the greedy traversal)
    other = binding.DFS_PATH_GREEDY if mode == binding.DFS_PATH_VITERBI else binding.DFS_PATH_VITERBI
    ms_other0, _, _ = timed(0.0, max(10, args.steps // 2), args.warmup, path_mode=other)
    ms_other_s, _, _ = timed(args.sampling_temperature, max(10, args.steps // 2), args.warmup,
                             path_mode=other)
    # the spread of single calls (greedy headline mode, T = 0)
    call_ms = per_call(0.0, max(20, args.steps // 4), args.warmup)

    # the same step with the LM head given quantised to E4M3 (one power-of-two scale per
    # vocabulary entry; rows quantised per call): half the LM-head bytes
    Wq, w_scale = wl.quantize_lmhead_e4m3(data["W"])
    Wq = binding.dfs_pack_e4m3_head(Wq)  # the head packed once, as a loader would

    def step_q(i):
        binding.dfs_select_verify_e4m3(dims, hs[i % nrot], Wq, w_scale, data["Wg"], data["A"],
                                       data["Bt"], data["x0"], Zs[i % nrot], mode, 0.0,
                                       spec.seed + i, ws, outputs=outs, stream=stream)

    for i in range(args.warmup):
        step_q(i)
    torch.cuda.synchronize()
    replicas.barrier()
    K_q = max(10, args.steps // 2)
    q0, q1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    q0.record(stream)
    for i in range(K_q):
        step_q(args.warmup + i)
    q1.record(stream)
    torch.cuda.synchronize()
    ms_q = q0.elapsed_time(q1) / K_q
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    del Wq, w_scale

    # the greedy step replayed from a CUDA graph (how a decode loop would issue it): 30 steps
    # over the rotating buffers recorded once, the recording replayed for the timed steps
    n_rec = 30
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(n_rec):
            step(i, 0.0)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = torch.cuda.current_stream()
        for i in range(n_rec):
            binding.dfs_select_verify(dims, hs[i % nrot], data["W"], data["Wg"], data["A"],
                                      data["Bt"], data["x0"], Zs[i % nrot], mode, 0.0,
                                      spec.seed + i, ws, outputs=outs, stream=cap)
    for _ in range(max(1, args.warmup // n_rec + 1)):
        graph.replay()
    torch.cuda.synchronize()
    replicas.barrier()
    n_rep = max(1, args.steps // n_rec)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(n_rep):
        graph.replay()
    g1.record(stream)
    torch.cuda.synchronize()
    ms_graph = g0.elapsed_time(g1) / (n_rep * n_rec)
    assert binding.dfs_get_device_error(ws) == binding.DFS_OK

    # the drafter-side two-tap convolution (dfs_conv2tap) at the workload's block shape: 16
    # rotating input sets (x and W_c: 147 MB, more than L2), 48 calls recorded into a CUDA
    # graph and replayed (the per-call host work is not the kernels' time); eager calls too
    cspec = wl.ConvSpec(f"conv_B{spec.B}_L{spec.L}_d{spec.d}", B=spec.B, L=spec.L, d=spec.d,
                        seed=spec.seed + 5)
    n_cset = 16
    csets = [wl.conv_inputs(cspec.with_(seed=cspec.seed + k), dev) for k in range(n_cset)]
    cws = binding.alloc_conv_workspace(cspec.B, cspec.L, cspec.d)
    cout = torch.empty_like(csets[0]["x"])

    def cstep(k, st):
        c = csets[k % n_cset]
        binding.dfs_conv2tap(c["x"], c["base"], c["Wc"], cws, out=cout, stream=st)

    for k in range(max(3, args.warmup)):
        cstep(k, stream)
    torch.cuda.synchronize()
    K_c = 200
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for k in range(K_c):
        cstep(k, stream)
    c1.record(stream)
    torch.cuda.synchronize()
    us_conv_eager = c0.elapsed_time(c1) / K_c * 1e3
    n_crec = 48
    with torch.cuda.stream(side):
        for k in range(n_crec):
            cstep(k, side)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    cgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(cgraph):
        cap = torch.cuda.current_stream()
        for k in range(n_crec):
            cstep(k, cap)
    cgraph.replay()
    torch.cuda.synchronize()
    n_crep = 10
    c0.record(stream)
    for _ in range(n_crep):
        cgraph.replay()
    c1.record(stream)
    torch.cuda.synchronize()
    us_conv = c0.elapsed_time(c1) / (n_crep * n_crec) * 1e3
    assert binding.dfs_get_device_error(cws) == binding.DFS_OK
    conv_rows = cspec.B * cspec.L
    conv_bytes = 4 * conv_rows * cspec.d + 2 * (cspec.d // 8) * cspec.d + 8 * cspec.d
    conv_flops = 2.0 * conv_rows * cspec.d * (cspec.d // 8)
    del csets, cgraph

    # multi-cycle decode loops (cycles.py). Fused: per cycle the fused step and the last-token
    # hand-off (dfs_next_tokens), the last verified tokens carried on the device, 30 cycles
    # recorded into one CUDA graph, for B = 1, 8 and the workload's B (its first requests).
    # Planted: at the workload's B, staged greedy cycles against targets whose argmax agrees
    # with each drafted token with the page's Table 1 Recall@1 rates (closed form 4.27).
    import planted
    from draft_speculative_decoding_gb300 import cycles as cyc_mod
    cyc_legs = {}
    n_cyc = 30
    for Bc in sorted({1, 8, spec.B}):
        if Bc > spec.B:
            continue
        dims_c = binding.make_dims(Bc, spec.L, spec.V, spec.d, spec.r, binding.DFS_BF16,
                                   binding.DFS_BF16)
        ws_c = binding.alloc_workspace(dims_c)
        hs_c, Zs_c = [h[:Bc] for h in hs], [Z[:Bc] for Z in Zs]
        x0c = data["x0"][:Bc].clone()
        P_ = spec.L - 1
        outs_c = (torch.empty(Bc, P_, dtype=torch.int32, device=dev),
                  torch.empty(Bc, spec.L, dtype=torch.int32, device=dev),
                  torch.empty(Bc, dtype=torch.int32, device=dev))
        side.wait_stream(stream)
        with torch.cuda.stream(side):  # warm-up, and the accept lengths of one eager pass
            _, accs = cyc_mod.fused_cycles(dims_c, data, hs_c, Zs_c, x0c, ws_c, mode, n_cyc,
                                           stream=side)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        mean_acc_c = torch.stack(accs).float().mean().item()
        g_c = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_c):
            cyc_mod.fused_cycles(dims_c, data, hs_c, Zs_c, x0c, ws_c, mode, n_cyc,
                                 outputs=outs_c, stream=torch.cuda.current_stream())
        g_c.replay()
        torch.cuda.synchronize()
        n_rep_c = 3
        c0.record(stream)
        for _ in range(n_rep_c):
            g_c.replay()
        c1.record(stream)
        torch.cuda.synchronize()
        ms_cyc = c0.elapsed_time(c1) / (n_rep_c * n_cyc)
        assert binding.dfs_get_device_error(ws_c) == binding.DFS_OK
        cyc_legs[f"B{Bc}"] = {"ms_per_cycle": round(ms_cyc, 4),
                              "cycles_per_s": round(1e3 / ms_cyc, 1),
                              "blocks_per_s": round(Bc * 1e3 / ms_cyc, 1),
                              "accepted_tokens_per_s": round(mean_acc_c * Bc * 1e3 / ms_cyc, 1),
                              "mean_accept_len": round(mean_acc_c, 3)}
        del g_c, ws_c
    if spec.L - 1 == len(planted.TABLE1_RECALL_AT_1):
        gen_p = torch.Generator(device=dev).manual_seed(spec.seed + 7)
        x0p = data["x0"].clone()
        runs = planted.planted_cycles(dims, data, hs, Zs[0], x0p, ws, planted.TABLE1_RECALL_AT_1,
                                      40, gen_p)
        torch.cuda.synchronize()
        acc_p = torch.stack([a for a, _ in runs]).float()
        exact_p = all(torch.equal(a.long(), planted.leading_agreements(g)) for a, g in runs)
        planted = {"cycles": 40, "requests": spec.B,
                   "mean_accept_len": round(acc_p.mean().item(), 3),
                   "std_error": round(acc_p.std().item() / math.sqrt(acc_p.numel()), 3),
                   "closed_form": round(planted.closed_form_accept_len(planted.TABLE1_RECALL_AT_1), 3),
                   "every_accept_len_as_planted": exact_p}
        assert binding.dfs_get_device_error(ws) == binding.DFS_OK
    else:  # the Recall@1 rates are given for blocks of 8 only
        planted = {"skipped": f"Table 1 rates cover 7 drafted positions, this workload has {spec.L - 1}"}

    # end to end through the public API: every step copies its inputs (h, Z, x0) from pinned
    # host memory and reads its results back to pinned host memory. As a serving loop would,
    # step i+1's inputs are copied while step i runs: two device input sets, two copy streams
    # (the target logits split by request halves over them), events for the hand-offs.
    host_h = [h.cpu().pin_memory() for h in hs]
    host_Z = [Z.cpu().pin_memory() for Z in Zs]
    host_x0 = data["x0"].cpu().pin_memory()
    nbuf = 2
    dev_in = [(torch.empty_like(hs[0]), torch.empty_like(Zs[0]), torch.empty_like(data["x0"]))
              for _ in range(nbuf)]
    host_res = [(torch.empty(outs[1].shape, dtype=torch.int32).pin_memory(),
                 torch.empty(outs[2].shape, dtype=torch.int32).pin_memory()) for _ in range(nbuf)]
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(2)]
    copied = [[torch.cuda.Event() for _ in copy_streams] for _ in range(nbuf)]
    freed = [torch.cuda.Event() for _ in range(nbuf)]  # the step using a set has read it
    B2 = spec.B // 2
    # at least 50 steps: the first step's copies cannot overlap a previous step (no copy of
    # the timed steps starts before the timed region), and over a handful of steps that one
    # exposed copy would stand for the leg's steady state
    K_e2e = max(50, args.steps // 2)

    def issue_copies(i):
        k = i % nbuf
        dh, dZ, dx = dev_in[k]
        hZ = host_Z[i % nrot]
        for c, cs in enumerate(copy_streams):
            cs.wait_event(freed[k])
            with torch.cuda.stream(cs):
                if c == 0:
                    dh.copy_(host_h[i % nrot], non_blocking=True)
                    dx.copy_(host_x0, non_blocking=True)
                    dZ[:B2].copy_(hZ[:B2], non_blocking=True)
                else:
                    dZ[B2:].copy_(hZ[B2:], non_blocking=True)
            copied[k][c].record(cs)

    def compute(i):
        k = i % nbuf
        for ev in copied[k]:
            stream.wait_event(ev)
        step(i, 0.0, *dev_in[k])
        freed[k].record(stream)
        ho, ha = host_res[k]
        ho.copy_(outs[1], non_blocking=True)
        ha.copy_(outs[2], non_blocking=True)

    def e2e_run(n, start):
        issue_copies(start)
        for i in range(n):
            if i + 1 < n:
                issue_copies(start + i + 1)
            compute(start + i)

    e2e_run(max(3, args.warmup), 0)
    torch.cuda.synchronize()
    replicas.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for cs in copy_streams:
        cs.wait_event(e0)  # no copy of the timed steps starts before the timed region
    e2e_run(K_e2e, 0)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = e0.elapsed_time(e1) / K_e2e
    h2d = hs[0].numel() * 2 + Zs[0].numel() * 2 + data["x0"].numel() * 4
    d2h = outs[1].numel() * 4 + outs[2].numel() * 4

    value = replicas.job_throughput(spec.B * args.steps, ms_greedy * args.steps / 1e3)
    ms_max = replicas.max_over_ranks(ms_greedy)
    value_samp = replicas.job_throughput(spec.B, ms_samp / 1e3)
    value_prop = replicas.job_throughput(spec.B, ms_prop / 1e3)
    value_joint = replicas.job_throughput(spec.B, ms_joint / 1e3)
    value_other0 = replicas.job_throughput(spec.B, ms_other0 / 1e3)
    value_other_s = replicas.job_throughput(spec.B, ms_other_s / 1e3)
    value_graph = replicas.job_throughput(spec.B, ms_graph / 1e3)
    value_q = replicas.job_throughput(spec.B, ms_q / 1e3)
    q_bytes = spec.d * spec.V + spec.B * spec.L * spec.V * 2  # E4M3 head + target logits
    value_e2e = replicas.job_throughput(spec.B, ms_e2e / 1e3)
    lm_max = replicas.max_over_ranks(lm_ms)

    peaks, peak_src = measured_peaks()
    # algorithmic bytes of one call, all read by the LM-head kernel: the vocabulary
    # projection once and the target logits once (their row statistics are folded into the
    # same kernel); hidden rows, gate projection and outputs (< 0.5 %) are not counted.
    # Algorithmic flops: the B*(L-1) draft rows against the vocabulary and gate projections.
    w_bytes = spec.d * spec.V * 2
    z_bytes = spec.B * spec.L * spec.V * 2
    lm_bytes = w_bytes + z_bytes
    lm_flops = 2.0 * spec.B * (spec.L - 1) * spec.d * (spec.V + spec.r)
    achieved = lm_bytes / (lm_max * 1e-3) / 1e9
    tflops = lm_flops / (lm_max * 1e-3) / 1e12
    step_achieved = lm_bytes / (ms_max * 1e-3) / 1e9
    traffic = ncu_traffic(args.workload)
    # the library's choice for this shape: more than 128 rows take the CTA-pair kernels, the
    # vocabulary-major one where its groups of up to 2 nb requests need fewer passes over W
    rows = spec.B * spec.L
    nb = 8 * (16 // (spec.L - 1)) if spec.L - 1 <= 16 else 0
    vt = rows > 128 and nb > 0 and -(-spec.B // (2 * nb)) < -(-rows // 256)
    lm_kernel = ("k_lmhead_vt" if vt else "k_lmhead_pair" if rows > 128 else "k_lmhead_tc") + \
        " (LM head + top-16 + gate tiles + target-row statistics)"

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gpu_ref = {}
        for T in (0.0, args.sampling_temperature):  # the inputs the oracle's leg reads
            res = binding.dfs_select_verify(dims, data["h"], data["W"], data["Wg"], data["A"],
                                            data["Bt"], data["x0"], data["Z"], mode, T, spec.seed,
                                            ws, want_intermediates=True, stream=stream)
            torch.cuda.synchronize()
            gpu_ref[T] = {k: v.cpu().numpy() for k, v in res.items()}
        cpu, parity = cpu_baseline(data, spec, args.cpu_seconds, mode,
                                   args.sampling_temperature, gpu_ref)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; shapes and distributions of the pages' block-8 workload)",
            "config": {"workload": spec.name, "B": spec.B, "L": spec.L, "K": 16, "V": spec.V,
                       "d": spec.d, "r": spec.r, "path_mode": args.path_mode,
                       "temperature": 0.0, "parallelism": f"replicas x{world}",
                       "l2": f"inputs larger than L2: W_vocab {w_bytes / 1e9:.2f} GB read "
                             f"every step"},
            "l2_rotation": f"{nrot} rotating target-logit and hidden buffers",
            "hbm_roofline_frac_step": round(step_achieved / peaks["hbm_gbs"], 4),
            "roofline": {"kernel": lm_kernel,
                         "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": traffic, "algorithmic_bytes_per_launch": lm_bytes,
                         "ms_per_launch": round(lm_max, 4),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                         "tensor": {"achieved": round(tflops, 1), "unit": "TFLOP/s",
                                    "peak": peaks["bf16_tflops"],
                                    "frac": round(tflops / peaks["bf16_tflops"], 4),
                                    "flops_per_launch": lm_flops}},
            "e2e": {"value": round(value_e2e, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_e2e, 4),
                    "overlap": "step i+1's inputs copied on two copy streams during step i"},
            "sampling": {"temperature": args.sampling_temperature, "value": round(value_samp, 1),
                         "unit": UNIT, "ms_per_step": round(ms_samp, 4),
                         "mean_accept_len": round(accept_samp, 3),
                         "path": args.path_mode,
                         "sampled_path": {"value": round(value_prop, 1), "unit": UNIT,
                                          "ms_per_step": round(ms_prop, 4),
                                          "mean_accept_len": round(accept_prop, 3)},
                         "joint_path": {"value": round(value_joint, 1), "unit": UNIT,
                                        "ms_per_step": round(ms_joint, 4),
                                        "mean_accept_len": round(accept_joint, 3)}},
            "other_path_mode": {
                "path": "greedy" if other == binding.DFS_PATH_GREEDY else "viterbi",
                "T0": {"value": round(value_other0, 1), "unit": UNIT,
                       "ms_per_step": round(ms_other0, 4)},
                f"T{args.sampling_temperature:g}": {"value": round(value_other_s, 1),
                                                    "unit": UNIT,
                                                    "ms_per_step": round(ms_other_s, 4)}},
            "spread": {
                "per_call": {**spread(call_ms),
                             "note": "events around each greedy T=0 call: no programmatic "
                                     "overlap with the previous call, so each pays its launch"},
                "lmhead_per_launch": spread(lm_list)},
            "e4m3_head": {"value": round(value_q, 1), "unit": UNIT,
                          "ms_per_step": round(ms_q, 4),
                          "hbm_roofline_frac_step": round(q_bytes / (ms_q * 1e-3) / 1e9 /
                                                          peaks["hbm_gbs"], 4),
                          "note": "LM head as E4M3 with per-vocabulary scales "
                                  "(dfs_select_verify_e4m3); not the headline's precision"},
            "conv2tap": {"workload": cspec.name, "us_per_call": round(us_conv, 3),
                         "us_per_call_eager": round(us_conv_eager, 3),
                         "roofline": {"bound": "hbm",
                                      "achieved": round(conv_bytes / (us_conv * 1e-6) / 1e9, 1),
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": round(conv_bytes / (us_conv * 1e-6) / 1e9 /
                                                    peaks["hbm_gbs"], 4),
                                      "algorithmic_bytes_per_call": conv_bytes},
                         "tensor_tflops": round(conv_flops / (us_conv * 1e-6) / 1e12, 1),
                         "note": "drafter-side two-tap dynamic depthwise convolution "
                                 "(dfs_conv2tap: correction GEMM + apply, two kernels), "
                                 "48 calls per CUDA graph over 16 rotating input sets"},
            "cycles": {"fused_graph": cyc_legs, "planted_table1": planted,
                       "note": "multi-cycle decode loops: fused step + last-token hand-off per "
                               "cycle, 30 cycles per CUDA graph (B = 1, 8, 32: the workload's "
                               "first requests); planted: staged greedy cycles against targets "
                               "agreeing with each drafted token at the page's Table 1 Recall@1 "
                               "rates"},
            "graph": {"value": round(value_graph, 1), "unit": UNIT,
                      "ms_per_step": round(ms_graph, 4),
                      "note": "greedy steps replayed from a CUDA graph of 30 recorded steps"},
            "mean_accept_len": round(accept, 3),
            "gpu_launches": launches,
            "clocks": clk,
            "cpu_baseline": cpu,
            "parity": parity,
        }
        print(json.dumps(line), flush=True)
    replicas.finalize()


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.lower().startswith(key.lower()) and ":" in line:
                    return f"{key}: {line.split(':', 1)[1].strip()}"
    except OSError:
        pass
    import platform
    return platform.machine()


def cpu_baseline(data, spec, budget_s, path_mode, T_samp, gpu_ref):
    """The fp64 oracle as it stands, on this host's cores: requests of the same batch, one
    call each, until the time budget is spent (at least one request), greedy (T = 0) and
    sampling (T_samp), all cores; and one request on one core. The oracle's outputs of the
    greedy and sampling runs are then compared with the GPU's outputs for the same inputs
    and seeds (gpu_ref), request by request, with the near-tie exclusions counted per rule."""
    import numpy as np

    import oracle
    import parity as par
    from draft_speculative_decoding_gb300 import workloads as wl

    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    threads = oracle.default_threads()
    oracle.build()

    def run(T, nthreads, budget, max_req):
        outs, n, t0 = [], 0, time.perf_counter()
        while n < max_req and (n == 0 or time.perf_counter() - t0 < budget):
            outs.append(oracle.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"],
                                             npd["x0"], npd["Z"], path_mode=path_mode,
                                             temperature=T, seed=spec.seed, reqs=[n],
                                             nthreads=nthreads))
            n += 1
        return n, time.perf_counter() - t0, outs

    n_g, dt_g, outs_g = run(0.0, threads, budget_s, spec.B)
    n_s, dt_s, outs_s = run(T_samp, threads, budget_s, spec.B)
    n_1, dt_1, _ = run(0.0, 1, 0.0, 1)
    checks = {}
    for T, outs in ((0.0, outs_g), (T_samp, outs_s)):
        o = {k: np.concatenate([x[k] for x in outs]) for k in outs[0] if k != "reqs"}
        tally = par.new_tally()
        tally["mismatch"] = 0
        for q in range(len(outs)):
            try:
                par.compare_request(gpu_ref[T], o, q, q, spec, T, tally)
            except AssertionError:
                tally["mismatch"] += 1
        checks["greedy" if T == 0 else f"sampling_T{T}"] = tally
    mode = {0: "greedy", 1: "viterbi"}[path_mode]
    base = {"value": round(n_g / dt_g, 4), "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{n_g} of {spec.B} requests of {spec.name}, {mode} path, T=0, "
                      f"{dt_g:.1f} s wall",
            "single_core": {"value": round(n_1 / dt_1, 4), "unit": UNIT, "cores": 1,
                            "sample": f"1 request, {mode} path, T=0, {dt_1:.1f} s wall"},
            "sampling": {"temperature": T_samp, "value": round(n_s / dt_s, 4), "unit": UNIT,
                         "cores": threads,
                         "sample": f"{n_s} of {spec.B} requests, {mode} path, T={T_samp}, "
                                   f"{dt_s:.1f} s wall"}}
    return base, {"workload": spec.name, "compared": "GPU vs oracle on the requests the "
                  "oracle ran above (same inputs and seeds)", **checks}


# ------------------------------------------------------------------- reference arm (oracle)
def run_reference(args):
    from draft_speculative_decoding_gb300 import replicas

    rank, world, _ = replicas.rank_info()
    if rank != 0:
        return
    import torch

    import oracle
    from draft_speculative_decoding_gb300 import workloads as wl

    spec = wl.WORKLOADS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    data = wl.generate(spec, dev)
    npd = {k: wl.to_numpy_bits(data[k]) for k in ("h", "W", "Wg", "A", "Bt", "x0", "Z")}
    del data
    oracle.build()
    threads = oracle.default_threads()

    def step(i):  # one request of the batch per step: a bounded sample
        oracle.select_verify(npd["h"], npd["W"], npd["Wg"], npd["A"], npd["Bt"], npd["x0"],
                             npd["Z"], path_mode=0, temperature=0.0, seed=spec.seed,
                             reqs=[i % spec.B], nthreads=threads)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    sample = f"1 of {spec.B} requests of {spec.name} per step (greedy path, T=0)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "L": spec.L, "K": 16, "V": spec.V,
                   "d": spec.d, "r": spec.r, "path_mode": "greedy", "temperature": 0.0,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: W_vocab {spec.d * spec.V * 2 / 1e9:.2f} GB "
                         f"read every step"},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    if args.steps is None:
        args.steps = 50 if args.impl == "reference" else 2000
    if args.warmup is None:
        args.warmup = 3 if args.impl == "reference" else 20
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
