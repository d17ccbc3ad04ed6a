#!/usr/bin/env python
"""Benchmark of the KDA gated delta-rule serving path on GB300.

One step is one pass of every phase of the path, each on its own synthetic
workload at 16 heads x 128 (the pages' single-GPU microbenchmark setting,
"[KDA] Support Helion MTP verification and harden prefill, decode", sglang
PR #42857, Speed Tests and Profiling):
  prefill   1 sequence x 4096 tokens, 16-slot FP32 pool      (the headline)
  decode    48 requests x 1 token, 240-slot pool
  verify    16 requests x 6 draft tokens, chain and tree, with snapshots
  commit    16 requests, accepted snapshot copied into the pool
  replay    the same verify keeping a ring of folded token inputs instead of
            snapshots, and its commit replaying the accepted prefix ("[KDA]
            Default GLM-5-Next spec verify to the CuTe DSL KDA kernel #42905",
            Results: ReplaySSM rings)
`value` is prefill tokens/s (the metric's first term) over the prefill phase
time.  Every phase is a CUDA-graph replay timed with CUDA events recorded as
graph nodes around its kernels, after an L2 flush (a 512 MiB write, then a
read of the same buffer).  Decode, verify and commit replay 8 layer calls back
to back, each on its own state pool and buffers, and report the span / 8.
`phases` carries the per-layer-call microseconds of every phase.  `e2e`
repeats the prefill with its inputs copied from pinned host memory and its
output copied back inside the timed region.

Multi-GPU: the path has no exchange step, so N ranks run N independent
replicas (weak scaling); `value` is the tokens of all ranks over the slowest
rank's time.

--impl reference times the FP64 CPU oracle (the slow reference program) on a
bounded sample of the same prefill workload, on this machine's host cores.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

H, K = 16, 128
CHUNK = 64
METRIC = "KDA prefill tok/s @16h×128; decode/verify µs/layer; % HBM/TC roofline"
PREFILL_T = 4096
LONG_T, LONG_CALLS = 32768, 8  # one long sequence, in one call or continued over 8 calls
DECODE_B = 48
VERIFY_B, VERIFY_T = 16, 6
COMMIT_B = VERIFY_B
FLUSH_BYTES = 512 << 20
LAYERS = 8  # default decode/verify/commit calls per timed replay (--layers)

# DRAM traffic per launch from ncu (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by kernel; valid only while the kernel sources hash to the recorded
# value (the figure is re-taken whenever they change; see the transform's ncu
# traffic summary under profiles/).
NCU_TRAFFIC = {
    # the transform launch of one 1x4096 prefill call, 16 heads, mean of two
    # captured launches: read 68.45 MB (its inputs) + write 83.41 MB (the part
    # of its per-chunk records that leaves L2 before the state pass reads it)
    "prefill_transform": {"bytes": 151863552, "src": "b299d1e64a6576be"},
}
VERIFY_SWEEP = (1, 2, 4, 8, 12, 16, 24, 32, 48)  # requests x 6 draft tokens, chain and tree
DECODE_SWEEP = (1, 16)  # besides the core step's 48


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("sm_max_mhz", 2070.0)), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, 2070.0, "fallback"


def _source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_serving_gated_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- #
# algorithmic work per launch (bytes moved at minimum, or flops of the chunk form)

def prefill_bytes(T, nseq=1):
    # q, k, v, gate input a, o (BF16, T x H x 128 each), beta (BF16), state read+write
    return 5 * T * H * K * 2 + T * H * 2 + nseq * 2 * H * K * K * 4


def transform_flops(T):
    # A, P, W, Util (C^2 K each, triangular) and the inverse (C^3 / 3) per chunk-head
    n = (T + CHUNK - 1) // CHUNK * H
    return n * (4 * CHUNK * CHUNK * K + CHUNK ** 3 / 3)


def transform_bytes(T):
    # the chunk transform's inputs: q, k, v, gate input a (BF16, T x H x 128 each) and beta
    return 4 * T * H * K * 2 + T * H * 2


def token_io_bytes():
    # one packed row (q, k, v), gate input, beta, output, all BF16
    return (3 * H * K + H * K + H + H * K) * 2


def decode_bytes(B):
    return B * (2 * H * K * K * 4 + token_io_bytes())


def verify_bytes(B, T):
    return B * (H * K * K * 4 + T * H * K * K * 4 + T * token_io_bytes())


RING_FLOATS = 3 * K + 4  # replay ring record per (request, token, head)


def verify_replay_bytes(B, T):
    # state read once, token rows, ring records written (no snapshots)
    return B * (H * K * K * 4 + T * token_io_bytes() + T * H * RING_FLOATS * 4)


def commit_replay_bytes(accepted, T):
    # per committing request: state read + write, ring records of the replayed prefix
    return sum(2 * H * K * K * 4 + (int(a) + 1) * H * RING_FLOATS * 4 for a in accepted if a >= 0)


def commit_bytes(B):
    return B * 2 * H * K * K * 4


def varlen_prefill_bytes(lengths, heads=H):
    # token tensors (q, k, v, gate input, o) and beta over the real tokens, the
    # gathered and scattered states
    T = int(sum(lengths))
    return 5 * T * heads * K * 2 + T * heads * 2 + len(lengths) * 2 * heads * K * K * 4


# --------------------------------------------------------------------------- #

class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        self.proc = None
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        mhz, max_mhz, reasons = [], 0.0, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                mhz.append(float(f[1]))
                max_mhz = max(max_mhz, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max_mhz,
                "reasons": sorted(reasons), "samples": len(mhz)}


def max_over_ranks(values, world, device="cpu"):
    """Element-wise max of a list of floats over all ranks (identity at world 1)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    vec = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(vec, op=dist.ReduceOp.MAX)
    return [float(x) for x in vec.tolist()]


def replica_throughput(units_per_rank_step, steps, world, slowest_seconds):
    """Whole-job throughput of N independent replicas: every rank's units over
    the slowest rank's time (weak scaling)."""
    return units_per_rank_step * steps * world / slowest_seconds


def physical_gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return local_rank


def run_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from linear_attention_serving_gated_gb300 import build as kbuild
    from linear_attention_serving_gated_gb300 import inputs, kda

    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    if rank == 0:
        kbuild.build()
    if world > 1:
        dist.barrier()
    kda.load()
    dev = torch.device("cuda", local_rank)
    stream = torch.cuda.current_stream()

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev).view(torch.bfloat16)

    def t(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    # ---- workloads (seeded, synthetic; per-rank seed so replicas differ) ----
    pf = inputs.prefill_inputs(seed=rank, lengths=[PREFILL_T], H=H, slots=16)
    gate = kda.Gate(A_log=t(pf["A_log"]), dt_bias=t(pf["dt_bias"]), lower_bound=-5.0)
    D = kda.dims(H)
    P = {n: bf(pf[n]) for n in ("q", "k", "v", "g", "beta")}
    p_pool = t(pf["pool"])
    p_idx = t(pf["state_idx"])
    p_cu = t(pf["cu_seqlens"])
    p_o = torch.empty((PREFILL_T, H, K), dtype=torch.bfloat16, device=dev)
    ws = torch.empty(kda.kda_prefill_workspace_size(D, 1, PREFILL_T), dtype=torch.uint8, device=dev)

    # The 1 x 4096 call again with the state at the start of every chunk
    # written out, and one 32768-token sequence prefilled by one call or by 8
    # calls of 4096 tokens that continue its state through the pool slot.
    p_inter = torch.empty((PREFILL_T // CHUNK, H, K, K), device=dev)
    if not args.no_long:
        lg = inputs.prefill_inputs(seed=50 + rank, lengths=[LONG_T], H=H, slots=2, state_idx=[1])
        LG = {n: bf(lg[n]) for n in ("q", "k", "v", "g", "beta")}
        lg_pool, lg_idx = t(lg["pool"]), t(lg["state_idx"])
        lg_cu = {T_: t(np.array([0, T_], np.int32)) for T_ in (LONG_T, LONG_T // LONG_CALLS)}
        lg_o = torch.empty((LONG_T, H, K), dtype=torch.bfloat16, device=dev)
        lg_ws = torch.empty(kda.kda_prefill_workspace_size(D, 1, LONG_T), dtype=torch.uint8, device=dev)
        del lg

    # Decode, verify and commit run args.layers calls back to back, each on its own
    # copy of the state pool, inputs and outputs (as consecutive KDA layers of
    # one model do), so every call starts from data no earlier call touched.
    dd = inputs.decode_inputs(seed=100 + rank, B=DECODE_B, H=H, slots=240)
    vd = inputs.verify_inputs(seed=200 + rank, B=VERIFY_B, T=VERIFY_T, H=H, slots=240)
    d_pool0, v_pool0 = t(dd["pool"]), t(vd["pool"])
    # every request accepts some prefix, so every commit moves one state
    acc_host = np.random.default_rng(rank).integers(0, VERIFY_T, size=COMMIT_B).astype(np.int32)
    L = []
    for _ in range(args.layers):
        L.append({
            "DX": {n: bf(dd[n]) for n in ("mixed_qkv", "a", "b")},
            "d_pool": d_pool0.clone(), "d_idx": t(dd["state_idx"]),
            "d_o": torch.empty((DECODE_B, H, K), dtype=torch.bfloat16, device=dev),
            "VX": {n: bf(vd[n]) for n in ("mixed_qkv", "a", "b")},
            "v_pool": v_pool0.clone(), "v_idx": t(vd["state_idx"]), "v_par": t(vd["parent"]),
            "v_o": torch.empty((VERIFY_B, VERIFY_T, H, K), dtype=torch.bfloat16, device=dev),
            "v_snap": torch.empty((VERIFY_B, VERIFY_T, H, K, K), device=dev),
            "v_snap2": torch.empty((VERIFY_B, VERIFY_T, H, K, K), device=dev),
            "v_pool_r": v_pool0.clone(),
            "ring": torch.empty((kda.kda_replay_ring_bytes(D, VERIFY_B, VERIFY_T) // 4,), device=dev),
            "accepted": t(acc_host),
        })
    del d_pool0, v_pool0
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def flush_l2():
        # A write larger than L2 evicts every line the previous phase left;
        # reading the buffer back then writes the flush's own dirty lines out,
        # so the next phase starts from a cold L2 with nothing left to write back.
        flush.zero_()
        flush.view(torch.int64).sum()

    phases = ["prefill", "decode", "verify_chain", "verify_tree", "commit", "verify_replay", "commit_replay",
              "prefill_states", "prefill_split"] + ([] if args.no_long else ["prefill_long", "prefill_long_calls"])
    # The prefill's state pass is a dependent launch of its chunk transform
    # (its CTAs start as the transform's leave), which an event between the
    # two kernels would turn into an ordinary launch.  So the headline prefill
    # phase has events around the call only, and "prefill_split" repeats the
    # same call with a third event between the kernels: the transform's span
    # (ev0 -> ev1) and the pass's (ev1 -> ev2).
    kernels = ["prefill_transform", "prefill_pass", "decode", "verify_chain", "verify_tree", "commit",
               "verify_replay", "commit_replay"]

    def run_call(name, x):
        if name in ("prefill", "prefill_split"):
            kda.kda_prefill(D, gate, P["q"], P["k"], P["v"], P["g"], P["beta"], p_pool, p_idx, p_cu, 1,
                            p_o, workspace=ws)
        elif name == "decode":
            kda.kda_decode_packed(D, gate, x["DX"]["mixed_qkv"], x["DX"]["a"], x["DX"]["b"], x["d_pool"],
                                  x["d_idx"], x["d_o"])
        elif name == "verify_chain":
            kda.kda_verify_chain(D, gate, x["VX"]["mixed_qkv"], x["VX"]["a"], x["VX"]["b"], VERIFY_B,
                                 VERIFY_T, x["v_pool"], x["v_idx"], x["v_o"], x["v_snap"])
        elif name == "verify_tree":
            kda.kda_verify_tree(D, gate, x["VX"]["mixed_qkv"], x["VX"]["a"], x["VX"]["b"], VERIFY_B,
                                VERIFY_T, x["v_par"], x["v_pool"], x["v_idx"], x["v_o"], x["v_snap2"])
        elif name == "verify_replay":
            kda.kda_verify_chain_replay(D, gate, x["VX"]["mixed_qkv"], x["VX"]["a"], x["VX"]["b"], VERIFY_B,
                                        VERIFY_T, x["v_pool_r"], x["v_idx"], x["v_o"], x["ring"])
        elif name == "commit_replay":
            kda.kda_commit_replay(D, x["ring"], COMMIT_B, VERIFY_T, x["accepted"], x["v_pool_r"], x["v_idx"])
        elif name == "prefill_states":
            kda.kda_prefill(D, gate, P["q"], P["k"], P["v"], P["g"], P["beta"], p_pool, p_idx, p_cu, 1,
                            p_o, p_inter, workspace=ws)
        elif name == "prefill_long":
            kda.kda_prefill(D, gate, *(LG[n] for n in ("q", "k", "v", "g", "beta")), lg_pool, lg_idx,
                            lg_cu[LONG_T], 1, lg_o, workspace=lg_ws)
        elif name == "prefill_long_calls":  # call x of 8, continuing the state
            n_ = LONG_T // LONG_CALLS
            part = slice(x * n_, (x + 1) * n_)
            kda.kda_prefill(D, gate, *(LG[n][part] for n in ("q", "k", "v", "g", "beta")), lg_pool, lg_idx,
                            lg_cu[n_], 1, lg_o[part], workspace=lg_ws)
        elif name == "commit":
            kda.kda_commit(D, x["v_snap"], COMMIT_B, VERIFY_T, x["accepted"], x["v_pool"], x["v_idx"])

    def calls(name):
        if name == "prefill_long_calls":
            return list(range(LONG_CALLS))
        return [None] if name.startswith("prefill") else L

    def run_phase(name, ev=None):
        """One phase; with events, ev[0] is recorded right before the first
        kernel and ev[2] right after the last (in "prefill_split" ev[1]
        between the two prefill kernels), as graph nodes when captured."""
        cs = calls(name)
        for i, x in enumerate(cs):
            if ev is not None:
                first, last = i == 0, i == len(cs) - 1
                kda.kda_set_stage_events([ev[0] if first else None, ev[1] if name == "prefill_split" else None,
                                          ev[2] if last else None])
            run_call(name, x)
        kda.kda_set_stage_events(None)

    def stage_events():
        # torch creates the CUDA event on first record(): record once so the
        # handle exists, then the library re-records it around its kernels
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in ev:
            e.record(stream)
        return ev

    # Each phase is captured in a CUDA graph and timed as graph replays (the
    # pages' microbenchmark method), so host-side launch latency stays out of
    # the measured intervals.  Every (step, phase) has its own graph and its
    # own events.
    for _ in range(max(args.warmup, 3)):
        for name in phases:
            flush_l2()
            run_phase(name)
    torch.cuda.synchronize()

    def capture(name, ev):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run_phase(name, ev)
        return g

    step_graphs = []
    for _ in range(args.steps):
        row = {}
        for n in phases:
            ev = stage_events()
            row[n] = (capture(n, ev), ev)
        step_graphs.append(row)
    torch.cuda.synchronize()
    for _ in range(2):  # warm the replays
        for n in phases:
            flush_l2()
            step_graphs[0][n][0].replay()
    torch.cuda.synchronize()

    def one_step(step):
        times = {}
        for name in phases:
            flush_l2()
            g, ev = step_graphs[step][name]
            g.replay()
            times[name] = ev
        return times

    sampler = ClockSampler(physical_gpu_index(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    records = [one_step(step) for step in range(args.steps)]
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None

    # per-call milliseconds of every phase (a layer phase's span / args.layers;
    # a prefill phase's whole span, however many calls it makes)
    ph_ms = {n: [r[n][0].elapsed_time(r[n][2]) / (1 if n.startswith("prefill") else len(calls(n)))
                 for r in records] for n in phases}
    k_ms = {
        "prefill_transform": [r["prefill_split"][0].elapsed_time(r["prefill_split"][1]) for r in records],
        "prefill_pass": [r["prefill_split"][1].elapsed_time(r["prefill_split"][2]) for r in records],
        "decode": ph_ms["decode"], "verify_chain": ph_ms["verify_chain"],
        "verify_tree": ph_ms["verify_tree"], "commit": ph_ms["commit"],
        "verify_replay": ph_ms["verify_replay"], "commit_replay": ph_ms["commit_replay"],
    }
    tot = {n: sum(v) for n, v in ph_ms.items()}
    tot = dict(zip(phases, max_over_ranks([tot[n] for n in phases], world, dev)))
    # a step is one pass over the hot path's phases; the chunk-state and long
    # prefills are reported on their own and kept out of ms_per_step
    core = [n for n in phases if n not in ("prefill_states", "prefill_split", "prefill_long", "prefill_long_calls")]

    # ---- e2e: prefill through the C ABI with host buffers ----
    host = {n: torch.from_numpy(np.ascontiguousarray(pf[n])).pin_memory()
            for n in ("q", "k", "v", "g", "beta", "state_idx", "cu_seqlens")}
    o_host = torch.empty((PREFILL_T, H, K), dtype=torch.int16).pin_memory()
    dbuf = {n: torch.empty(host[n].shape, dtype=host[n].dtype, device=dev) for n in host}
    h2d = sum(x.numel() * x.element_size() for x in host.values())
    d2h = o_host.numel() * o_host.element_size()
    e2e_steps = max(3, min(args.steps, 50))
    ev_e2e = []
    for i in range(e2e_steps + 3):
        flush_l2()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for n in host:
            dbuf[n].copy_(host[n], non_blocking=True)
        kda.kda_prefill(D, gate, *(dbuf[n].view(torch.bfloat16) for n in ("q", "k", "v", "g", "beta")),
                        p_pool, dbuf["state_idx"], dbuf["cu_seqlens"], 1, p_o, workspace=ws)
        o_host.copy_(p_o.view(torch.int16), non_blocking=True)
        e1.record(stream)
        if i >= 3:
            ev_e2e.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks([sum(a.elapsed_time(b) for a, b in ev_e2e)], world, dev)[0]

    # ---- e2e of the layer phases: decode B=48 and chain verify 16x6 with their
    # inputs copied from pinned host memory and o read back every call ----
    e2e_layers = {}
    for name, rows_host, B_, T_ in (("decode_b48", dd, DECODE_B, 1), ("verify_chain_b16x6", vd, VERIFY_B, VERIFY_T)):
        hx = {n: torch.from_numpy(np.ascontiguousarray(rows_host[n])).pin_memory() for n in ("mixed_qkv", "a", "b")}
        dx = {n: torch.empty(hx[n].shape, dtype=torch.int16, device=dev) for n in hx}
        x0 = L[0]
        o_dev = x0["d_o"] if T_ == 1 else x0["v_o"]
        o_h = torch.empty(o_dev.shape, dtype=torch.int16).pin_memory()
        ev_l = []
        for i in range(e2e_steps + 3):
            flush_l2()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for n in hx:
                dx[n].copy_(hx[n], non_blocking=True)
            if T_ == 1:
                kda.kda_decode_packed(D, gate, *(dx[n].view(torch.bfloat16) for n in ("mixed_qkv", "a", "b")),
                                      x0["d_pool"], x0["d_idx"], o_dev)
            else:
                kda.kda_verify_chain(D, gate, *(dx[n].view(torch.bfloat16) for n in ("mixed_qkv", "a", "b")),
                                     B_, T_, x0["v_pool"], x0["v_idx"], o_dev, x0["v_snap"])
            o_h.copy_(o_dev.view(torch.int16), non_blocking=True)
            e1.record(stream)
            if i >= 3:
                ev_l.append((e0, e1))
        torch.cuda.synchronize()
        us = statistics.mean(a.elapsed_time(b) for a, b in ev_l) * 1e3
        e2e_layers[name] = {"us_per_call": round(us, 2),
                            "h2d_bytes": sum(x.numel() * x.element_size() for x in hx.values()),
                            "d2h_bytes": o_h.numel() * o_h.element_size()}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    del L, step_graphs, records
    torch.cuda.empty_cache()
    extras = {} if args.no_extras else run_extras(args, dev, stream, flush_l2, gate_seed=rank)

    hbm, bf16_tf, sm_max, peak_kind = _peaks()
    # every prefill call here (bounded gate) is a chunk transform and a state pass
    def launches_of(T_):
        return 2

    prefill_launches = launches_of(PREFILL_T)
    # the chunk-state and split-timing prefills, and the long ones
    extra_launches = 2 * prefill_launches + (0 if args.no_long else
                                             launches_of(LONG_T) + LONG_CALLS * launches_of(LONG_T // LONG_CALLS))
    steps = args.steps
    prefill_s = tot["prefill"] / 1e3
    value = replica_throughput(PREFILL_T, steps, world, prefill_s)
    mean_k = {n: statistics.mean(v) for n, v in k_ms.items()}
    # The chunk transform's slower roofline is HBM: its input bytes at the
    # measured copy bandwidth (9.9 us at 1 x 4096) take far longer than its
    # algorithmic flops (2.2 GFLOP, hi/lo split passes not counted) at the
    # dense BF16 peak (1.2 us).  It is judged on those bytes over the span of
    # its launch; its flop rate is reported beside.  The state pass (its span
    # after the transform) has no roofline of its own.
    work = {
        "prefill_transform": ("hbm", transform_bytes(PREFILL_T) / 1e9, hbm, "GB/s"),
        "prefill_pass": None,
        "decode": ("hbm", decode_bytes(DECODE_B) / 1e9, hbm, "GB/s"),
        "verify_chain": ("hbm", verify_bytes(VERIFY_B, VERIFY_T) / 1e9, hbm, "GB/s"),
        "verify_tree": ("hbm", verify_bytes(VERIFY_B, VERIFY_T) / 1e9, hbm, "GB/s"),
        "commit": ("hbm", commit_bytes(COMMIT_B) / 1e9, hbm, "GB/s"),
        "verify_replay": ("hbm", verify_replay_bytes(VERIFY_B, VERIFY_T) / 1e9, hbm, "GB/s"),
        "commit_replay": ("hbm", commit_replay_bytes(acc_host, VERIFY_T) / 1e9, hbm, "GB/s"),
    }
    dom = max((n for n in mean_k if work[n] is not None), key=mean_k.get)
    bound, per_launch, peak, unit = work[dom]
    achieved = per_launch / (mean_k[dom] / 1e3)
    src = _source_hash()
    tr = NCU_TRAFFIC.get(dom)
    traffic = tr["bytes"] if tr and tr.get("src") == src else None
    roofline = {"kernel": dom, "bound": bound, "achieved": round(achieved, 3), "peak": peak,
                "tensor_tflops": round(transform_flops(PREFILL_T) / 1e12 / (mean_k["prefill_transform"] / 1e3), 3),
                "tensor_frac": round(transform_flops(PREFILL_T) / 1e12 / (mean_k["prefill_transform"] / 1e3) / bf16_tf, 5),
                "unit": unit, "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": f"{peak_kind} ({'dense BF16 burst' if bound == 'tensor' else 'HBM copy'})"}
    kern = {}
    for n in kernels:
        if work[n] is None:
            kern[n] = {"us": round(mean_k[n] * 1e3, 2)}
            continue
        b_, w_, p_, u_ = work[n]
        a_ = w_ / (mean_k[n] / 1e3)
        kern[n] = {"us": round(mean_k[n] * 1e3, 2), "bound": b_, "achieved": round(a_, 2), "unit": u_,
                   "frac": round(a_ / p_, 4)}
    phase_out = {
        "prefill_1x4096": {"us": round(statistics.mean(ph_ms["prefill"]) * 1e3, 2),
                           "tok_s": round(value / world, 1),
                           "hbm_frac_of_call": round(prefill_bytes(PREFILL_T) / (statistics.mean(ph_ms["prefill"]) / 1e3) / 1e9 / hbm, 4)},
        "layers_per_replay": args.layers,
        "decode_b48": {"us": round(statistics.mean(ph_ms["decode"]) * 1e3, 2)},
        "verify_chain_b16x6": {"us": round(statistics.mean(ph_ms["verify_chain"]) * 1e3, 2)},
        "verify_tree_b16x6": {"us": round(statistics.mean(ph_ms["verify_tree"]) * 1e3, 2)},
        "commit_b16": {"us": round(statistics.mean(ph_ms["commit"]) * 1e3, 2)},
        "verify_replay_b16x6": {"us": round(statistics.mean(ph_ms["verify_replay"]) * 1e3, 2)},
        "commit_replay_b16": {"us": round(statistics.mean(ph_ms["commit_replay"]) * 1e3, 2)},
        "kernels": kern,
        # chunk-start states out, and a long sequence in one call or continued
        # over several calls through its pool slot
        "prefill_1x4096_chunk_states": {
            "us": round(statistics.mean(ph_ms["prefill_states"]) * 1e3, 2),
            "states_bytes": PREFILL_T // CHUNK * H * K * K * 4},
    }
    if not args.no_long:
        phase_out["prefill_1x32768"] = {"us": round(statistics.mean(ph_ms["prefill_long"]) * 1e3, 2),
                                        "tok_s": round(LONG_T / statistics.mean(ph_ms["prefill_long"]) * 1e3, 1)}
        phase_out["prefill_32768_as_8x4096"] = {
            "us": round(statistics.mean(ph_ms["prefill_long_calls"]) * 1e3, 2),
            "tok_s": round(LONG_T / statistics.mean(ph_ms["prefill_long_calls"]) * 1e3, 1)}
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(sum(tot[n] for n in core) / steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in / fp32 state",
        "data": "synthetic (seeded; q,k,v,a,beta ~N(0,1) BF16, A_log~U(-1,1), dt_bias~N(0,0.1), state~N(0,0.02))",
        "config": {"workload": "KDA prefill 1x4096 tokens, 16 heads x 128 (+ decode B=48, verify 16x6 chain/tree/replay, commit 16 snapshot/replay)",
                   "timing": (f"CUDA-graph replay per phase; CUDA events recorded as graph nodes around the phase's kernels; "
                              f"decode/verify/commit: {args.layers} layer calls back to back, each on its own state pool and "
                              f"buffers, time per call = span / {args.layers}"),
                   "global_batch": world, "seq_len": PREFILL_T, "heads": H, "head_dim": K,
                   "parallelism": f"replicas x{world}", "l2": "flushed before every phase (512 MiB write, then the same buffer read back); layer calls touch disjoint buffers larger than L2"},
        "gpu_launches": steps * (prefill_launches + (len(core) - 1) * args.layers + extra_launches),
        "phases": phase_out,
        "roofline": roofline,
        "e2e": {"value": round(replica_throughput(PREFILL_T, e2e_steps, world, e2e_ms / 1e3), 1),
                "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clocks, "wall_s_timed": round(wall, 3), "source_hash": src,
    }
    phase_out["e2e_layers"] = e2e_layers
    phase_out.update(extras)
    if world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(pf, budget_s=10.0)
        out["cpu_baseline"]["single_thread"] = cpu_baseline(pf, budget_s=5.0, tokens=256, threads=1)
    print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


def cpu_baseline(pf, budget_s=10.0, tokens=None, threads=None):
    """The oracle, as it stands, on this host's cores (all of them, or
    `threads`)."""
    from oracle import kda_oracle as ko

    T = PREFILL_T if tokens is None else tokens
    gate = ko.Gate(H, K, K, A_log=pf["A_log"], dt_bias=pf["dt_bias"], lower_bound=-5.0)
    cores = threads or os.cpu_count() or 1
    sl = {n: np.ascontiguousarray(pf[n][:T]) for n in ("q", "k", "v", "g", "beta")}
    runs, t0 = 0, time.perf_counter()
    while True:
        pool = pf["pool"].astype(np.float64)
        ko.prefill(gate, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], pool, pf["state_idx"],
                   np.array([0, T], np.int32), nthreads=cores)
        runs += 1
        el = time.perf_counter() - t0
        if el >= budget_s or runs >= 50:
            break
    return {"value": round(T * runs / el, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"prefill 1x{T} tokens x 16 heads ({'full call' if T == PREFILL_T else 'first tokens of the 1x4096 call'}), "
                      f"{runs} run(s) in {el:.1f} s"}


def run_extras(args, dev, stream, flush_l2, gate_seed=0):
    """Every other configuration of the workload, each timed on its own and
    reported beside the step (not in ms_per_step): the 1x128 prefill at 4
    heads, 1x8192 and 2x4096 at 16 heads, 8 varlen sequences in a 32768-row
    bucket with garbage padding rows and a 240-slot pool, 256 sequences of
    128 tokens in one call, decode at 1 and 16
    requests, and chain and tree verify over the request sweep at 6 draft
    tokens.  Each is one CUDA graph (8 layer calls on disjoint buffers for the
    layer phases) replayed after an L2 flush, its kernels bracketed by events
    recorded as graph nodes."""
    import torch

    from linear_attention_serving_gated_gb300 import inputs, kda

    hbm = _peaks()[0]
    reps = max(3, min(args.steps, 20))

    def bf(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev).view(torch.bfloat16)

    def t(x):
        return torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    def timed(fn):
        for _ in range(3):
            flush_l2()
            fn(None)
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for e in ev:
            e.record(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn(ev)
        ms = []
        for _ in range(reps):
            flush_l2()
            g.replay()
            torch.cuda.synchronize()
            ms.append(ev[0].elapsed_time(ev[2]))
        del g
        return statistics.mean(ms)

    def with_events(ev, calls):
        for i, c in enumerate(calls):
            if ev is not None:
                first, last = i == 0, i == len(calls) - 1
                kda.kda_set_stage_events([ev[0] if first else None, ev[1] if first and last else None,
                                          ev[2] if last else None])
            c()
        kda.kda_set_stage_events(None)

    out = {}

    # ---- prefills ----
    rng0 = np.random.default_rng(0)
    prefills = [
        ("prefill_1x128_h4", dict(seed=0, lengths=[128], H=4, slots=4, state_idx=[0]), True),
        ("prefill_1x8192", dict(seed=1, lengths=[8192], H=H, slots=16), True),
        ("prefill_2x4096_fixed", dict(seed=3, lengths=[4096, 4096], H=H, slots=16, varlen=False), False),
        ("prefill_varlen_8seq_32k_bucket", dict(seed=0, lengths=inputs.varlen_lengths(rng0), H=H, slots=240,
                                                gb_rows=32768), True),
        # a batch of many short prefills: 256 sequences x 128 tokens
        ("prefill_256x128", dict(seed=5, lengths=[128] * 256, H=H, slots=256), True),
    ]
    for name, kw, varlen in prefills:
        d = inputs.prefill_inputs(**kw)
        heads = kw["H"]
        Dh = kda.dims(heads)
        gate = kda.Gate(A_log=t(d["A_log"]), dt_bias=t(d["dt_bias"]), lower_bound=-5.0)
        x = {n: bf(d[n]) for n in ("q", "k", "v", "g", "beta")}
        pool, idx = t(d["pool"]), t(d["state_idx"])
        cu = t(d["cu_seqlens"]) if varlen else None
        lens = [int(v) for v in d["lengths"]]
        T_ = sum(lens)
        o = torch.empty((T_, heads, K), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(kda.kda_prefill_workspace_size(Dh, len(lens), T_), dtype=torch.uint8, device=dev)
        del d
        ms = timed(lambda ev: with_events(ev, [lambda: kda.kda_prefill(
            Dh, gate, x["q"], x["k"], x["v"], x["g"], x["beta"], pool, idx, cu, len(lens), o, workspace=ws)]))
        byts = varlen_prefill_bytes(lens, heads)
        out[name] = {"us": round(ms * 1e3, 2), "tok_s": round(T_ / (ms / 1e3), 1), "tokens": T_,
                     "sequences": len(lens), "heads": heads,
                     "hbm_frac_of_call": round(byts / (ms / 1e3) / 1e9 / hbm, 4)}
        del x, pool, idx, cu, o, ws
        torch.cuda.empty_cache()

    # ---- decode and verify sweeps, 8 layer calls on disjoint buffers ----
    layers = args.layers
    D = kda.dims(H)
    for B in DECODE_SWEEP:
        d = inputs.decode_inputs(seed=100 + B + gate_seed, B=B, H=H, slots=240)
        gate = kda.Gate(A_log=t(d["A_log"]), dt_bias=t(d["dt_bias"]), lower_bound=-5.0)
        Lx = [{"x": {n: bf(d[n]) for n in ("mixed_qkv", "a", "b")}, "pool": t(d["pool"]),
               "idx": t(d["state_idx"]), "o": torch.empty((B, H, K), dtype=torch.bfloat16, device=dev)}
              for _ in range(layers)]
        ms = timed(lambda ev: with_events(ev, [
            (lambda y=y: kda.kda_decode_packed(D, gate, y["x"]["mixed_qkv"], y["x"]["a"], y["x"]["b"], y["pool"],
                                               y["idx"], y["o"])) for y in Lx]))
        us = ms * 1e3 / layers
        out[f"decode_b{B}"] = {"us": round(us, 2), "hbm_frac": round(decode_bytes(B) / (us / 1e6) / 1e9 / hbm, 4)}
        del Lx
        torch.cuda.empty_cache()
    sweep = {}
    for B in VERIFY_SWEEP:
        d = inputs.verify_inputs(seed=200 + B + gate_seed, B=B, T=VERIFY_T, H=H, slots=240)
        gate = kda.Gate(A_log=t(d["A_log"]), dt_bias=t(d["dt_bias"]), lower_bound=-5.0)
        Lx = [{"x": {n: bf(d[n]) for n in ("mixed_qkv", "a", "b")}, "pool": t(d["pool"]),
               "idx": t(d["state_idx"]), "par": t(d["parent"]),
               "o": torch.empty((B, VERIFY_T, H, K), dtype=torch.bfloat16, device=dev),
               "snap": torch.empty((B, VERIFY_T, H, K, K), device=dev)} for _ in range(layers)]
        row = {}
        for mode in ("chain", "tree"):
            def call(y, mode=mode):
                if mode == "chain":
                    kda.kda_verify_chain(D, gate, y["x"]["mixed_qkv"], y["x"]["a"], y["x"]["b"], B, VERIFY_T,
                                         y["pool"], y["idx"], y["o"], y["snap"])
                else:
                    kda.kda_verify_tree(D, gate, y["x"]["mixed_qkv"], y["x"]["a"], y["x"]["b"], B, VERIFY_T,
                                        y["par"], y["pool"], y["idx"], y["o"], y["snap"])
            ms = timed(lambda ev: with_events(ev, [(lambda y=y: call(y)) for y in Lx]))
            us = ms * 1e3 / layers
            row[mode] = {"us": round(us, 2),
                         "hbm_frac": round(verify_bytes(B, VERIFY_T) / (us / 1e6) / 1e9 / hbm, 4)}
        sweep[str(B)] = row
        del Lx
        torch.cuda.empty_cache()
    out["verify_sweep_x6"] = sweep
    out["extras_timing"] = f"one CUDA graph per configuration, {reps} replays after an L2 flush, mean"
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import kda_oracle as ko
    from linear_attention_serving_gated_gb300 import inputs

    ko.build()
    pf = inputs.prefill_inputs(seed=0, lengths=[PREFILL_T], H=H, slots=16)
    sample_T = 512  # bounded sample of the 1x4096 workload per step
    gate = ko.Gate(H, K, K, A_log=pf["A_log"], dt_bias=pf["dt_bias"], lower_bound=-5.0)
    cores = os.cpu_count() or 1
    sl = {n: np.ascontiguousarray(pf[n][:sample_T]) for n in ("q", "k", "v", "g", "beta")}

    def step():
        pool = pf["pool"].astype(np.float64)
        ko.prefill(gate, sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], pool, pf["state_idx"],
                   np.array([0, sample_T], np.int32), nthreads=cores)

    for _ in range(max(args.warmup, 1)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = sample_T * args.steps / el
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same generator)",
        "config": {"workload": "KDA prefill 1x4096 tokens, 16 heads x 128 (oracle on a 512-token sample per step)",
                   "seq_len": PREFILL_T, "heads": H, "head_dim": K},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {sample_T} tokens of the 1x4096 x 16-head prefill per step"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="decode/verify/commit calls per timed replay, each on its own buffers")
    ap.add_argument("--no-long", action="store_true",
                    help="skip the 32768-token prefill phases (about 1.4 GB less device memory, e.g. under ncu)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other configurations (1x128 at 4 heads, 1x8192, 2x4096, varlen 32K bucket, 256x128, "
                         "decode 1/16, verify sweep)")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", args.gpus if "RANK" in os.environ else 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
