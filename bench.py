#!/usr/bin/env python
"""Decode-step throughput of retrieval-based sparse decode attention.

Workload: one Llama-3-8B-shaped decode-attention layer at 128K context
(B=1, 32 query / 8 KV heads, head_dim 128, bf16 K/V, candidate budget 8192,
top-k 2048, local window 128). A step is one pass of the whole hot path for
one layer: append one token (encode its key), select (coarse score,
candidates, exact rescoring, top-k) and attend, by default through
kvr_select_attend (one launch). Steps rotate over 32 layer caches (17.7 GB)
so every step reads its cache cold from HBM (inputs larger than L2); each
step appends a token and takes a fresh query. The timed loop replays one
CUDA graph per decode iteration (every layer once) plus one for a remainder
of steps, so any step count times the same chained kernels.

Output: one JSON line (rank 0). --impl reference times the CPU oracle on the
host cores instead, on the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse decode-attention steps/s at 128K ctx; achieved HBM GB/s vs peak"
OFFLOAD_METRIC = "sparse decode-attention steps/s at 1M ctx, K/V in host memory"
MILLION_METRIC = "sparse decode-attention steps/s at 1M ctx, K/V in HBM; achieved HBM GB/s vs peak"
LAYERS = 32
LAYERS_DEFAULT = LAYERS


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_traffic(kernel, workload):
    """DRAM bytes per launch of `kernel` on `workload` from the ncu capture
    recorded in profiles/traffic.json (under "kernel/workload", or under
    "kernel" when captured on that workload), or None when there is no
    capture of that kernel on that workload or its sources have changed
    since the capture (the counters then describe another launch)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            table = json.load(f)
        rec = table.get(kernel + "/" + workload, table.get(kernel))
        if rec is None or rec["workload"] != workload:
            return None
        m = hashlib.sha256()
        for name in rec["sources"]:
            with open(os.path.join(ROOT, "sparse_decode_attention_gb300", "csrc", name), "rb") as f:
                m.update(f.read())
    except (OSError, KeyError, ValueError):
        return None
    return int(rec["dram_bytes_per_launch"]) if m.hexdigest() == rec["sources_sha256"] else None


def algorithmic_bytes(w, rerank="exact"):
    """Bytes the hot path must read or write per step per unit (batch x kv
    head). With the reranker, a candidate costs its record (6 d/8 bytes)
    instead of its K row, and the appended key also gets a record."""
    N = w.N
    pool = N - w.W
    Cp = min(w.C, pool)
    kp = min(w.k, Cp)
    row = w.d * 2  # bf16 row
    rec = 6 * w.d // 8
    codes = pool * (w.d // 8)
    cand_rows = Cp * (rec if rerank == "rsq" else row)
    sel_kv = (kp + w.W) * 2 * row
    q = w.G * w.d * 2
    units = w.B * w.Hkv
    enc = row + w.d // 8 + (rec if rerank == "rsq" else 0)
    return dict(select=units * (codes + cand_rows + q), attend=units * (sel_kv + q),
                encode=units * enc, units=units)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.strip().split(", ") for r in self.f.read().splitlines() if r.strip()]
        self.f.close()
        os.unlink(self.f.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() in ("active", "1"):
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# CPU oracle arm (cpu_baseline leg and --impl reference)
# --------------------------------------------------------------------------

def oracle_unit_inputs(w, device, h=0):
    """Unit (b=0, kv head h) of layer 0 of the workload, as host fp32 arrays,
    with 64 of its per-step query groups."""
    import torch
    import workloads as wl
    import oracle
    K, V, qb = wl.make_cache(w.with_(B=1), device=device, cap=w.N)
    K0 = oracle.f32(K[0, h].cpu())
    V0 = oracle.f32(V[0, h].cpu())
    sgn = wl.srht_signs(w.d).numpy()
    codes = oracle.encode(K0, sgn)
    G = w.G
    qs = [oracle.f32(wl.step_query(w, qb, t)[0, h * G:(h + 1) * G].cpu()) for t in range(64)]
    del K, V
    if device != "cpu":
        torch.cuda.empty_cache()
    return K0, V0, codes, sgn, qs


def _oracle_steps(w, inputs, budget_s, min_steps=1, max_steps=None):
    """Oracle decode steps of one unit until the budget is spent: (unit-steps, s)."""
    import numpy as np
    import oracle
    K0, V0, codes, sgn, qs = inputs
    scale = np.float32(1 / math.sqrt(w.d))
    done, t0 = 0, time.perf_counter()
    while True:
        q = qs[done % len(qs)]
        idx, cnt = oracle.select_unit(q, K0, codes, w.N, sgn, w.C, w.k, w.W, w.lut)
        oracle.attend_unit(q, K0, V0, w.N, idx[:cnt], cnt, w.W, scale)
        done += 1
        el = time.perf_counter() - t0
        if (el >= budget_s and done >= min_steps) or (max_steps and done >= max_steps):
            break
    return done, el


def time_oracle(w, budget_s, device, min_steps=1, max_steps=None):
    """Oracle decode steps on one host core: each step runs one unit and
    counts 1/units of a whole step. Returns (steps/s, seconds, unit-steps)."""
    units = w.B * w.Hkv
    done, el = _oracle_steps(w, oracle_unit_inputs(w, device), budget_s, min_steps, max_steps)
    return (done / units) / el, el, done


def box_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def time_oracle_all_cores(w, budget_s, device):
    """The oracle on every host core: one thread per (batch 0, kv head) unit,
    up to the core count (the oracle's C calls release the interpreter lock).
    Returns (steps/s, seconds, unit-steps, threads)."""
    import concurrent.futures as cf
    threads = max(1, min(box_cores(), w.B * w.Hkv))
    inputs = [oracle_unit_inputs(w, device, h=h % w.Hkv) for h in range(threads)]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        res = list(ex.map(lambda x: _oracle_steps(w, x, budget_s), inputs))
    el = time.perf_counter() - t0
    done = sum(r[0] for r in res)
    return (done / (w.B * w.Hkv)) / el, el, done, threads


def cpu_baseline_line(w, seconds, device):
    """cpu_baseline: the oracle on all host cores (headline) and on one."""
    units = w.B * w.Hkv
    v1, el1, d1 = time_oracle(w, seconds / 2, device)
    va, ela, da, th = time_oracle_all_cores(w, seconds / 2, device)
    return {"value": va, "unit": "steps/s", "cores": th, "kind": "oracle",
            "box_cores": box_cores(),
            "sample": "%d unit-steps of the %s workload on %d threads (one per kv head of batch "
                      "entry 0) in %.1f s; steps/s = unit-steps / %d / s"
                      % (da, w.name, th, ela, units),
            "single_thread": {"value": v1, "unit": "steps/s", "cores": 1,
                              "sample": "%d unit-steps (batch 0, kv head 0) in %.1f s"
                                        % (d1, el1)}}


def run_reference(args, w):
    rank, local, world = dist_setup(args)
    if rank != 0:
        return
    import torch
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    per_step_budget = float(os.environ.get("KVR_REF_STEP_SECONDS", "0.5"))
    # warm-up: one unit-step per warm-up step (untimed)
    time_oracle(w, 0.0, dev, max_steps=max(1, min(args.warmup, 3)))
    budget = per_step_budget * args.steps
    value, el, done = time_oracle(w, budget, dev, min_steps=args.steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(config_of(w), rerank="exact", votes="hamming"),
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": 1, "kind": "oracle",
                         "box_cores": box_cores(),
                         "sample": "%d unit-steps (batch 0, kv head 0 of %d units) of the %s "
                                   "workload, %.1f s; steps/s = unit-steps / %d / s"
                                   % (done, w.B * w.Hkv, w.name, el, w.B * w.Hkv)},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(w):
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
            "context": w.N, "C": w.C, "k": w.k, "W": w.W, "lut": list(w.lut),
            "layers_rotated": LAYERS,
            "l2": "inputs larger than L2: steps rotate over %d layer caches" % LAYERS,
            "parallelism": "replicas (independent units per GPU)"}


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------

class Layer:
    def __init__(self, w, l, kvr, wl, torch, sgn, cap, nq, rerank="exact", host=False, mag=False):
        dev = "cuda"
        # rows [N, cap) hold the keys and values the appending steps add
        K, V, qb = wl.make_cache(w, device=dev, cap=cap, seed=w.seed + 1000 * l)
        self.K, self.V = K, V
        # fresh per-step queries q_t = q_base + 0.1 N(0, 1), one per decode iteration
        self.qs = [wl.step_query(w, qb, t, seed=w.seed + 1000 * l).contiguous() for t in range(nq)]
        self.q = self.qs[0]
        self.codes = kvr.codes_buffer(kvr.Shape.of(K, self.q), dev)
        kvr.kvr_encode_keys(K, torch.zeros(w.B, dtype=torch.int32, device=dev), w.N, sgn,
                            self.codes)
        self.out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
        self.rec = None
        if rerank == "rsq":
            # reranker records of every key, kept beside the codes
            self.rec = kvr.rsq_buffer(K)
            kvr.kvr_encode_rsq(K, torch.zeros(w.B, dtype=torch.int32, device=dev), w.N, sgn,
                               self.rec)
        if host:
            # the full-precision cache moves to page-locked host memory; the
            # kernels read it through the device's mapping (no copy calls)
            self.K = torch.empty(K.shape, dtype=K.dtype, pin_memory=True)
            self.V = torch.empty(V.shape, dtype=V.dtype, pin_memory=True)
            self.K.copy_(K)
            self.V.copy_(V)
            del K, V
            torch.cuda.empty_cache()
        # the codes, K, V and lengths are never written by the kernel before a
        # selection in the step chain (the previous layer's attention), so it
        # may start on them early; V as an L2-prefetch hint for the separate
        # attention (the fused call reads V itself)
        flags = kvr.SELECT_EARLY_INPUTS | (kvr.SELECT_MAGNITUDE_VOTES if mag else 0)
        self.params = kvr.SelectParams(w.C, w.k, w.W, w.lut, flags=flags,
                                       V_prefetch=None if host else self.V, rsq_records=self.rec)

    def encode_new(self, kvr, pos_new, sgn, err, stream=None):
        """Code (and record) of the appended key."""
        kvr.kvr_encode_keys(self.K, pos_new, 1, sgn, self.codes, err, stream=stream)
        if self.rec is not None:
            kvr.kvr_encode_rsq(self.K, pos_new, 1, sgn, self.rec, err, stream=stream)


def run_gpu(args, w):
    import torch
    import sparse_decode_attention_gb300 as kvr
    import workloads as wl

    rank, local, world = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    kvr.load()
    sgn = wl.srht_signs(w.d, device=dev)
    host = args.workload == "million_offload"
    rerank = args.rerank or ("rsq" if host else "exact")
    mag = args.votes == "magnitude"
    fused = args.path == "fused"
    NQ = 16
    e2e_n = min(args.steps, args.e2e_steps)
    warm_iters = max(1, -(-args.warmup // LAYERS))
    timed_iters, rem = divmod(args.steps, LAYERS)
    # every appending step of a layer adds one row: warm-up and timed
    # iterations, the remainder, and the end-to-end passes (two modes)
    margin = warm_iters + timed_iters + 2 + 2 * (e2e_n // LAYERS + 2) + 8
    cap = w.N + margin
    layers = [Layer(w, l, kvr, wl, torch, sgn, cap, NQ, rerank, host, mag) for l in range(LAYERS)]
    shape = kvr.Shape.of(layers[0].K, layers[0].q)
    params = layers[0].params   # the flags of every layer's selection (workspace size)
    ws_s = kvr.workspace(kvr.kvr_select_workspace_size(shape, params), dev)
    ws_a = kvr.workspace(kvr.kvr_attend_workspace_size(shape, w.k, w.W), dev)
    idx = torch.empty((w.B, w.Hkv, w.k), dtype=torch.int32, device=dev)
    cnt = torch.empty((w.B, w.Hkv), dtype=torch.int32, device=dev)
    # the sequence lengths, then the appended key's rows; every decode
    # iteration first adds one to both (one small torch kernel per iteration)
    seqpos = torch.tensor([w.N] * w.B + [w.N - 1] * w.B, dtype=torch.int32, device=dev)
    seq, pos_new = seqpos[:w.B], seqpos[w.B:]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(w.d)

    def call(L, j):
        if fused:
            kvr.kvr_select_attend(L.qs[j], L.K, L.V, L.codes, seq, sgn, L.params, scale, idx, cnt,
                                  L.out, ws_s, err)
        else:
            kvr.kvr_select(L.qs[j], L.K, L.codes, seq, sgn, L.params, idx, cnt, ws_s, err)
            kvr.kvr_sparse_attend(L.qs[j], L.K, L.V, idx, cnt, seq, w.W, scale, L.out, ws_a, err)

    side = torch.cuda.Stream(device=dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def iteration(nl, j):
        # One decode iteration over the first nl layers: the lengths advance,
        # then each layer appends its key and runs its step. A key's code is
        # first read when it leaves the window, W iterations later, so the
        # encodes form one chain on a side stream, joined at the end; the main
        # stream is a chain of selection (+ attention) kernels linked by
        # programmatic dependent launch.
        main = torch.cuda.current_stream()
        seqpos.add_(1)
        fork.record(main)
        side.wait_event(fork)
        for L in layers[:nl]:
            L.encode_new(kvr, pos_new, sgn, err, stream=side)
            call(L, j)
        join.record(side)
        main.wait_event(join)

    # encode(s), selection (+ its vote lists), attention (fused: one launch)
    launches_per_step = (2 if fused else 3) + (1 if rerank == "rsq" else 0) + (1 if mag else 0)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):   # eager warm-up of the calls (no append)
        seqpos.sub_(1)
        iteration(2, 0)
    stream.synchronize()
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during warm-up")
    # Timed graphs carry no event nodes between kernels: an event between two
    # kernels serialises them and turns off programmatic dependent launch.
    # One graph per query set runs a whole decode iteration; the last graph
    # covers a remainder of steps (the first `rem` layers), so any step count
    # times the same chained path.
    graphs = []
    for j in range(NQ):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            iteration(LAYERS, j)
        graphs.append(g)
    g_rem = None
    if rem:
        g_rem = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_rem, stream=stream):
            iteration(rem, (warm_iters + timed_iters) % NQ)
    torch.cuda.synchronize()

    with torch.cuda.stream(stream):
        for i in range(warm_iters):
            graphs[i % NQ].replay()
    stream.synchronize()

    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(timed_iters)]
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(timed_iters):
            graphs[(warm_iters + i) % NQ].replay()
            marks[i].record()
        if g_rem is not None:
            g_rem.replay()
        t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms, world)
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the timed region")
    iter_us = []
    prev = t_start
    for m in marks:
        iter_us.append(prev.elapsed_time(m) * 1e3 / LAYERS)
        prev = m
    n_mid = w.N + warm_iters + timed_iters // 2

    # per-call durations: every layer's event graph, replayed in layer order
    # (each layer's inputs cold again), after the timed region, no append
    try:
        mk = lambda: torch.cuda.Event(enable_timing=True, external=True)
        mk()
        external = True
    except TypeError:
        external = False
    per = {"encode": [], "call": [], "select": [], "attend": []}
    if external:
        graphs_ev, evs = [], []
        for L in layers:
            ge = torch.cuda.CUDAGraph()
            ev = [mk() for _ in range(5)]
            with torch.cuda.graph(ge, stream=stream):
                ev[0].record()
                L.encode_new(kvr, pos_new, sgn, err)
                ev[1].record()
                call(L, 0)
                ev[2].record()
                kvr.kvr_select(L.q, L.K, L.codes, seq, sgn, L.params, idx, cnt, ws_s, err)
                ev[3].record()
                kvr.kvr_sparse_attend(L.q, L.K, L.V, idx, cnt, seq, w.W, scale, L.out, ws_a, err)
                ev[4].record()
            graphs_ev.append(ge)
            evs.append(ev)
        for rep in range(2):
            with torch.cuda.stream(stream):
                for ge in graphs_ev:
                    ge.replay()
            stream.synchronize()
            if rep == 0:
                continue
            for ev in evs:
                per["encode"].append(ev[0].elapsed_time(ev[1]))
                per["call"].append(ev[1].elapsed_time(ev[2]))
                per["select"].append(ev[2].elapsed_time(ev[3]))
                per["attend"].append(ev[3].elapsed_time(ev[4]))
        del graphs_ev
    avg = {k: (sum(v) / len(v) if v else None) for k, v in per.items()}

    # warm figure: layer 0's step replayed back to back (its inputs in L2), no append
    g_w = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_w, stream=stream):
        main = torch.cuda.current_stream()
        fork.record(main)
        side.wait_event(fork)
        layers[0].encode_new(kvr, pos_new, sgn, err, stream=side)
        call(layers[0], 0)
        join.record(side)
        main.wait_event(join)
    with torch.cuda.stream(stream):
        for _ in range(32):
            g_w.replay()
        w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        w0.record()
        for _ in range(256):
            g_w.replay()
        w1.record()
    stream.synchronize()
    warm_us = w0.elapsed_time(w1) * 1e3 / 256

    # end to end through the public API with pinned host buffers
    e2e = run_e2e(args, w, layers, kvr, torch, sgn, ws_s, idx, cnt, seqpos, err, scale, world,
                  e2e_n, fused)

    recall = rerank_recall(w, layers[0], kvr, torch, sgn, ws_s, seq) if rerank == "rsq" else None
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits after the timed region")

    steps_total = args.steps * world
    value = steps_total / (ms / 1000.0)
    if rank != 0:
        return
    ab = algorithmic_bytes(w.with_(N=n_mid), rerank)
    sel_key = ("select_kernel_rsq" if rerank == "rsq" else
               "select_kernel_mag" if args.votes == "magnitude" else "select_kernel")
    peak, peak_kind = peaks()
    roof = None
    # kvr_select_attend runs as one launch for groups of up to 4 heads with
    # exact rescoring and Hamming-ring votes, otherwise as the two kernels
    one_launch = w.G <= 4 and rerank == "exact" and args.votes == "hamming"
    if avg["call"]:
        if fused:
            byts = ab["select"] + ab["attend"]
            ach = byts / (avg["call"] * 1e-3) / 1e9
            if one_launch:
                kern = "select_kernel with the attention tail (kvr_select_attend, one launch)"
                traffic = measured_traffic("select_attend_kernel", w.name)
            else:
                kern = "select_kernel then attend_kernel (kvr_select_attend, two launches)"
                t_sel, t_att = measured_traffic(sel_key, w.name), measured_traffic("attend_kernel", w.name)
                traffic = None if host or None in (t_sel, t_att) else t_sel + t_att
            roof = {"bound": "hbm", "kernel": kern, "achieved": ach, "peak": peak,
                    "unit": "GB/s", "frac": ach / peak, "frac_of_8TBs": ach / 8000.0,
                    "peak_kind": peak_kind, "traffic": traffic,
                    "algorithmic_bytes": byts, "avg_ms": avg["call"]}
        else:
            ach = ab["select"] / (avg["select"] * 1e-3) / 1e9
            roof = {"bound": "hbm", "kernel": "select_kernel (kvr_select, one launch)",
                    "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                    "peak_kind": peak_kind, "traffic": measured_traffic(sel_key, w.name),
                    "algorithmic_bytes": ab["select"], "avg_ms": avg["select"]}
    path = None
    if avg["select"] and avg["attend"]:
        # the two separate calls (each timed alone), for comparison
        tsum = (avg["select"] + avg["attend"]) * 1e-3
        ach = (ab["select"] + ab["attend"]) / tsum / 1e9
        path = {"calls": "kvr_select + kvr_sparse_attend (two launches, each timed alone)",
                "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "frac_of_8TBs": ach / 8000.0, "us": tsum * 1e6,
                "algorithmic_bytes": ab["select"] + ab["attend"],
                "select_us": avg["select"] * 1e3, "attend_us": avg["attend"] * 1e3,
                "select_frac": ab["select"] / (avg["select"] * 1e-3) / 1e9 / peak,
                "traffic": (None if host or None in (measured_traffic(sel_key, w.name),
                                                     measured_traffic("attend_kernel", w.name))
                            else measured_traffic(sel_key, w.name)
                            + measured_traffic("attend_kernel", w.name))}
    link = None
    if host and avg["attend"]:
        # the attention's gathers cross the host link: its bytes over its time
        # against a page-locked host -> device copy measured on this machine
        lpk = link_peak(torch)
        ach = ab["attend"] / (avg["attend"] * 1e-3) / 1e9
        link = {"bound": "host link", "kernel": "attend_kernel (rows gathered from host memory)",
                "achieved": ach, "peak": lpk, "unit": "GB/s", "frac": ach / lpk,
                "peak_kind": "measured here: 1 GiB pinned host -> device copy, best of 5",
                "algorithmic_bytes": ab["attend"], "avg_ms": avg["attend"]}
    # the whole step against its measured time: every byte the step must read
    # (codes, candidate rows, selected K / V, query, the appended key) over
    # ms_per_step
    step_bytes = ab["select"] + ab["attend"] + ab["encode"]
    step_ach = step_bytes / (ms / args.steps * 1e-3) / 1e9
    step_roof = {"bytes": step_bytes, "achieved": step_ach, "peak": peak, "unit": "GB/s",
                 "frac": step_ach / peak, "frac_of_8TBs": step_ach / 8000.0,
                 "us": ms / args.steps * 1e3}
    timing = {"iterations_timed": timed_iters, "remainder_steps": rem,
              "median_us_per_step": statistics.median(iter_us) if iter_us else None,
              "min_us_per_step": min(iter_us) if iter_us else None,
              "max_us_per_step": max(iter_us) if iter_us else None,
              "warm_single_layer_us_per_step": warm_us,
              "warm_single_layer_steps_per_s": 1e6 / warm_us,
              "encode_us": avg["encode"] * 1e3 if avg["encode"] else None,
              "call_us": avg["call"] * 1e3 if avg["call"] else None}
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline_line(w, args.cpu_seconds, "cuda")
    cfg = dict(config_of(w), rerank=rerank, votes=args.votes,
               path=("kvr_select_attend (one launch)" if one_launch else
                     "kvr_select_attend (two launches: optional modes)") if fused else
               "kvr_select + kvr_sparse_attend (two launches)",
               appending="each step appends one token (its K / V row and code) and uses a "
                         "fresh query; lengths %d -> %d over the run"
                         % (w.N, w.N + warm_iters + timed_iters + (1 if rem else 0)))
    if host:
        cfg["kv_residency"] = "K, V in page-locked host memory read through the device mapping"
    line = {
        "metric": OFFLOAD_METRIC if host else (MILLION_METRIC if w.name == "million_token"
                                               else METRIC),
        "value": value, "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": cfg, "roofline": roof,
        "path_roofline": path, "link_roofline": link, "rerank_recall": recall,
        "step_roofline": step_roof, "timing": timing,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def link_peak(torch):
    """GB/s of a 1 GiB page-locked host -> device copy (best of 5, CUDA events)."""
    src = torch.empty(1 << 30, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(1 << 30, dtype=torch.uint8, device="cuda")
    best = None
    for _ in range(5):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1)
        best = t if best is None else min(best, t)
    del src, dst
    return (1 << 30) / (best * 1e-3) / 1e9


def rerank_recall(w, L, kvr, torch, sgn, ws_s, seq):
    """Share of the exact path's top-k that the reranked top-k keeps, over
    every unit of one layer (a quality figure, untimed)."""
    exact = kvr.SelectParams(w.C, w.k, w.W, w.lut)
    ia = torch.empty((w.B, w.Hkv, w.k), dtype=torch.int32, device=L.codes.device)
    ie = torch.empty_like(ia)
    ca = torch.empty((w.B, w.Hkv), dtype=torch.int32, device=L.codes.device)
    ce = torch.empty_like(ca)
    kvr.kvr_select(L.q, L.K, L.codes, seq, sgn, L.params, ia, ca, ws_s)
    kvr.kvr_select(L.q, L.K, L.codes, seq, sgn, exact, ie, ce, ws_s)
    a, e = ia.cpu().reshape(-1, w.k), ie.cpu().reshape(-1, w.k)
    ca, ce = ca.cpu().reshape(-1), ce.cpu().reshape(-1)
    kept = [len(set(a[u, :ca[u]].tolist()) & set(e[u, :ce[u]].tolist())) / max(1, int(ce[u]))
            for u in range(a.shape[0])]
    return {"of": "exact q_bar.k top-%d" % w.k, "mean": sum(kept) / len(kept), "min": min(kept)}


def run_e2e(args, w, layers, kvr, torch, sgn, ws_s, idx, cnt, seqpos, err, scale, world, n,
            fused):
    """End to end through the public API, appending: per step the host
    provides the step's query, the appended token's K and V rows and the new
    lengths in pinned memory; they are copied to the device, the step runs as
    one library call (kvr_decode_step: the appended key's code, selection and
    attention), the output is copied back and the host synchronises."""
    import numpy as np
    dev = layers[0].K.device
    B = w.B
    NQ = len(layers[0].qs)
    on_dev = layers[0].K.is_cuda
    hq = [[q.cpu().pin_memory() for q in L.qs] for L in layers]
    n_it = -(-n // LAYERS) + 1
    N0 = int(seqpos[0].item())   # the lengths so far: the e2e steps append after them
    # the rows these steps append, per layer, in pinned host memory
    hk = [L.K[:, :, N0:N0 + 2 * n_it].cpu().pin_memory() if on_dev else None for L in layers]
    hv = [L.V[:, :, N0:N0 + 2 * n_it].cpu().pin_memory() if on_dev else None for L in layers]
    hsp = torch.empty(2 * B, dtype=torch.int32).pin_memory()
    hout = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32).pin_memory()
    qd = [torch.empty_like(L.q) for L in layers]
    seq, pos = seqpos[:B], seqpos[B:]
    # a host-resident cache takes the appended K/V row by a host-side write
    # (the kernels read it through the mapping): only q and the lengths cross
    row_bytes = 2 * B * w.Hkv * w.d * 2 if on_dev else 0
    h2d = hq[0][0].numel() * hq[0][0].element_size() + row_bytes + hsp.numel() * 4
    d2h = hout.numel() * hout.element_size()
    steps = [kvr.DecodeStep(qd[l], L.K, L.V, L.codes, seq, pos, sgn, L.params, idx, cnt, scale,
                            L.out, ws_s, err) for l, L in enumerate(layers)]

    def host_inputs(i, base):
        """Lengths of step i (counted from `base`), in the pinned buffer."""
        it = i // LAYERS + 1
        hsp[:B] = base + it
        hsp[B:] = base + it - 1
        return it - 1

    def one(i, base, off):
        l = i % LAYERS
        L = layers[l]
        r = host_inputs(i, base)
        seqpos.copy_(hsp, non_blocking=True)
        qd[l].copy_(hq[l][(i // LAYERS) % NQ], non_blocking=True)
        if on_dev:
            L.K[:, :, base + r].copy_(hk[l][:, :, off + r], non_blocking=True)
            L.V[:, :, base + r].copy_(hv[l][:, :, off + r], non_blocking=True)
        steps[l]()
        hout.copy_(L.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    base = N0
    for i in range(min(args.warmup, 8)):
        one(i, base, 0)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n):
        one(i, base, 0)
    el = time.perf_counter() - t0
    el = max_over_ranks(el, world)
    eager = n * world / el
    res = {"value": eager, "unit": "steps/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": n,
           "mode": "kvr_decode_step per step (one C-ABI call), appending, sync per step"}
    if not on_dev:
        return res   # the appended rows are host-side writes: nothing to capture
    # the serving form: per layer one CUDA graph of the same step (one copy of
    # the step's inputs, packed in a pinned host buffer: q, the appended K / V
    # rows, the lengths and the appended position; the rows scattered into
    # the cache at that position, the decode step, the output copied back),
    # replayed and synchronised every step; the host fills the pinned buffer
    # (through numpy views, 16-bit words for bf16) before each replay
    base = N0 + n_it
    qbytes = qd[0].numel() * qd[0].element_size()
    krow_shape = (B, w.Hkv, 1, w.d)
    rbytes = B * w.Hkv * w.d * layers[0].K.element_size()

    def al16(x):
        return (x + 15) // 16 * 16
    o_k = al16(qbytes)
    o_v = o_k + al16(rbytes)
    o_s = o_v + al16(rbytes)
    o_p = o_s + al16(2 * B * 4)
    total = o_p + 8
    hst = [torch.empty(total, dtype=torch.uint8).pin_memory() for _ in layers]
    dst = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in layers]
    kdt = layers[0].K.dtype
    gstream = torch.cuda.Stream(device=dev)
    graphs = []
    for l, L in enumerate(layers):
        D = dst[l]
        dq = D[:qbytes].view(qd[l].dtype).view(qd[l].shape)
        dk = D[o_k:o_k + rbytes].view(kdt).view(krow_shape)
        dv = D[o_v:o_v + rbytes].view(kdt).view(krow_shape)
        dsp = D[o_s:o_s + 2 * B * 4].view(torch.int32)
        dp = D[o_p:o_p + 8].view(torch.int64)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            D.copy_(hst[l], non_blocking=True)
            L.K.index_copy_(2, dp, dk)
            L.V.index_copy_(2, dp, dv)
            kvr.DecodeStep(dq, L.K, L.V, L.codes, dsp[:B], dsp[B:], sgn, L.params, idx, cnt,
                           scale, L.out, ws_s, err)()
            hout.copy_(L.out, non_blocking=True)
        graphs.append(g)
    torch.cuda.synchronize()

    def words(t):
        return (t.view(torch.int16) if t.element_size() == 2 else t).numpy()
    n_q = [words(H[:qbytes].view(qd[0].dtype).view(qd[0].shape)) for H in hst]
    n_k = [words(H[o_k:o_k + rbytes].view(kdt).view(krow_shape)) for H in hst]
    n_v = [words(H[o_v:o_v + rbytes].view(kdt).view(krow_shape)) for H in hst]
    n_sp = [H[o_s:o_s + 2 * B * 4].view(torch.int32).numpy() for H in hst]
    n_p = [H[o_p:o_p + 8].view(torch.int64).numpy() for H in hst]
    n_hq = [[words(q) for q in Q] for Q in hq]
    n_hk, n_hv = [words(t) for t in hk], [words(t) for t in hv]

    def replay(i):
        l = i % LAYERS
        it = i // LAYERS + 1
        r = it - 1
        n_sp[l][:B] = base + it
        n_sp[l][B:] = base + it - 1
        n_p[l][0] = base + r
        np.copyto(n_q[l], n_hq[l][(i // LAYERS) % NQ])
        np.copyto(n_k[l], n_hk[l][:, :, n_it + r:n_it + r + 1])
        np.copyto(n_v[l], n_hv[l][:, :, n_it + r:n_it + r + 1])
        graphs[l].replay()
        torch.cuda.current_stream().synchronize()

    for i in range(min(args.warmup, 8)):
        replay(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(n):
        replay(i)
    el = max_over_ranks(time.perf_counter() - t0, world)
    res.update(value=n * world / el, eager_value=eager, h2d_bytes_per_step=total,
               mode="per step: one CUDA-graph replay (one pinned-host copy in of q, the lengths, "
                    "the position and the appended K / V rows, the rows scattered into the cache, "
                    "kvr_decode_step%s, output copied out) and a sync, appending; eager_value: "
                    "the same calls issued one by one"
                    % (" = encode + kvr_select_attend" if fused else ""))
    return res


# --------------------------------------------------------------------------
# tiered window cache workload (--workload tiered_window_cache)
# --------------------------------------------------------------------------

def tiered_bytes(w, n_bf, n_q, open_rows):
    """Algorithmic bytes of one tiered attention step: the bf16 windows' K and
    V rows, the INT2 windows' ledgers, the open window's rows and the query."""
    row = 2 * w.d
    return n_bf * 64 * 2 * row + n_q * 48 * w.d + open_rows * 2 * row + w.Hq * w.d * 2 // w.Hkv


def run_gpu_tiered(args, w):
    import numpy as np
    import torch
    import sparse_decode_attention_gb300 as kvr
    import workloads as wl

    rank, local, world = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    kvr.load()
    n_e2e = min(args.steps, 64)
    total = args.warmup + args.steps + n_e2e + 8   # every appended token fits the cache
    cap = w.N + total
    n_win = -(-cap // 64)
    U = w.B * w.Hkv
    K, V, qb = wl.make_cache(w, device=dev, cap=cap)
    closed = w.N // 64
    plan = np.zeros((U, n_win), dtype=np.int8)
    for u in range(U):
        plan[u, :closed] = wl.random_tier_plan(closed, seed=w.seed + u).numpy()
    st = kvr.TierState(U, n_win, w.d, dev)
    seq = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvr.kvr_tier_init(st, torch.from_numpy(plan).to(dev), K, V, seq, w.Hq, err)
    shape = kvr.Shape.of(K, qb)
    ws_a = kvr.workspace(kvr.kvr_tiered_attend_workspace_size(shape, n_win), dev)
    ws_u = kvr.workspace(kvr.kvr_tier_update_workspace_size(shape, n_win), dev)
    mass = torch.zeros((U, n_win), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
    stats = torch.zeros((U, 3), dtype=torch.int32, device=dev)
    NQ = 8
    qs = [wl.step_query(w, qb, t).contiguous() for t in range(NQ)]
    scale = 1.0 / math.sqrt(w.d)
    torch.cuda.synchronize()
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the tier set-up")

    def step(q, ev=None):
        # the appended token's K / V rows are already in the cache: the step
        # advances the length by one, attends, and routes
        seq.add_(1)
        if ev:
            ev[0].record()
        kvr.kvr_sparse_attend_tiered(st, q, K, V, seq, scale, out, mass, ws_a, err)
        if ev:
            ev[1].record()
        kvr.kvr_tier_update(st, mass, seq, K, V, w.Hq, stats, ws_u, err)
        if ev:
            ev[2].record()

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        step(qs[0])
        seq.sub_(1)
    stream.synchronize()
    graphs, evs = [], []
    for q in qs:
        g = torch.cuda.CUDAGraph()
        ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
        with torch.cuda.graph(g, stream=stream):
            step(q, ev)
        graphs.append(g)
        evs.append(ev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            graphs[i % NQ].replay()
    stream.synchronize()
    n0 = int(seq[0].item())
    tiers = st.tier.cpu().numpy()
    c0 = n0 // 64
    n_bf = int((tiers[:, :c0] == 0).sum()) // U
    n_q = int((tiers[:, :c0] == 1).sum()) // U

    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    per = {"attend": [], "update": []}
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record()
        for i in range(args.steps):
            graphs[i % NQ].replay()
        t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    for ev in evs:
        per["attend"].append(ev[0].elapsed_time(ev[1]))
        per["update"].append(ev[1].elapsed_time(ev[2]))
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the timed region")
    att_ms = sum(per["attend"]) / len(per["attend"])
    upd_ms = sum(per["update"]) / len(per["update"])
    st_tot = stats.sum(0).tolist()

    # end to end: query in from pinned memory, output out, synchronised per step
    n = n_e2e
    hq = [q.cpu().pin_memory() for q in qs]
    hout = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32).pin_memory()
    qd = torch.empty_like(qs[0])
    t0 = time.perf_counter()
    for i in range(n):
        qd.copy_(hq[i % NQ], non_blocking=True)
        seq.add_(1)
        kvr.kvr_sparse_attend_tiered(st, qd, K, V, seq, scale, out, mass, ws_a, err)
        kvr.kvr_tier_update(st, mass, seq, K, V, w.Hq, stats, ws_u, err)
        hout.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()
    el = max_over_ranks(time.perf_counter() - t0, world)
    e2e = {"value": n * world / el, "unit": "steps/s",
           "h2d_bytes_per_step": hq[0].numel() * hq[0].element_size(),
           "d2h_bytes_per_step": hout.numel() * hout.element_size(), "steps": n,
           "mode": "eager C-ABI calls, sync per step"}
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the end-to-end steps")
    if rank != 0:
        return
    ab = U * tiered_bytes(w, n_bf, n_q, 32)
    peak, peak_kind = peaks()
    ach = ab / (att_ms * 1e-3) / 1e9
    line = {
        "metric": "tiered decode steps/s (B4, 131072 tokens in 64-token windows)",
        "value": args.steps * world / (ms / 1000.0), "unit": "steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
                   "context": w.N, "window": 64, "initial_tiers": "25% bf16 / 50% INT2 / 25% "
                   "evicted", "windows_per_unit": closed,
                   "l2": "inputs larger than L2: each step reads %.0f MB" % (ab / 1e6)},
        "roofline": {"bound": "hbm", "kernel": "tiered_attend_kernel + tiered_combine_kernel "
                     "(kvr_sparse_attend_tiered)", "achieved": ach, "peak": peak,
                     "unit": "GB/s", "frac": ach / peak, "peak_kind": peak_kind,
                     "traffic": measured_traffic("tiered_attend_kernel", w.name),
                     "algorithmic_bytes": ab, "avg_ms": att_ms},
        "tier_update_us": upd_ms * 1e3, "windows_bf16_int2_per_unit": [n_bf, n_q],
        "moves_last_step": {"promotions": st_tot[0], "demotions": st_tot[1],
                            "evictions": st_tot[2]},
        "cpu_baseline": None, "e2e": e2e, "gpu_launches": 4 * args.steps, "clocks": clk,
    }
    if args.diagnostics:
        del K, V, st
        torch.cuda.empty_cache()
        line["cache_dynamics"] = tiered_dynamics(w, args.diagnostics, dev)
    print(json.dumps(line), flush=True)


def tiered_dynamics(w, steps, dev):
    """Untimed: Future Missed Mass, Global LIR and selection churn of the
    routing policy over `steps` appending steps with fresh queries. The
    full-attention window masses come from the tiered attention over an
    all-bf16 state and an unmodified copy of the cache."""
    import numpy as np
    import torch
    import sparse_decode_attention_gb300 as kvr
    import workloads as wl
    import bench_diagnostics as dg

    cap = w.N + steps + 8
    n_win = -(-cap // 64)
    U = w.B * w.Hkv
    K, V, qb = wl.make_cache(w, device=dev, cap=cap)
    K0, V0 = K.clone(), V.clone()
    closed = w.N // 64
    plan = np.zeros((U, n_win), dtype=np.int8)
    for u in range(U):
        plan[u, :closed] = wl.random_tier_plan(closed, seed=w.seed + u).numpy()
    seq = torch.full((w.B,), w.N, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = kvr.TierState(U, n_win, w.d, dev)
    kvr.kvr_tier_init(st, torch.from_numpy(plan).to(dev), K, V, seq, w.Hq, err)
    dense = dg.full_mass_state(U, n_win, w.d, K0, V0, seq, w.Hq, err)
    shape = kvr.Shape.of(K, qb)
    ws_a = kvr.workspace(kvr.kvr_tiered_attend_workspace_size(shape, n_win), dev)
    ws_u = kvr.workspace(kvr.kvr_tier_update_workspace_size(shape, n_win), dev)
    mass = torch.zeros((U, n_win), dtype=torch.float32, device=dev)
    full = torch.zeros((U, n_win), dtype=torch.float32, device=dev)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
    stats = torch.zeros((U, 3), dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(w.d)
    dyn = dg.CacheDynamics()
    for t in range(steps):
        seq.add_(1)
        q = wl.step_query(w, qb, 1000 + t).contiguous()
        kvr.kvr_sparse_attend_tiered(dense, q, K0, V0, seq, scale, out, full, ws_a, err)
        before = st.tier.clone()
        kvr.kvr_sparse_attend_tiered(st, q, K, V, seq, scale, out, mass, ws_a, err)
        kvr.kvr_tier_update(st, mass, seq, K, V, w.Hq, stats, ws_u, err)
        dyn.record(full, before, st.tier, w.N + t + 1)
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the diagnostics pass")
    res = dyn.summary()
    res["definitions"] = ("FMM: full-attention mass on evicted windows / total, per step and "
                          "unit; LIR: active-set leaves later reactivated / leaves; churn: "
                          "|A_t xor A_t-1| / |A_t-1|; active = bf16 closed windows")
    return res


# --------------------------------------------------------------------------
# batched drift workload (--workload batched_drift)
# --------------------------------------------------------------------------

def run_gpu_drift(args, w):
    """B 8 units x 8 kv heads, 32768 prefill tokens, then w.steps appending
    steps whose keys and queries drift. An untimed pass measures the recall of
    every step's top-k against the fp64 top-k of q_bar . k over the pool; the
    timed pass replays one CUDA graph per step with the step counters on the
    device (query row, encode position, sequence length)."""
    import torch
    import sparse_decode_attention_gb300 as kvr
    import workloads as wl

    rank, local, world = dist_setup(args)
    dev = torch.device("cuda", torch.cuda.current_device())
    kvr.load()
    T, N0 = w.steps, w.N
    K, V, qb = wl.make_cache(w, device=dev, cap=N0 + T)
    k_new, qs = wl.drift_inputs(w, K, N0, T)
    K[:, :, N0:N0 + T] = k_new
    del k_new
    sgn = wl.srht_signs(w.d, device=dev)
    shape = kvr.Shape.of(K, qb)
    vflags = kvr.SELECT_MAGNITUDE_VOTES if args.votes == "magnitude" else 0
    regions = None
    if args.regions:
        # Sink / Local / Update buffer sizes in tokens (cache regions)
        regions = tuple(int(x) for x in args.regions.split(","))
        S_r, L_r, U_r = regions
        rend = torch.zeros(w.B, dtype=torch.int32, device=dev)
        params = kvr.SelectParams(w.C, w.k, 0, w.lut, V_prefetch=V, sink=S_r, region_end=rend,
                                  flags=vflags)
    else:
        params = kvr.SelectParams(w.C, w.k, w.W, w.lut, V_prefetch=V, flags=vflags)
    ws_s = kvr.workspace(kvr.kvr_select_workspace_size(shape, params), dev)
    ws_a = kvr.workspace(kvr.kvr_attend_workspace_size(shape, w.k, w.W), dev)
    codes = kvr.codes_buffer(shape, dev)
    idx = torch.empty((w.B, w.Hkv, w.k), dtype=torch.int32, device=dev)
    cnt = torch.empty((w.B, w.Hkv), dtype=torch.int32, device=dev)
    out = torch.empty((w.B, w.Hq, w.d), dtype=torch.float32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    zero = torch.zeros(w.B, dtype=torch.int32, device=dev)
    kvr.kvr_encode_keys(K, zero, N0, sgn, codes, err)
    scale = 1.0 / math.sqrt(w.d)
    pos = torch.empty(w.B, dtype=torch.int32, device=dev)
    seq = torch.empty(w.B, dtype=torch.int32, device=dev)
    tt = torch.zeros(1, dtype=torch.int64, device=dev)
    q = torch.empty_like(qs[0])

    def reset():
        pos.fill_(N0)
        if regions:
            seq.fill_(N0)
            kvr.kvr_regions_update(seq, S_r, L_r, U_r, rend, init=True, err=err)
        seq.fill_(N0 + 1)
        tt.zero_()

    def step(ev=None):
        torch.index_select(qs, 0, tt, out=q.view(1, *q.shape))
        if ev:
            ev[0].record()
        kvr.kvr_encode_keys(K, pos, 1, sgn, codes, err)
        if regions:
            kvr.kvr_regions_update(seq, S_r, L_r, U_r, rend, err=err)
        if ev:
            ev[1].record()
        kvr.kvr_select(q, K, codes, seq, sgn, params, idx, cnt, ws_s, err)
        if ev:
            ev[2].record()
        if regions:
            kvr.kvr_sparse_attend_regions(q, K, V, idx, cnt, seq, S_r, rend, scale, out, ws_a, err)
        else:
            kvr.kvr_sparse_attend(q, K, V, idx, cnt, seq, w.W, scale, out, ws_a, err)
        if ev:
            ev[3].record()
        pos.add_(1)
        seq.add_(1)
        tt.add_(1)

    # recall pass (untimed): fp64 exact scores of the pool against q_bar
    K64 = K.double()
    G = w.G
    recall = []
    reset()
    for t in range(T):
        step()
        N = N0 + t + 1
        p0, pool = 0, N - w.W
        if regions:
            p0, pool = min(S_r, N), int(rend[0])
        kk = min(w.k, min(w.C, pool - p0))
        qbar = qs[t].double().view(w.B, w.Hkv, G, w.d).mean(2)
        S = torch.einsum("bhnd,bhd->bhn", K64[:, :, p0:pool], qbar)
        top = torch.topk(S, kk, dim=-1).indices + p0
        got = idx[:, :, :kk].long()
        hit = (torch.sort(got, -1).values.unsqueeze(-1) ==
               torch.sort(top, -1).values.unsqueeze(-2)).any(-1).sum(-1)
        recall.append((hit.double() / kk).mean().item())
    del K64
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits in the recall pass")

    stream = torch.cuda.Stream(device=dev)
    reset()
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    with torch.cuda.graph(g, stream=stream):
        step(ev)
    torch.cuda.synchronize()
    reset()
    with torch.cuda.stream(stream):
        for _ in range(min(args.warmup, T)):
            g.replay()
    stream.synchronize()
    reset()
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.25 if clocks else 0)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record()
        for _ in range(T):
            g.replay()
        t_end.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(t_start.elapsed_time(t_end), world)
    if kvr.kvr_read_error(err):
        raise RuntimeError("device error bits during the timed region")
    sel_ms, att_ms = ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])
    if rank != 0:
        return
    wl_mid = w.with_(N=N0 + T // 2)
    ab = algorithmic_bytes(wl_mid)
    peak, peak_kind = peaks()
    ach = ab["select"] / (sel_ms * 1e-3) / 1e9
    r = recall
    line = {
        "metric": "batched drift decode steps/s (B8, 32768 prefill + %d appending steps) and "
                  "exact-top-k recall per step" % T
                  + (", sink / local / update-buffer regions" if regions else "")
                  + (", magnitude-aware votes" if vflags else ""),
        "value": T * world / (ms / 1000.0), "unit": "steps/s", "n_gpus": world, "steps": T,
        "warmup": args.warmup, "ms_per_step": ms / T, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "head_dim": w.d,
                   "prefill": N0, "appending_steps": T, "C": w.C, "k": w.k, "W": w.W,
                   "votes": args.votes,
                   "regions": None if not regions else
                   {"sink": regions[0], "local": regions[1], "buffer": regions[2]},
                   "l2": "inputs larger than L2: each step reads %.0f MB"
                         % ((ab["select"] + ab["attend"]) / 1e6)},
        "recall": {"mean": sum(r) / len(r), "min": min(r), "first_step": r[0],
                   "last_step": r[-1], "mean_first_512": sum(r[:512]) / len(r[:512]),
                   "mean_last_512": sum(r[-512:]) / len(r[-512:]),
                   "reference": "fp64 top-k of q_bar . k over the pool, per step and unit"},
        "roofline": {"bound": "hbm", "kernel": "select_kernel (kvr_select, one launch)",
                     "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                     "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes": ab["select"], "avg_ms": sel_ms},
        "attend_us": att_ms * 1e3, "cpu_baseline": None, "e2e": None,
        "gpu_launches": (3 + (1 if regions else 0) + (1 if vflags else 0)) * T, "clocks": clk,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["kvr", "reference"], default="kvr")
    ap.add_argument("--e2e-steps", type=int, default=2000)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=LAYERS,
                    help="layer caches rotated (fewer = a small case for profiling; the "
                         "default keeps every step's inputs cold in L2)")
    ap.add_argument("--workload", choices=["llama3_8b_128k", "million_token", "tiered_window_cache",
                                           "batched_drift", "million_offload"],
                    default="llama3_8b_128k",
                    help="the timed workload (the 128K decode layer is the headline)")
    ap.add_argument("--path", choices=["fused", "separate"], default="fused",
                    help="selection and attention as one call (kvr_select_attend: one launch "
                         "where it fuses them) or as kvr_select + kvr_sparse_attend")
    ap.add_argument("--diagnostics", type=int, default=0, metavar="STEPS",
                    help="tiered_window_cache only: also run STEPS untimed appending steps and "
                         "report Future Missed Mass, Global LIR and selection churn")
    ap.add_argument("--votes", choices=["hamming", "magnitude"], default="hamming",
                    help="coarse votes: Hamming rings of the query code (default) or centroids "
                         "ranked by the rotated query's magnitudes")
    ap.add_argument("--regions", default=None, metavar="S,L,U",
                    help="batched_drift only: sink, local and update-buffer sizes (tokens); "
                         "selection over the retrieval region, attention over sink + top-k + "
                         "local and buffer")
    ap.add_argument("--rerank", choices=["exact", "rsq"], default=None,
                    help="candidate ranking: exact q_bar.k from the K rows (default for "
                         "device caches), or the calibrated estimate from per-key records "
                         "(default for million_offload)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    globals()["LAYERS"] = max(1, args.layers)
    import workloads as wl
    if args.workload == "tiered_window_cache":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the tiered workload has no "
                              "reference line; the oracle arm covers the 128K workload"}))
            return
        run_gpu_tiered(args, wl.TIERED)
        return
    if args.workload == "batched_drift":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the drift workload has no "
                              "reference line; the oracle arm covers the 128K workload"}))
            return
        run_gpu_drift(args, wl.DRIFT)
        return
    if args.workload == "million_offload":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the host-resident workload "
                              "has no reference line; the oracle arm covers the 128K workload"}))
            return
        # two layers of 2^20 tokens: 8.6 GB of page-locked host cache, and the
        # device-side codes and records (2 x 0.94 GB) exceed L2
        if args.layers == LAYERS_DEFAULT:
            globals()["LAYERS"] = 2
        run_gpu(args, wl.MILLION)
        return
    if args.workload == "million_token":
        # 2^20 tokens with K / V in HBM: 8 layers (34.6 GB; codes alone 1.07 GB,
        # every step's inputs cold in L2)
        if args.layers == LAYERS_DEFAULT:
            globals()["LAYERS"] = 8
        w = wl.MILLION
        if args.impl == "reference":
            run_reference(args, w)
        else:
            run_gpu(args, w)
        return
    w = wl.LLAMA_128K
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_gpu(args, w)


if __name__ == "__main__":
    main()
