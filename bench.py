"""Benchmark of the KV retention hot path on GB300.

One step = one pass of the whole path on one session:
  IntentKV token step (8B-shaped: L36 Hq32 Hkv8 D128, N=32768 tokens, bf16 K in
  16-slot shuffled pages): QueryMemory update with the turn's 256 query rows,
  rule scores over all candidates, top-C* retention (C=8192), dead-slot redirect;
  KVMEM block step (1M-token workspace: L64 Hq40 Hkv8 D128, 32768 Mean-K blocks):
  incremental Mean-K build of 4096 new tokens, R_b over all candidate blocks for
  2048 query tokens, sink 4 + recent 128 + top-2048 working set, re-RoPE scatter
  of the 65,536 staged tokens into a shuffled page pool.

Metric: KV rows scored per second = (L*Hkv*|H| token rows + L*Hkv*|C| index
rows) per step / step time.  With --gpus N (torchrun, one rank per GPU) every
rank runs its own session (replicas, weak scaling, no collective on the data
path); the value is the rows of all ranks over the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

TOKEN_WL = "8b"
BLOCK_WL = "ws1m"


def aggregate(ms_local, rows_per_step, steps, dist=None, device=None):
    """Whole-job throughput of replicas: every rank ran `steps` steps of
    `rows_per_step` rows; the job takes as long as its slowest rank.
    Returns (rows/s over all ranks, max ms over ranks)."""
    import torch
    t = torch.tensor([float(ms_local)], dtype=torch.float64, device=device)
    world = 1
    if dist is not None and dist.is_initialized():
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        world = dist.get_world_size()
    ms_max = float(t.item())
    return world * rows_per_step * steps / (ms_max / 1e3), ms_max


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "src": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def workload_rows(tw, bw):
    token_rows = tw.L * tw.Hkv * tw.n_cand
    block_rows = bw.L * bw.Hkv * bw.n_cand
    return token_rows, block_rows


def config_dict(tw, bw, n):
    return {"workload": f"IntentKV token step [{tw.name}] + KVMEM block step [{bw.name}]",
            "token": {"L": tw.L, "Hq": tw.Hq, "Hkv": tw.Hkv, "D": tw.D, "N": tw.N, "C": tw.C, "pi": tw.pi,
                      "span": tw.span, "page": tw.page, "query_rows": tw.R},
            "block": {"L": bw.L, "Hq": bw.Hq, "Hkv": bw.Hkv, "D": bw.D, "blocks": bw.n_blocks, "block": bw.block,
                      "M": bw.M, "sink": bw.n_sink, "recent": bw.n_recent, "k": bw.k, "new_tokens": bw.new_tokens,
                      "staged_tokens": min(bw.k, bw.n_cand) * bw.block},
            "l2": "inputs larger than L2 (K pool 2.4 GB, index 4.3 GB, staging 8.6 GB); no flush",
            "parallelism": f"replicas x{n} (independent sessions, no collective)"}


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"kvsel_clocks_{os.getpid()}_{gpu_index}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for name, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(name)
            os.unlink(self.path)
        except Exception:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def setup_session(kv, synth, ctx, tw, bw, torch):
    """Device-resident state and per-step inputs of one session."""
    t = synth.token_inputs(tw, "cuda")
    b = synth.block_inputs(bw, "cuda")
    s = {"tw": tw, "bw": bw, "pool": t["pool"], "slot_map": t["slot_map"], "turns": t["turns"],
         "q_last": t["turns"][tw.turns - 1].contiguous(),
         "M": torch.zeros((tw.L, tw.Hq, tw.D), device="cuda"),
         "rule": torch.empty(tw.N, device="cuda"),
         "keep": torch.empty(tw.N, device="cuda", dtype=torch.uint8),
         "keep_idx": torch.empty(tw.N, device="cuda", dtype=torch.int32),
         "slot_out": torch.empty(tw.N, device="cuda", dtype=torch.int32),
         "raw_new": b["raw"], "index": b["index"], "q": b["q"], "staging": b["staging"], "kpool": b["pool"],
         "R": torch.empty(bw.n_blocks, device="cuda"),
         "ids": torch.empty(bw.n_sel, device="cuda", dtype=torch.int32)}
    # the session's earlier turns (state before the timed turn)
    for i in range(tw.turns - 1):
        ctx.memory_update(t["turns"][i], tw.lam, s["M"], first_turn=(i == 0))
    s["src_block"], s["dst_page"], s["dst_pos0"] = synth.scatter_plan_incremental(bw, b["page_perm"])
    return s


# kernel launches per C-ABI call (counted from the launchers in csrc/)
LAUNCHES = {"memory_update": 1, "rule_scores": 3, "topk_retain": 1, "redirect_slots": 1, "meank_build": 1,
            "block_scores": 4, "select_blocks": 1, "rerope_scatter": 1}


# Highest fraction of the peak a call's algorithm allows: R_b computes every logit twice on the
# tensor cores (once for each row's total, once for the block masses) against the one contraction
# counted as algorithmic flops.
ALGORITHMIC_CEILING = {"block_scores": 0.5}


# the step input each call reads first (end-to-end leg: the call waits for that input's copy only)
INPUT_OF = {"memory_update": "q_last", "meank_build": "raw_new", "block_scores": "q", "rerope_scatter": "staging"}


def run_step(ctx, s, ev=None, ready=None):
    """One pass of the whole path; ev: optional dict name -> list of (start, end) events;
    ready: optional dict input name -> CUDA event recorded when that input's copy has landed."""
    tw, bw = s["tw"], s["bw"]

    def mark(name, fn):
        if ready is not None and name in INPUT_OF:
            import torch
            torch.cuda.current_stream().wait_event(ready[INPUT_OF[name]])
        if ev is None:
            fn()
            return
        import torch
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ev.setdefault(name, []).append((a, b))

    mark("memory_update", lambda: ctx.memory_update(s["q_last"], tw.lam, s["M"]))
    mark("rule_scores", lambda: ctx.rule_scores(s["pool"], s["M"], tw.L, tw.Hq, tw.Hkv, tw.N, tw.D, tw.pi, tw.q_s,
                                                tw.q_e, s["rule"], slot_map=s["slot_map"], n_slots=tw.N))
    mark("topk_retain", lambda: ctx.topk_retain(s["rule"], tw.pi, tw.q_s, tw.q_e, tw.C, keep=s["keep"],
                                                keep_idx=s["keep_idx"]))
    mark("redirect_slots", lambda: ctx.redirect_slots(s["slot_map"], s["keep"], tw.dead_slot, s["slot_out"]))
    mark("meank_build", lambda: ctx.meank_build(s["raw_new"], bw.block, s["index"], first_block=bw.first_new_block))
    mark("block_scores", lambda: ctx.block_scores(s["q"], s["index"], bw.n_blocks, bw.n_sink, bw.n_recent, s["R"]))
    mark("select_blocks", lambda: ctx.select_blocks(s["R"], bw.n_sink, bw.n_recent, bw.k, s["ids"]))
    mark("rerope_scatter", lambda: ctx.rerope_scatter(s["staging"], s["src_block"], s["dst_page"], s["dst_pos0"],
                                                      s["kpool"], bw.rope_base))


def kernel_algorithmic(tw, bw):
    """Algorithmic bytes (HBM kernels) or flops (tensor kernel) per call."""
    n_top = min(bw.k, bw.n_cand)
    return {
        "rule_scores": ("hbm", tw.L * tw.n_cand * tw.Hkv * tw.D * 2 + tw.N * 4),
        "memory_update": ("hbm", tw.L * tw.Hq * tw.R * tw.D * 2 + 2 * tw.L * tw.Hq * tw.D * 4),
        "meank_build": ("hbm", bw.L * bw.Hkv * bw.new_tokens * bw.D * 2 + bw.L * bw.Hkv * (bw.new_tokens // bw.block) * bw.D * 2),
        "rerope_scatter": ("hbm", 2 * bw.L * bw.Hkv * n_top * bw.block * bw.D * 2),
        "block_scores": ("tensor", 2 * bw.L * bw.Hq * bw.M * bw.n_cand * bw.D),
    }


def ours(args, rank, world, local_rank):
    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    tw, bw = synth.TOKEN[TOKEN_WL], synth.BLOCK[BLOCK_WL]
    ctx = kv.Context(local_rank)
    s = setup_session(kv, synth, ctx, tw, bw, torch)
    torch.cuda.synchronize()

    def barrier():
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        run_step(ctx, s)
    ctx.check_device()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev = {}
    start.record()
    for _ in range(args.steps):
        run_step(ctx, s, ev)
    end.record()
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms_total = start.elapsed_time(end)
    per_call = {k: sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in ev.items()}
    ctx.check_device()

    # end-to-end: fresh per-step inputs from pinned host memory, results back to the host.  The inputs are
    # double-buffered on the device and copied on a second stream, so step t+1's inputs move while step t
    # computes, and each call waits only for the input it reads; every copy and every step lies inside the
    # timed region.
    in_keys = ("q_last", "raw_new", "q", "staging")
    h_in = {k: s[k].detach().cpu().pin_memory() for k in in_keys}
    h_out = {k: torch.empty_like(s[k], device="cpu").pin_memory() for k in ("rule", "slot_out", "keep_idx", "R", "ids")}
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())
    sets = [s, dict(s)]
    for k in in_keys:
        sets[1][k] = torch.empty_like(s[k])
    copy_stream = torch.cuda.Stream()
    compute_stream = torch.cuda.current_stream()
    # one event per input and buffer set: a step's kernels start as soon as the input they read
    # has landed (the small query copies first; the 8.6 GB staging copy overlaps R_b)
    ev_copied = [{k: torch.cuda.Event() for k in in_keys} for _ in range(2)]
    ev_done = [torch.cuda.Event(), torch.cuda.Event()]

    def issue_copy(i, spans=None):
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(ev_done[i % 2])  # step i-2 is done with this buffer set
            if spans is not None:
                spans.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                spans[-1][0].record(copy_stream)
            for k in in_keys:
                sets[i % 2][k].copy_(h_in[k], non_blocking=True)
                ev_copied[i % 2][k].record(copy_stream)
            if spans is not None:
                spans[-1][1].record(copy_stream)

    def e2e_run(n, start_event=None, spans=None):
        if start_event is not None:
            copy_stream.wait_event(start_event)
        issue_copy(0, spans)
        for i in range(n):
            if i + 1 < n:
                issue_copy(i + 1, spans)
            run_step(ctx, sets[i % 2], ready=ev_copied[i % 2])
            ev_done[i % 2].record(compute_stream)
            for k, t in h_out.items():
                t.copy_(sets[i % 2][k], non_blocking=True)

    e2e_steps = max(1, args.steps)
    e2e_run(max(2, min(args.warmup, 3)))
    torch.cuda.synchronize()
    barrier()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record()
    copy_spans = []  # each step's input copies, start to end on the copy stream (the link rate under load)
    e2e_run(e2e_steps, e_start, copy_spans)
    e_end.record()
    torch.cuda.synchronize()
    barrier()
    h2d_in_e2e_ms = sum(a.elapsed_time(b) for a, b in copy_spans) / len(copy_spans)
    # the same per-step input copies alone (no kernels), for reading the e2e figure:
    # when they take longer than the device step, e2e is bound by the host link
    c_start, c_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(copy_stream):
        c_start.record(copy_stream)
        for i in range(2):
            for k in in_keys:
                sets[i % 2][k].copy_(h_in[k], non_blocking=True)
        c_end.record(copy_stream)
    torch.cuda.synchronize()
    h2d_alone_ms = c_start.elapsed_time(c_end) / 2
    token_rows, block_rows = workload_rows(tw, bw)
    rows_step = token_rows + block_rows
    value, ms_max = aggregate(ms_total, rows_step, args.steps, dist, "cuda")
    e2e_value, e2e_ms_max = aggregate(e_start.elapsed_time(e_end), rows_step, e2e_steps, dist, "cuda")

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peaks = _peaks()
    alg = kernel_algorithmic(tw, bw)
    kernels = {}
    for name, (bound, amount) in alg.items():
        ms = per_call.get(name)
        if not ms:
            continue
        if bound == "hbm":
            ach = amount / (ms / 1e3) / 1e9
            kernels[name] = {"bound": "hbm", "ms": ms, "achieved": ach, "unit": "GB/s", "peak": peaks["hbm_gbs"],
                             "frac": ach / peaks["hbm_gbs"], "algorithmic_bytes": amount}
        else:
            ach = amount / (ms / 1e3) / 1e12
            kernels[name] = {"bound": "tensor", "ms": ms, "achieved": ach, "unit": "TFLOP/s",
                             "peak": peaks["bf16_tflops_sustained"], "frac": ach / peaks["bf16_tflops_sustained"],
                             "algorithmic_flops": amount}
    for name in ("topk_retain", "redirect_slots", "select_blocks"):
        if name in per_call:
            kernels[name] = {"bound": "latency", "ms": per_call[name]}
    if "block_scores" in kernels:  # (query token x candidate block) pairs scored, over all layer-heads
        kernels["block_scores"]["pairs_per_s"] = bw.L * bw.Hq * bw.M * bw.n_cand / (kernels["block_scores"]["ms"] / 1e3)
    dom = max((k for k in kernels if "achieved" in kernels[k]), key=lambda k: kernels[k]["ms"])
    d = kernels[dom]
    traffic = _profiled_traffic(dom)
    ceiling = ALGORITHMIC_CEILING.get(dom, 1.0)
    roofline = {"kernel": dom, "bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
                "frac": d["frac"], "ceiling": ceiling, "frac_of_ceiling": d["frac"] / ceiling, "traffic": traffic,
                "peak_src": f"{peaks['src']} ({'bf16_tflops_sustained' if d['bound'] == 'tensor' else 'hbm_gbs'})"}
    cpu = cpu_baseline(args, tw, bw) if not args.no_cpu_baseline else None
    line = {
        "metric": "KV rows scored/s", "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "us_per_select_step": 1e3 * ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' workloads)", "config": config_dict(tw, bw, world),
        "rows_per_step": {"token": token_rows, "block": block_rows},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": e2e_ms_max / e2e_steps,
                "h2d_alone_ms_per_step": h2d_alone_ms, "h2d_alone_gbs": h2d / (h2d_alone_ms / 1e3) / 1e9,
                "h2d_during_ms_per_step": h2d_in_e2e_ms, "h2d_during_gbs": h2d / (h2d_in_e2e_ms / 1e3) / 1e9,
                "inputs": "per-step query rows, new raw K and staged top-block K from pinned host, double-buffered "
                          "and copied on a second stream with one event per input (each call waits for the input "
                          "it reads; step t+1's inputs move while step t computes); K pool and Mean-K index "
                          "resident on the device"},
        "gpu_launches": sum(LAUNCHES.values()) * args.steps,
        "roofline": roofline, "kernels": kernels, "clocks": clk, "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# DRAM bytes (read + write) per call from an ncu capture of the current kernel code, scaled to the
# bench workload; an entry is removed whenever its kernel changes.
PROFILED_TRAFFIC = {
    # block_scores_tc, 4-layer capture of the three tensor-core launches (row pass 352.0 + 4.7 MB,
    # exact pass 0.06 + 0 MB, column pass 353.8 + 6.9 MB), x16 for 64 layers:
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,... -k regex:block_scores_tc -c 3
    # on python bench.py --profile-kernel block_scores --profile-layers 4 --steps 3 --warmup 1
    "block_scores": 16 * (351.990016 + 4.710912 + 0.063488 + 353.807360 + 6.911232) * 1e6,
}


def _profiled_traffic(kernel):
    return PROFILED_TRAFFIC.get(kernel)


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the fp64 oracle, timed on the host cores
# ---------------------------------------------------------------------------

BLOCK_SLICE_QUERIES = 64  # query tokens per (layer, kv head) in the timed slice of the block step


def _oracle_worker(conn, root):
    """A host process running the unchanged oracle on a fixed slice of the step.

    ("load", tw, bw, token_slices, block_jobs): keep this worker's (layer, kv head)
    slices of the token step's K pool ([N][D] rows of one kv head) and its block-step
    jobs (q [1][G][m][D], index [1][1][B][D] bf16 bits).
    ("rules", M_slices): the sum of the rule-score contributions of its slices, in
    slice order (fp64 [N]).  ("block",): run its block-step jobs.  ("stop",): exit."""
    sys.path.insert(0, root)
    import numpy as np

    import oracle
    oracle.build()
    tw = bw = None
    slices, jobs, slot_map = [], [], None
    while True:
        msg = conn.recv()
        if msg[0] == "stop":
            break
        if msg[0] == "load":
            _, tw, bw, slot_map, slices, jobs = msg
            conn.send("ok")
        elif msg[0] == "rules":
            G = tw.Hq // tw.Hkv
            acc = np.zeros(tw.N)
            for k, Mlg in zip(slices, msg[1]):
                acc += oracle.rule_scores(k.ravel(), Mlg.reshape(1, G, tw.D), 1, G, 1, tw.N, tw.D, tw.pi, tw.q_s,
                                          tw.q_e, slot_map=slot_map, layer_stride=tw.N * tw.D, slot_stride=tw.D)
            conn.send(acc)
        elif msg[0] == "block":
            for q, ix in jobs:
                oracle.block_mass(q, ix, bw.n_blocks, bw.n_sink, bw.n_recent, 0, 0)
            conn.send("ok")
    conn.close()


class OracleStep:
    """The oracle's select step on the host cores, run as `procs` processes.

    Token part (IntentKV, the whole step, measured): QueryMemory update of the timed
    turn, rule scores of every (layer, kv head) (the unchanged oracle on disjoint
    (layer, kv head) slices, one fixed share per process, partial rule vectors added
    in a fixed order), top-C*, redirect.
    Block part (KVMEM R_b, a declared slice): one (layer, kv head) mass row per
    process with BLOCK_SLICE_QUERIES query tokens and every candidate block; its wall
    time over its work fraction estimates the whole block part at the same process
    count (the (layer, kv head) rows are independent).
    Inputs are drawn on the host with the workloads' shapes (the oracle shares no
    state with the GPU path); drawing and loading them is outside the timing."""

    def __init__(self, tw, bw, procs=None):
        import multiprocessing as mp

        import numpy as np
        import torch

        import oracle
        import synth
        oracle.build()
        self.tw, self.bw = tw, bw
        self.procs = procs or max(1, min(16, os.cpu_count() or 1))
        P, G = self.procs, tw.Hq // tw.Hkv
        ti = synth.token_inputs(tw, "cpu")
        bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
        pool = bits(ti["pool"])                                   # [L][N][Hkv][D]
        self.slot_map = ti["slot_map"].numpy()
        self.q_last = bits(ti["turns"][tw.turns - 1])
        M = None
        for t in range(tw.turns - 1):  # the session's earlier turns (state before the timed turn)
            M, _ = oracle.memory_update(bits(ti["turns"][t]), tw.lam, M=M, first_turn=(t == 0))
        self.M_prev = M
        self.pairs = [[(l, g) for i, (l, g) in enumerate((l, g) for l in range(tw.L) for g in range(tw.Hkv))
                       if i % P == r] for r in range(P)]
        bstd = (bw.offset_sigma ** 2 + 1.0 / bw.block) ** 0.5
        mp_ctx = mp.get_context("spawn")
        self.workers = []
        for r in range(P):
            a, b = mp_ctx.Pipe()
            proc = mp_ctx.Process(target=_oracle_worker, args=(b, ROOT), daemon=True)
            proc.start()
            l, g = (r * 37) % bw.L, r % bw.Hkv
            q = synth.bf16_bits(synth.portable_normal((1, bw.Hq // bw.Hkv, BLOCK_SLICE_QUERIES, bw.D),
                                                      (bw.seed, synth.PORTABLE_Q, l, g)))
            ix = synth.bf16_bits(synth.portable_normal((1, 1, bw.n_blocks, bw.D), (bw.seed, synth.PORTABLE_INDEX, l, g),
                                                       bstd))
            a.send(("load", tw, bw, self.slot_map, [np.ascontiguousarray(pool[l_, :, g_, :]) for l_, g_ in self.pairs[r]],
                    [(q, ix)]))
            self.workers.append((proc, a))
        del ti, pool
        for _, a in self.workers:
            assert a.recv() == "ok"
        self.G = G
        self.frac_block = P * BLOCK_SLICE_QUERIES / (bw.L * bw.Hkv * bw.M)

    def close(self):
        for proc, a in self.workers:
            try:
                a.send(("stop",))
            except Exception:
                pass
        for proc, _ in self.workers:
            proc.join(timeout=30)

    def step(self):
        """One sample step; returns (token step s, block slice wall s)."""
        import numpy as np

        import oracle
        tw, G = self.tw, self.G
        t0 = time.perf_counter()
        M, _ = oracle.memory_update(self.q_last, tw.lam, M=self.M_prev)
        for r, (_, a) in enumerate(self.workers):
            a.send(("rules", [M[l, g * G:(g + 1) * G] for l, g in self.pairs[r]]))
        rule = np.zeros(tw.N)
        for _, a in self.workers:
            rule += a.recv()
        keep, _ = oracle.topk_retain(rule, tw.pi, tw.q_s, tw.q_e, tw.C)
        oracle.redirect_slots(self.slot_map, keep, tw.dead_slot)
        t1 = time.perf_counter()
        for _, a in self.workers:
            a.send(("block",))
        for _, a in self.workers:
            assert a.recv() == "ok"
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1

    def figures(self, t_tok, t_blk):
        """The baseline's fields from the measured parts (medians over steps)."""
        tw, bw = self.tw, self.bw
        token_rows, block_rows = workload_rows(tw, bw)
        est = t_tok + t_blk / self.frac_block
        desc = (f"oracle (fp64 C) on {self.procs} processes: whole token step ({t_tok:.2f} s measured; rule scores "
                f"over {tw.L * tw.Hkv} (layer, kv head) slices); R_b slice of {self.procs} of {bw.L * bw.Hkv} "
                f"(layer, kv head) rows x {BLOCK_SLICE_QUERIES} of {bw.M} query tokens ({t_blk:.2f} s measured, "
                f"work fraction {self.frac_block:.3g}); full step estimated {est:.0f} s")
        return {"value": (token_rows + block_rows) / est, "unit": "rows/s", "cores": self.procs, "kind": "oracle",
                "sample": desc, "measured_s": t_tok + t_blk, "extrapolated": True, "est_full_step_s": est,
                "token_step": {"measured_s": t_tok, "rows": token_rows, "procs": self.procs, "work_fraction": 1.0,
                               "extrapolated": False},
                "block_step": {"measured_s": t_blk, "rows": block_rows, "procs": self.procs,
                               "work_fraction": self.frac_block, "extrapolated": True,
                               "slice": f"{self.procs} (layer, kv head) rows x {BLOCK_SLICE_QUERIES} query tokens, "
                                        f"all {bw.n_blocks} blocks"},
                "nproc": os.cpu_count(), "host": host_cpu()}


def host_cpu():
    """The host's CPU model (x86: the model name; Arm: implementer and part from MIDR) and core count."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for line in info.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
        if not model:
            imp = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU implementer")]
            part = [ln.split(":", 1)[1].strip() for ln in info.splitlines() if ln.startswith("CPU part")]
            if imp and part:
                model = f"arm implementer {imp[0]} part {part[0]}"
    except OSError:
        pass
    import platform
    return {"model": model or platform.machine(), "nproc": os.cpu_count()}


def cpu_baseline(args, tw, bw):
    """The oracle on the host cores: one sample step (rank 0, N=1)."""
    o = OracleStep(tw, bw)
    try:
        t_tok, t_blk = o.step()
        return o.figures(t_tok, t_blk)
    finally:
        o.close()


def reference(args, rank, world):
    """The reference arm: the fp64 oracle, each step one sample step of the workload
    (the whole token step and a slice of the block step, OracleStep).  ms_per_step is
    the measured time of a sample step; value is the whole step's rows over the
    estimated whole-step time (fields say which parts are measured and which scaled)."""
    if rank != 0:
        return
    import synth
    tw, bw = synth.TOKEN[TOKEN_WL], synth.BLOCK[BLOCK_WL]
    o = OracleStep(tw, bw)
    try:
        for _ in range(args.warmup):
            o.step()
        toks, blks = [], []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            a, b = o.step()
            toks.append(a)
            blks.append(b)
        wall = time.perf_counter() - t0
    finally:
        o.close()
    cpu = o.figures(statistics.median(toks), statistics.median(blks))
    value = cpu["value"]
    line = {"impl": "reference", "metric": "KV rows scored/s", "value": value, "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * wall / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes of the pages' workloads)", "config": config_dict(tw, bw, world),
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "timing": "ms_per_step: measured wall time of one sample step (whole token step + block slice); "
                      "value: whole-step rows / (token step measured + block slice wall / its work fraction)",
            "wall_s": wall}
    print(json.dumps(line), flush=True)


EXTRA_CASES = ("restore_blocks", "rerope_shift", "workset_diff", "span_keep", "rule_scores_batch", "index_to_fp8",
               "index_from_fp8", "topk_small")


def extra_profile_case(args):
    """The widened rows at representative sizes, for ncu captures and per-call timing:
    restore_blocks / rerope_shift: 2048 blocks of the 1M-workspace dims (L64 Hkv8 D128, 32-token
    pages); workset_diff: two 2180-block working sets sharing two thirds; span_keep: N=92160 with
    100 of 400 cursors deleted; rule_scores_batch: 36 sessions of 1024-8192 tokens at the 8B shape;
    index_to_fp8 / index_from_fp8: the 1M-workspace index (32768 blocks, Hkv8 D128) per layer;
    topk_small: top-C* of a 16384-token session (C=4096, the 8-CTA cluster path); topk_n<N>: top-C* of an
    N-token session (C = N/4)."""
    import numpy as np
    import torch

    import kv_cache_retention_gb300 as kv

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    rng = np.random.default_rng(1)
    name = args.profile_kernel
    L, Hkv, D, page = args.profile_layers, 8, 128, 32
    if name in ("restore_blocks", "rerope_shift"):
        n, P = 2048, 2180
        k = torch.empty((L, Hkv, n * page, D), device="cuda", dtype=torch.bfloat16).normal_()
        v = torch.empty_like(k).normal_()
        kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
        vp = torch.zeros_like(kp)
        pages = torch.as_tensor(rng.permutation(P)[:n].astype(np.int32), device="cuda")
        if name == "restore_blocks":
            src = torch.arange(n, device="cuda", dtype=torch.int32)
            fn = lambda: ctx.restore_blocks(k, v, src, pages, src * page, kp, vp, 1e6)  # noqa: E731
            moved = 2 * 4 * L * Hkv * n * page * D  # K and V, read and written, 2 bytes each
        else:
            shifts = torch.as_tensor(rng.integers(-4096, 4096, n).astype(np.int32) * page, device="cuda")
            fn = lambda: ctx.rerope_shift(kp, pages, shifts, 1e6)  # noqa: E731
            moved = 2 * 2 * L * Hkv * n * page * D  # K read and written in place, 2 bytes each
    elif name == "workset_diff":
        prev = np.sort(rng.choice(40000, 2180, replace=False)).astype(np.int32)
        keep = prev[rng.random(prev.size) < 0.67]
        new = np.sort(np.concatenate([keep, rng.choice(np.setdiff1d(np.arange(40000), prev), 2180 - keep.size,
                                                       replace=False)])).astype(np.int32)
        ti = [torch.as_tensor(a, device="cuda") for a in (prev, rng.permutation(2180).astype(np.int32), new)]
        fn = lambda: ctx.workset_diff(ti[0], ti[1], ti[2], 2180, page)  # noqa: E731
        moved = 0
    elif name in ("index_to_fp8", "index_from_fp8"):
        nb = 32768
        ix = torch.empty((L, Hkv, nb, D), device="cuda", dtype=torch.bfloat16).normal_()
        codes = torch.empty(ix.shape, dtype=torch.uint8, device="cuda")
        exps = torch.empty(ix.shape[:-1], dtype=torch.int8, device="cuda")
        out = torch.empty_like(ix)
        ctx.index_to_fp8(ix, codes, exps)
        if name == "index_to_fp8":
            fn = lambda: ctx.index_to_fp8(ix, codes, exps)  # noqa: E731
        else:
            fn = lambda: ctx.index_from_fp8(codes, exps, out)  # noqa: E731
        moved = L * Hkv * nb * (3 * D + 1)
    elif name == "topk_small" or name.startswith("topk_n"):
        N = 16384 if name == "topk_small" else int(name[len("topk_n"):])
        score = torch.rand(N, device="cuda")
        keep = torch.empty(N, dtype=torch.uint8, device="cuda")
        keep_idx = torch.empty(N, dtype=torch.int32, device="cuda")
        C = 4096 if name == "topk_small" else N // 4
        fn = lambda: ctx.topk_retain(score, 256, N - 512, N, C, keep=keep, keep_idx=keep_idx)  # noqa: E731
        moved = 5 * N
    elif name == "span_keep":
        N = 92160
        start = torch.as_tensor(rng.integers(0, N, 400).astype(np.int32), device="cuda")
        end = start + torch.as_tensor(rng.integers(16, 2048, 400).astype(np.int32), device="cuda")
        dels = torch.as_tensor(rng.choice(400, 100, replace=False).astype(np.int32), device="cuda")
        keep = torch.ones(N, dtype=torch.uint8, device="cuda")
        fn = lambda: ctx.span_keep(start, end, dels, N, keep, keep_in=keep)  # noqa: E731
        moved = 2 * N
    else:
        S, Hq = 36, 32
        Ns = [int(x) for x in rng.integers(1024, 8193, S)]
        n_slots = sum((x + 15) // 16 for x in Ns) * 16
        pool = torch.empty((L, n_slots, Hkv, D), device="cuda", dtype=torch.bfloat16).normal_()
        perm, at, smaps = rng.permutation(n_slots // 16), 0, []
        for x in Ns:
            m = (x + 15) // 16
            j = np.arange(x)
            smaps.append(torch.as_tensor((perm[at:at + m][j // 16] * 16 + j % 16).astype(np.int32), device="cuda"))
            at += m
        Ms = [torch.nn.functional.normalize(torch.randn((L, Hq, D), device="cuda"), dim=-1) for _ in Ns]
        rules = [torch.empty(x, device="cuda") for x in Ns]
        forced = [(64, x - 256, x) for x in Ns]
        fn = lambda: ctx.rule_scores_batch(pool, Ms, L, Hq, Hkv, Ns, D, forced, rules, slot_maps=smaps,  # noqa: E731
                                           n_slots=n_slots)
        moved = sum(L * Hkv * (x - 320) * D * 2 for x in Ns)
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(args.steps):
        fn()
    b0.record()
    torch.cuda.synchronize()
    ctx.check_device()
    ms = a0.elapsed_time(b0) / args.steps
    line = {"profile_case": name, "layers": L, "ms_per_call": ms}
    if moved:
        line["GBs"] = moved / (ms / 1e3) / 1e9
    print(json.dumps(line), flush=True)


def profile_case(args):
    """Small case for ncu captures: only `--profile-kernel` runs, on the bench's
    workloads cut to `--profile-layers` layers (inputs still larger than L2)."""
    import dataclasses

    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    if args.profile_kernel in EXTRA_CASES or args.profile_kernel.startswith("topk_n"):
        extra_profile_case(args)
        return
    torch.cuda.set_device(0)
    tw = dataclasses.replace(synth.TOKEN[TOKEN_WL], L=args.profile_layers)
    bw = dataclasses.replace(synth.BLOCK[BLOCK_WL], L=args.profile_layers)
    ctx = kv.Context(0)
    s = setup_session(kv, synth, ctx, tw, bw, torch)
    name = args.profile_kernel
    ev = {}

    def one():
        sub = {}
        run_step_only(ctx, s, name, sub)
        for k, v in sub.items():
            ev.setdefault(k, []).extend(v)

    for _ in range(args.warmup):
        run_step_only(ctx, s, name, None)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        one()
    torch.cuda.synchronize()
    ctx.check_device()
    ms = sum(a.elapsed_time(b) for a, b in ev[name]) / len(ev[name])
    print(json.dumps({"profile_case": name, "layers": args.profile_layers, "ms_per_call": ms}), flush=True)


def all_configs(args):
    """One JSON line per workload: per-call device times of its select step
    (CUDA events, mean over --steps after --warmup), the step replayed from one
    CUDA graph, rows/s and the roofline fraction of its bandwidth- or tensor-bound calls.  Token workloads run the
    IntentKV step, block workloads the KVMEM step (full Mean-K build when the
    workload is not incremental; the scatter then reads the raw K of the
    selected blocks)."""
    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    peaks = _peaks()

    def timed(calls):
        for _ in range(args.warmup):
            for _, fn in calls:
                fn()
        torch.cuda.synchronize()
        ev = {}
        for _ in range(args.steps):
            for name, fn in calls:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                ev.setdefault(name, []).append((a, b))
        torch.cuda.synchronize()
        ctx.check_device()
        per_call = {k: statistics.median(a.elapsed_time(b) for a, b in v) for k, v in ev.items()}
        # whole steps with no per-call events (what a caller sees per step; for the µs-scale
        # workloads the per-call events themselves cost host time); median over steps
        marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        marks[0].record()
        for i in range(args.steps):
            for _, fn in calls:
                fn()
            marks[i + 1].record()
        torch.cuda.synchronize()
        ctx.check_device()
        return per_call, 1e3 * statistics.median(marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps))

    def graph_us(calls):
        """The step's calls captured once in a CUDA graph; mean wall time of a replay (CUDA events)."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _, fn in calls:
                fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _, fn in calls:
                fn()
        for _ in range(args.warmup):
            g.replay()
        a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a0.record()
        for _ in range(max(1, args.steps)):
            g.replay()
        b0.record()
        torch.cuda.synchronize()
        ctx.check_device()
        return 1e3 * a0.elapsed_time(b0) / max(1, args.steps)

    def frac(bound, amount, ms):
        if bound == "hbm":
            ach = amount / (ms / 1e3) / 1e9
            return {"achieved_GBs": ach, "frac_hbm": ach / peaks["hbm_gbs"]}
        ach = amount / (ms / 1e3) / 1e12
        return {"achieved_TFLOPs": ach, "frac_tensor_sustained": ach / peaks["bf16_tflops_sustained"]}

    for name, tw in synth.TOKEN.items():
        t = synth.token_inputs(tw, "cuda")
        M = torch.zeros((tw.L, tw.Hq, tw.D), device="cuda")
        for i in range(tw.turns - 1):
            ctx.memory_update(t["turns"][i], tw.lam, M, first_turn=(i == 0))
        q_last = t["turns"][tw.turns - 1].contiguous()
        rule = torch.empty(tw.N, device="cuda")
        keep = torch.empty(tw.N, device="cuda", dtype=torch.uint8)
        keep_idx = torch.empty(tw.N, device="cuda", dtype=torch.int32)
        smap = t["slot_map"] if t["slot_map"] is not None else torch.arange(tw.N, device="cuda", dtype=torch.int32)
        slot_out = torch.empty(tw.N, device="cuda", dtype=torch.int32)
        calls = [
            ("memory_update", lambda: ctx.memory_update(q_last, tw.lam, M)),
            ("rule_scores", lambda: ctx.rule_scores(t["pool"], M, tw.L, tw.Hq, tw.Hkv, tw.N, tw.D, tw.pi, tw.q_s,
                                                    tw.q_e, rule, slot_map=t["slot_map"], n_slots=tw.N)),
            ("topk_retain", lambda: ctx.topk_retain(rule, tw.pi, tw.q_s, tw.q_e, tw.C, keep=keep, keep_idx=keep_idx)),
            ("redirect_slots", lambda: ctx.redirect_slots(smap, keep, tw.dead_slot, slot_out)),
        ]
        ms, step_us = timed(calls)
        es = 2 if tw.dtype == "bf16" else 4
        rows = tw.L * tw.Hkv * tw.n_cand
        line = {"workload": tw.name, "kind": "IntentKV token step", "us_per_select_step": step_us,
                "us_per_select_step_graph": graph_us(calls),
                "rows_scored_per_s": rows / (step_us / 1e6), "ms": ms,
                "rule_scores": frac("hbm", tw.L * tw.n_cand * tw.Hkv * tw.D * es + tw.N * 4, ms["rule_scores"])}
        print(json.dumps(line), flush=True)
        del t, M
        torch.cuda.empty_cache()

    for name, bw in synth.BLOCK.items():
        b = synth.block_inputs(bw, "cuda")
        R = torch.empty(bw.n_blocks, device="cuda")
        ids = torch.empty(bw.n_sel, device="cuda", dtype=torch.int32)
        n_top = min(bw.k, bw.n_cand)
        if bw.incremental:
            src_block, dst_page, dst_pos0 = synth.scatter_plan_incremental(bw, b["page_perm"])
            build = lambda: ctx.meank_build(b["raw"], bw.block, b["index"], first_block=bw.first_new_block)  # noqa: E731
            scatter = lambda: ctx.rerope_scatter(b["staging"], src_block, dst_page, dst_pos0, b["pool"],  # noqa: E731
                                                 bw.rope_base)
            built_tokens, moved_blocks = bw.new_tokens, n_top
        else:
            dst_page, dst_pos0 = synth.scatter_plan_full(bw, b["page_perm"])
            build = lambda: ctx.meank_build(b["raw"], bw.block, b["index"])  # noqa: E731
            scatter = lambda: ctx.rerope_scatter(b["raw"], ids, dst_page, dst_pos0, b["pool"], bw.rope_base)  # noqa: E731
            built_tokens, moved_blocks = bw.n_blocks * bw.block, bw.n_sel
        calls = [
            ("meank_build", build),
            ("block_scores", lambda: ctx.block_scores(b["q"], b["index"], bw.n_blocks, bw.n_sink, bw.n_recent, R)),
            ("select_blocks", lambda: ctx.select_blocks(R, bw.n_sink, bw.n_recent, bw.k, ids)),
            ("rerope_scatter", scatter),
        ]
        ms, step_us = timed(calls)
        rows = bw.L * bw.Hkv * bw.n_cand
        build_bytes = bw.L * bw.Hkv * (built_tokens + built_tokens // bw.block) * bw.D * 2
        line = {"workload": bw.name, "kind": "KVMEM block step", "us_per_select_step": step_us,
                "us_per_select_step_graph": graph_us(calls),
                "rows_scored_per_s": rows / (step_us / 1e6), "ms": ms,
                "meank_build": frac("hbm", build_bytes, ms["meank_build"]),
                "block_scores": frac("tensor", 2 * bw.L * bw.Hq * bw.M * bw.n_cand * bw.D, ms["block_scores"]),
                "rerope_scatter": frac("hbm", 2 * bw.L * bw.Hkv * moved_blocks * bw.block * bw.D * 2,
                                       ms["rerope_scatter"])}
        line["block_scores"]["pairs_per_s"] = bw.L * bw.Hq * bw.M * bw.n_cand / (ms["block_scores"] / 1e3)
        print(json.dumps(line), flush=True)
        del b
        torch.cuda.empty_cache()


def restore_pipeline(args):
    """Throughput of the packed, pipelined host -> device restore (kvsel_stage_restore) at the 1M-workspace
    dims (L64 Hkv8 D128, 32-token blocks: 4 MiB of K+V per block): 256 blocks restored from a 384-block host
    repository in shuffled order, per batch size, from pageable and from pinned memory; beside it the
    host -> device link alone (one pinned copy of the same bytes) and the restore kernel alone (from device
    memory)."""
    import numpy as np
    import torch

    import kv_cache_retention_gb300 as kv

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    L, Hkv, D, page, n_repo, n, P = 64, 8, 128, 32, 384, 256, 2180
    g = torch.Generator().manual_seed(77)
    seed_k = torch.randn((L, Hkv, 16 * page, D), generator=g).to(torch.bfloat16)
    seed_v = torch.randn((L, Hkv, 16 * page, D), generator=g).to(torch.bfloat16)
    hk = seed_k.repeat(1, 1, n_repo // 16, 1).contiguous()
    hv = seed_v.repeat(1, 1, n_repo // 16, 1).contiguous()
    rng = np.random.default_rng(5)
    blocks = rng.choice(n_repo, n, replace=False).astype(np.int32)
    pages = rng.choice(P, n, replace=False).astype(np.int32)
    pos0 = (np.arange(n) * page).astype(np.int32)
    kp = torch.zeros((L, P, page, Hkv, D), device="cuda", dtype=torch.bfloat16)
    vp = torch.zeros_like(kp)
    nbytes = 2 * L * Hkv * n * page * D * 2

    def timed(fn, reps=3):
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    out = {"workload": "restore 256 of 384 host blocks, L64 Hkv8 D128, 32-token blocks (K+V 4 MiB per block)",
           "bytes": nbytes, "staged": {}}
    pk, pv = hk.pin_memory(), hv.pin_memory()
    for mem, (k_src, v_src) in (("pageable", (hk, hv)), ("pinned", (pk, pv))):
        for chunk in (4, 16, 64):
            for threads in (8, 16):
                sec = timed(lambda: ctx.stage_restore(k_src, v_src, blocks, pages, pos0, kp, vp, 1e6,
                                                      chunk_blocks=chunk, gather_threads=threads,
                                                      mode=kv.STAGE_PACKED))
                out["staged"][f"{mem}_chunk{chunk}_threads{threads}"] = {"ms": 1e3 * sec, "GBs": nbytes / sec / 1e9}
    sec = timed(lambda: ctx.stage_restore(pk, pv, blocks, pages, pos0, kp, vp, 1e6, mode=kv.STAGE_DIRECT))
    out["direct_pinned"] = {"ms": 1e3 * sec, "GBs": nbytes / sec / 1e9}
    ctx.check_device()
    link_src = torch.empty(nbytes // 2, dtype=torch.bfloat16).pin_memory()
    link_dst = torch.empty(nbytes // 2, dtype=torch.bfloat16, device="cuda")
    sec = timed(lambda: link_dst.copy_(link_src, non_blocking=True))
    out["link_h2d"] = {"ms": 1e3 * sec, "GBs": nbytes / sec / 1e9}
    dk, dv = hk.cuda(), hv.cuda()
    sb, dpg, d0 = (torch.as_tensor(a, device="cuda") for a in (blocks, pages, pos0))
    sec = timed(lambda: ctx.restore_blocks(dk, dv, sb, dpg, d0, kp, vp, 1e6))
    out["kernel_only"] = {"ms": 1e3 * sec, "GBs": 2 * nbytes / sec / 1e9, "note": "read + write bytes"}
    ctx.check_device()
    print(json.dumps(out), flush=True)


def block_sweep(args):
    """Mean-K block size sweep (beta = 16 / 32 / 64) at a fixed history and a fixed token budget: the
    Mean-K workload's 262,144-token history (L64 Hq40 Hkv8 D128, 512 query tokens), keeping 128 sink and
    2048 recent tokens plus the top 32,768 tokens' worth of blocks; full Mean-K build, R_b, working set and
    re-RoPE scatter of the working set per beta (CUDA events, mean over --steps)."""
    import dataclasses

    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    base = synth.BLOCK["meank262k"]
    tokens = base.n_blocks * base.block
    for beta in (16, 32, 64):
        bw = dataclasses.replace(base, block=beta, n_blocks=tokens // beta, n_sink=128 // beta,
                                 n_recent=2048 // beta, k=32768 // beta)
        b = synth.block_inputs(bw, "cuda")
        R = torch.empty(bw.n_blocks, device="cuda")
        ids = torch.empty(bw.n_sel, device="cuda", dtype=torch.int32)
        dst_page, dst_pos0 = synth.scatter_plan_full(bw, b["page_perm"])
        calls = [
            ("meank_build", lambda: ctx.meank_build(b["raw"], bw.block, b["index"])),
            ("block_scores", lambda: ctx.block_scores(b["q"], b["index"], bw.n_blocks, bw.n_sink, bw.n_recent, R)),
            ("select_blocks", lambda: ctx.select_blocks(R, bw.n_sink, bw.n_recent, bw.k, ids)),
            ("rerope_scatter", lambda: ctx.rerope_scatter(b["raw"], ids, dst_page, dst_pos0, b["pool"], bw.rope_base)),
        ]
        for _ in range(args.warmup):
            for _, fn in calls:
                fn()
        torch.cuda.synchronize()
        ev = {}
        for _ in range(args.steps):
            for name, fn in calls:
                a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record()
                fn()
                b0.record()
                ev.setdefault(name, []).append((a0, b0))
        torch.cuda.synchronize()
        ctx.check_device()
        ms = {k: sum(x.elapsed_time(y) for x, y in v) / len(v) for k, v in ev.items()}
        index_bytes = bw.L * bw.Hkv * bw.n_blocks * bw.D * 2
        print(json.dumps({"beta": beta, "blocks": bw.n_blocks, "candidates": bw.n_cand, "selected": bw.n_sel,
                          "index_MB": index_bytes / 1e6, "ms": ms,
                          "select_step_ms": ms["block_scores"] + ms["select_blocks"] + ms["rerope_scatter"]}),
              flush=True)
        del b
        torch.cuda.empty_cache()


def fp8_index(args):
    """FP8 (E4M3) index storage at the 1M-token workspace (L64 Hq40 Hkv8 D128, 32768 blocks of 32, 2048
    queries): the Mean-K index stored as codes + a scale exponent per row, expanded to bf16 before R_b.
    Reports index bytes, the quantise and expand calls' times (CUDA events, mean over --steps) with their
    HBM fraction, and how the FP8 index changes the selected working set (overlap of the top-k blocks)."""
    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    peaks = _peaks()
    bw = synth.BLOCK[BLOCK_WL]
    b = synth.block_inputs(bw, "cuda", with_staging=False)
    index = b["index"]
    ctx.meank_build(b["raw"], bw.block, index, first_block=bw.first_new_block)  # the new blocks' Mean-K rows
    rows = bw.L * bw.Hkv * index.shape[2]
    D = bw.D
    codes = torch.empty(index.shape, dtype=torch.uint8, device="cuda")
    exps = torch.empty(index.shape[:-1], dtype=torch.int8, device="cuda")
    back = torch.empty_like(index)
    calls = [("index_to_fp8", lambda: ctx.index_to_fp8(index, codes, exps)),
             ("index_from_fp8", lambda: ctx.index_from_fp8(codes, exps, back))]
    for _ in range(args.warmup):
        for _, fn in calls:
            fn()
    torch.cuda.synchronize()
    ev = {}
    for _ in range(args.steps):
        for name, fn in calls:
            a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record()
            fn()
            b0.record()
            ev.setdefault(name, []).append((a0, b0))
    torch.cuda.synchronize()
    ctx.check_device()
    ms = {k: sum(x.elapsed_time(y) for x, y in v) / len(v) for k, v in ev.items()}
    moved = rows * (2 * D + D + 1)  # bf16 row read + codes and exponent written (or the reverse)
    out = {"workload": f"1M workspace index [L{bw.L} Hkv{bw.Hkv} {index.shape[2]} blocks D{D}]",
           "index_bf16_MB": rows * 2 * D / 1e6, "index_fp8_MB": rows * (D + 1) / 1e6}
    for k, v in ms.items():
        gbs = moved / (v / 1e3) / 1e9
        out[k] = {"ms": v, "GB_s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"], "bytes": moved}
    # the working set selected from the FP8 index against the one from the bf16 index
    R16, R8 = torch.empty(bw.n_blocks, device="cuda"), torch.empty(bw.n_blocks, device="cuda")
    ids16 = torch.empty(bw.n_sel, device="cuda", dtype=torch.int32)
    ids8 = torch.empty(bw.n_sel, device="cuda", dtype=torch.int32)
    ctx.block_scores(b["q"], index, bw.n_blocks, bw.n_sink, bw.n_recent, R16)
    ctx.block_scores(b["q"], back, bw.n_blocks, bw.n_sink, bw.n_recent, R8)
    ctx.select_blocks(R16, bw.n_sink, bw.n_recent, bw.k, ids16)
    ctx.select_blocks(R8, bw.n_sink, bw.n_recent, bw.k, ids8)
    torch.cuda.synchronize()
    ctx.check_device()
    C = slice(bw.n_sink, bw.n_blocks - bw.n_recent)
    same = len(set(ids16.cpu().tolist()) & set(ids8.cpu().tolist()))
    out["R_b_max_rel_change"] = float(((R8[C] - R16[C]).abs() / R16[C]).max())
    out["working_set_overlap"] = same / bw.n_sel
    out["data"] = "synthetic: the bench's 1M-workspace index (drawn old blocks + Mean-K of the new raw K)"
    print(json.dumps(out), flush=True)


def batch_sessions(args):
    """A serving batch of 36 sessions (8B shape: L36 Hq32 Hkv8 D128, bf16 K in one shared pool of 16-slot
    pages, N drawn from 1024-8192 per session, 64 query rows per turn, C = N/4): the IntentKV step
    (QueryMemory update, rule scores, top-C*) as three batched calls, against the same sessions stepped
    one by one with the single-session calls on the same stream (CUDA events, mean over --steps)."""
    import numpy as np
    import torch

    import kv_cache_retention_gb300 as kv

    torch.cuda.set_device(0)
    ctx = kv.Context(0)
    S, L, Hq, Hkv, D, page = 36, 36, 32, 8, 128, 16
    rng = np.random.default_rng(36)
    Ns = [int(n) for n in rng.integers(1024, 8193, S)]
    n_slots = sum((n + page - 1) // page for n in Ns) * page
    pool = torch.empty((L, n_slots, Hkv, D), device="cuda", dtype=torch.bfloat16).normal_()
    perm = rng.permutation(n_slots // page)
    smaps, Ms, qs, rules, keeps, forced, Cs = [], [], [], [], [], [], []
    at = 0
    for N in Ns:
        np_ = (N + page - 1) // page
        pages = perm[at:at + np_]
        at += np_
        j = np.arange(N)
        smaps.append(torch.as_tensor((pages[j // page] * page + j % page).astype(np.int32), device="cuda"))
        Ms.append(torch.nn.functional.normalize(torch.randn((L, Hq, D), device="cuda"), dim=-1))
        qs.append(torch.randn((L, Hq, 64, D), device="cuda").to(torch.bfloat16))
        rules.append(torch.empty(N, device="cuda"))
        keeps.append(torch.empty(N, dtype=torch.uint8, device="cuda"))
        forced.append((64, N - 256, N))
        Cs.append(N // 4)

    def batched():
        ctx.memory_update_batch(qs, [0.3] * S, Ms)
        ctx.rule_scores_batch(pool, Ms, L, Hq, Hkv, Ns, D, forced, rules, slot_maps=smaps, n_slots=n_slots)
        ctx.topk_retain_batch(rules, forced, Cs, keeps)

    def one_by_one():
        for i in range(S):
            ctx.memory_update(qs[i], 0.3, Ms[i])
            ctx.rule_scores(pool, Ms[i], L, Hq, Hkv, Ns[i], D, *forced[i], rules[i], slot_map=smaps[i],
                            n_slots=n_slots)
            ctx.topk_retain(rules[i], *forced[i], Cs[i], keep=keeps[i])

    out = {"workload": "36 sessions, L36 Hq32 Hkv8 D128, N 1024-8192 per session", "sessions": S,
           "tokens": sum(Ns)}
    rows = sum(L * Hkv * (N - 64 - 256) for N in Ns)
    for name, fn in (("batched", batched), ("one_by_one", one_by_one)):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(args.steps):
            fn()
        b0.record()
        torch.cuda.synchronize()
        ms = a0.elapsed_time(b0) / args.steps
        out[name] = {"ms": ms, "rows_per_s": rows / (ms / 1e3),
                     "launches": 5 if name == "batched" else 5 * S}
    ctx.check_device()
    out["speedup"] = out["one_by_one"]["ms"] / out["batched"]["ms"]
    print(json.dumps(out), flush=True)


def run_step_only(ctx, s, name, ev):
    """Run only the call `name` of the step (for profiling captures)."""
    tw, bw = s["tw"], s["bw"]
    table = {
        "memory_update": lambda: ctx.memory_update(s["q_last"], tw.lam, s["M"]),
        "rule_scores": lambda: ctx.rule_scores(s["pool"], s["M"], tw.L, tw.Hq, tw.Hkv, tw.N, tw.D, tw.pi, tw.q_s,
                                               tw.q_e, s["rule"], slot_map=s["slot_map"], n_slots=tw.N),
        "topk_retain": lambda: ctx.topk_retain(s["rule"], tw.pi, tw.q_s, tw.q_e, tw.C, keep=s["keep"],
                                               keep_idx=s["keep_idx"]),
        "meank_build": lambda: ctx.meank_build(s["raw_new"], bw.block, s["index"], first_block=bw.first_new_block),
        "block_scores": lambda: ctx.block_scores(s["q"], s["index"], bw.n_blocks, bw.n_sink, bw.n_recent, s["R"]),
        "select_blocks": lambda: ctx.select_blocks(s["R"], bw.n_sink, bw.n_recent, bw.k, s["ids"]),
        "rerope_scatter": lambda: ctx.rerope_scatter(s["staging"], s["src_block"], s["dst_page"], s["dst_pos0"],
                                                     s["kpool"], bw.rope_base),
    }
    fn = table[name]
    if ev is None:
        fn()
        return
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    ev.setdefault(name, []).append((a, b))


def e2e_timeline(args):
    """The end-to-end loop of the bench line with CUDA events on both streams: when each
    step's input copies start and land (copy stream) and when its calls run (compute
    stream), in ms from the loop's start, plus the copies alone afterwards.  Shows whether
    the copies of step t+1 overlap step t and which side waits."""
    import torch

    import kv_cache_retention_gb300 as kv
    import synth

    torch.cuda.set_device(0)
    tw, bw = synth.TOKEN[TOKEN_WL], synth.BLOCK[BLOCK_WL]
    ctx = kv.Context(0)
    s = setup_session(kv, synth, ctx, tw, bw, torch)
    for _ in range(args.warmup):
        run_step(ctx, s)
    torch.cuda.synchronize()
    in_keys = ("q_last", "raw_new", "q", "staging")
    h_in = {k: s[k].detach().cpu().pin_memory() for k in in_keys}
    h_out = {k: torch.empty_like(s[k], device="cpu").pin_memory() for k in ("rule", "slot_out", "keep_idx", "R", "ids")}
    sets = [s, dict(s)]
    for k in in_keys:
        sets[1][k] = torch.empty_like(s[k])
    copy_stream, comp = torch.cuda.Stream(), torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ev_copied = [{k: ev() for k in in_keys} for _ in range(2)]
    ev_done = [ev(), ev()]
    marks = []

    def issue_copy(i):
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(ev_done[i % 2])
            a = ev()
            a.record(copy_stream)
            marks.append((f"copy {i} start", a))
            for k in in_keys:
                sets[i % 2][k].copy_(h_in[k], non_blocking=True)
                ev_copied[i % 2][k].record(copy_stream)  # reused two steps later: the wait's event
                m = ev()  # the mark's own event
                m.record(copy_stream)
                marks.append((f"copy {i} {k} landed", m))

    start = ev()
    start.record()
    copy_stream.wait_event(start)
    issue_copy(0)
    n = max(2, args.steps)
    for i in range(n):
        if i + 1 < n:
            issue_copy(i + 1)
        calls = {}
        run_step(ctx, sets[i % 2], calls, ready=ev_copied[i % 2])
        for name, v in calls.items():
            marks.append((f"step {i} {name} start", v[0][0]))
            marks.append((f"step {i} {name} end", v[0][1]))
        ev_done[i % 2].record(comp)
        for k, t in h_out.items():
            t.copy_(sets[i % 2][k], non_blocking=True)
    end = ev()
    end.record()
    torch.cuda.synchronize()
    rows = []
    for name, e in marks:
        rows.append((round(start.elapsed_time(e), 2), name))
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    c0, c1 = ev(), ev()
    with torch.cuda.stream(copy_stream):
        c0.record(copy_stream)
        for k in in_keys:
            sets[0][k].copy_(h_in[k], non_blocking=True)
        c1.record(copy_stream)
    torch.cuda.synchronize()
    print(json.dumps({"e2e_timeline": "bench step, inputs from pinned host memory", "steps": n,
                      "ms_per_step": start.elapsed_time(end) / n, "h2d_bytes_per_step": h2d,
                      "copies_alone_ms": c0.elapsed_time(c1), "events": sorted(rows)}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-kernel", default=None,
                    help="run only this call (or these, comma-separated) on a cut-down case (for ncu)")
    ap.add_argument("--profile-layers", type=int, default=4)
    ap.add_argument("--all-configs", action="store_true", help="time the select step of every workload, one line each")
    ap.add_argument("--restore-pipeline", action="store_true", help="throughput of the staged host -> device restore")
    ap.add_argument("--block-sweep", action="store_true", help="Mean-K block size sweep (16 / 32 / 64 tokens)")
    ap.add_argument("--batch-sessions", action="store_true", help="36-session batched IntentKV step vs one by one")
    ap.add_argument("--fp8-index", action="store_true", help="FP8 (E4M3) index storage: quantise / expand cost, R_b change")
    ap.add_argument("--e2e-timeline", action="store_true",
                    help="the end-to-end loop with events on the copy and compute streams (overlap check)")
    args = ap.parse_args()
    if args.e2e_timeline:
        e2e_timeline(args)
        return
    if args.batch_sessions:
        batch_sessions(args)
        return
    if args.fp8_index:
        fp8_index(args)
        return
    if args.block_sweep:
        block_sweep(args)
        return
    if args.all_configs:
        all_configs(args)
        return
    if args.restore_pipeline:
        restore_pipeline(args)
        return
    if args.profile_kernel:
        for name in args.profile_kernel.split(","):  # several calls in turn, each on its own case
            profile_case(argparse.Namespace(**{**vars(args), "profile_kernel": name}))
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if "RANK" in os.environ else 1)))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference(args, rank, world)
    else:
        ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
