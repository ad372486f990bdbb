#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify transaction on one GB300.

Workload (default): Qwen3-4B-shaped decoder (36 layers, hidden 2560, 32/8 heads
of 128, FFN 9728, vocab 151936, bf16 weights N(0, 0.02) from seed 2), batch 1,
848 uniform-random context tokens prefilled into the paged KV (page 16), then
verify steps of S = K+1 = 8 rows with uniform-random drafts. A step is the
whole hot path: propose -> ensure_capacity -> spec_forward (verify) ->
accept_greedy -> rewind_cache, replayed as one CUDA graph.

Metric: committed tokens/s (whole job, all GPUs). The JSON line also carries
the batch-16 (contexts U[512, 4096]) and 32768-token-context lines as
sub-objects, the per-S latency sweep (S = 1..17), the HBM roofline of the
dominant kernel (the tcgen05 weight-streaming GEMM) timed inside the captured
step from the device timeline, the end-to-end figure through host buffers, and
the CPU oracle timed on the host cores in a fresh process.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                  [--workload b1|b16|ctx32k|ngram] [--no-extra] [--no-sweep] [--no-cpu-baseline]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CONTEXT = 848
K_DRAFT = 7
SEED = 2
N_LAYERS = 36
# Weight bytes of one forward (bf16): per layer the four GEMMs' matrices
# (q/k/v 6144 x 2560, o 2560 x 4096, gate+up 2 x 9728 x 2560, down 2560 x 9728) and the four norm
# gains; then the LM head (151936 x 2560) and the final norm.
GEMM_BYTES_PER_LAYER = 201_850_880
GEMM_BYTES = {"qkv": 31_457_280, "o": 20_971_520, "gate_up": 99_614_720, "down": 49_807_360,
              "lm_head": 777_912_320}
# weights streamed per 36-layer step: 36 x (201,850,880 + 10,752 norm gains) + LM head + final norm
# = 8,044,936,192 B
KV_BYTES_PER_TOKEN = 147_456               # 2 (K,V) x 8 heads x 128 x 2 B x 36 layers
EMBED_BYTES_PER_ROW = 2560 * 2
# DRAM bytes (read + write) that ncu measured per launch of the weight-streaming GEMM, in a
# 2-layer case of the same shapes (profiles/gemm_tcgen05_qwen3_4b_verify_N16.md); a launch streams
# its own weights, so a 36-layer step is 36 layers of the first four plus one LM head.
GEMM_TRAFFIC_MB = {"qkv": 31.6983, "o": 21.3682, "gate_up": 99.9138, "down": 50.5648, "lm_head": 778.4595}
from speculative_decoding_verify_02_gb300 import TRACE_REGION_CTAS, TRACE_STAMPS  # noqa: E402
TRACE_REGION_WORDS = TRACE_REGION_CTAS * TRACE_STAMPS  # sdv_fwd_trace: one region per launch
PROJ = ("qkv", "o", "gate_up", "down")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def aggregate_replicas(committed, ms, e2e_committed, e2e_s, device):
    """Whole-job totals over independent replicas (one per rank, no exchange on the data path):
    committed tokens summed over the ranks, times the maximum over the ranks (the job ends with its
    slowest replica). Returns (committed, ms, e2e committed, e2e seconds)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([committed, ms, e2e_committed, e2e_s], dtype=torch.float64, device=device)
    tot, mx = t.clone(), t.clone()
    dist.all_reduce(tot, op=dist.ReduceOp.SUM)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    return float(tot[0]), float(mx[1]), float(tot[2]), float(mx[3])


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            sel = ["-i", str(self.idx)] if self.idx is not None else []
            self.proc = subprocess.Popen(["nvidia-smi", *sel, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(float(r[2]) for r in rows),
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ----------------------------------------------------------------------------- helpers

def build_weights(shape, seed, device="cuda"):
    import synth
    from speculative_decoding_verify_02_gb300 import upload_bf16
    dev = {}
    for name in shape.tensor_shapes():
        dev[name] = upload_bf16(synth.tensor(shape, seed, name), device)
    return dev


def timed_replays(loop, steps, stream):
    """Device time (ms) of `steps` graph replays, CUDA events on the launching stream."""
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        loop.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def trace_launches(buf, n_layers):
    """The launches of the last traced step from the device timeline, in stream order (per layer
    QKV, attention, O, gate/up, down; then the LM head). For each launch: its first CTA start, the
    first CTA past its wait on the previous kernel ("ready"), and its last CTA end (ns). Each
    launch's exclusive window is its end minus the previous launch's end: the windows partition
    the step, so PDL's early CTA starts are not counted twice."""
    t = buf.view(-1, TRACE_REGION_WORDS // 16, 16).cpu().numpy()
    first = t[1, :, 0]
    t0 = int(first[first > 0].min())          # every CTA of layer 0's QKV launch runs each step
    order = []
    for l in range(n_layers):
        order += [("qkv", 5 * l + 1), ("attention", 5 * l), ("o", 5 * l + 2), ("gate_up", 5 * l + 3),
                  ("down", 5 * l + 4)]
    order.append(("lm_head", 5 * n_layers))
    launches = []
    for name, region in order:
        c = t[region]
        attn = name == "attention"
        end_ev = 6 if attn else 8
        ok = (c[:, 0] >= t0) & (c[:, end_ev] >= c[:, 0])
        c = c[ok]
        ready = c[:, 0] if attn else c[:, 1]      # the attention stamps its start after its wait
        pass0 = None
        if not attn:  # the first row pass of the CTAs' first warp: partials summed, rows written
            w = (c[:, 9] >= c[:, 6]) & (c[:, 10] >= c[:, 9]) & (c[:, 6] > 0)
            if w.any():
                pass0 = (float(np.median(c[w, 9] - c[w, 6])), float(np.median(c[w, 10] - c[w, 9])))
        launches.append({"name": name, "start": int(c[:, 0].min()), "ready": int(ready.min()),
                         "end": int(c[:, end_ev].max()),
                         "first_stage": None if attn else int(c[:, 2].max()),
                         "last_mma": None if attn else int(c[:, 3].max()),
                         "reduced": None if attn else int(c[:, 6].max()),
                         "rows": None if attn else int(c[:, 7].max()), "pass0": pass0})
    prev_end = launches[0]["start"]
    for x in launches:
        x["excl"] = x["end"] - prev_end
        x["handoff"] = x["ready"] - prev_end
        prev_end = x["end"]

    def med(name, key):
        v = [x[key] for x in launches if x["name"] == name]
        return round(statistics.median(v) / 1e3, 2)

    names = PROJ + ("attention",)
    return {"launches": launches,
            "gemm_ns": sum(x["excl"] for x in launches if x["name"] != "attention"),
            "attention_ns": sum(x["excl"] for x in launches if x["name"] == "attention"),
            "step_ns": launches[-1]["end"] - launches[0]["start"],
            "excl_us": {**{n: med(n, "excl") for n in names}, "lm_head": med("lm_head", "excl")},
            "handoff_us": {n: med(n, "handoff") for n in names},
            "stream_us": {n: round(statistics.median(x["last_mma"] - x["first_stage"] for x in launches
                                                     if x["name"] == n) / 1e3, 2) for n in PROJ},
            "tail_us": {n: {**{k: round(statistics.median(x[b] - x[a] for x in launches if x["name"] == n) / 1e3, 2)
                               for k, a, b in (("first_stage", "ready", "first_stage"),
                                               ("park_sync", "last_mma", "reduced"), ("rows", "reduced", "rows"),
                                               ("exit", "rows", "end"))},
                            **{k: round(statistics.median(x["pass0"][i] for x in launches
                                                          if x["name"] == n and x["pass0"]) / 1e3, 2)
                               for i, k in enumerate(("rows_sum_first_pass", "rows_write_first_pass"))
                               if any(x["name"] == n and x["pass0"] for x in launches)}}
                        for n in PROJ}}


# ----------------------------------------------------------------------------- the headline (b1)

def run_ours(args, rank, world, dev):
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_TABLE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop

    dev_index = int(os.environ.get("LOCAL_RANK", 0))
    shape = synth.QWEN3_4B if args.layers <= 0 else synth.QWEN3_4B.with_layers(args.layers)
    t_setup = time.time()
    sweep_steps = 8 if args.sweep else 0
    total_steps = 2 * args.warmup + 4 * args.steps + 17 * (sweep_steps + 3) + 16
    max_ctx = CONTEXT + total_steps * 17 + 256
    n_pages = -(-max_ctx // 16) + 8
    v = Verifier(shape, dev, page_size=16, n_pages=n_pages, max_batch=1, max_rows=128, max_span=128,
                 max_context=max_ctx)
    loop = SpecLoop(v, B=1, max_span=K_DRAFT + 1)
    ctx_tokens = workloads.uniform_context(SEED, CONTEXT, shape.vocab)
    loop.prefill([ctx_tokens], chunk=128)
    budget = 10_000_000
    table_len = total_steps * 20 + 64
    table_np = synth.tokens(SEED, "drafts", table_len, shape.vocab)       # uniform-random drafts
    table = torch.as_tensor(table_np).cuda()
    loop.start([budget], k_init=K_DRAFT)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    setup_s = time.time() - t_setup

    seq_len = torch.zeros(1, dtype=torch.int32, device="cuda")

    def cache_len():
        v.cache_seq_len(seq_len)
        torch.cuda.synchronize()
        return int(seq_len[0].item())

    step_kw = dict(drafter=SDV_DRAFT_TABLE, table=table, table_stride=table_len, ngram=False)
    loop.capture(**step_kw)
    for _ in range(args.warmup):
        loop.replay()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(dev_index if world > 1 else None)
    clocks.start()
    L0 = cache_len()
    ctx_start = L0
    s = torch.cuda.current_stream()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")           # profilers can select the timed steps by this range
    ms = timed_replays(loop, args.steps, s)
    torch.cuda.nvtx.range_pop()
    clk = clocks.stop()
    committed = cache_len() - L0
    assert v.get_status() == 0

    # The same step captured with the device timeline on (a few %globaltimer stores per CTA):
    # every launch's first-CTA-start to last-CTA-end inside the graph, PDL overlap included.
    n_regions = 5 * shape.n_layers + 1
    trace_buf = torch.zeros(n_regions * TRACE_REGION_WORDS, dtype=torch.int64, device="cuda")
    v.fwd_trace(trace_buf)
    tloop = SpecLoop(v, B=1, max_span=K_DRAFT + 1)
    tloop.first.copy_(loop.committed[:1])
    tloop.capture(**step_kw)
    v.fwd_trace(None)
    for _ in range(args.warmup):
        tloop.replay()
    trace_buf.zero_()
    traced_ms = timed_replays(tloop, args.steps, s)
    tr = trace_launches(trace_buf, shape.n_layers)
    assert v.get_status() == 0
    del trace_buf

    # per-phase kernel time with each launch group run alone (CUDA events around each group,
    # eager steps): serialised, so it is an upper bound on each kernel's in-graph time
    v.profile_enable(True)
    v.profile_read()
    for _ in range(args.steps):
        loop.step(**step_kw)
    prof = v.profile_read()
    v.profile_enable(False)

    # end to end through host buffers: the step's drafts go up from pinned memory, its result comes back
    pinned_drafts = torch.empty(K_DRAFT, dtype=torch.int32).pin_memory()
    pinned_out = torch.empty(K_DRAFT + 2, dtype=torch.int32).pin_memory()
    e2e_rng = synth.tokens(SEED, "drafts.e2e", args.steps * K_DRAFT, shape.vocab)
    gen = cache_len() - CONTEXT + 1                   # tokens generated so far (the table cursor)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e2e_committed = 0
    for i in range(args.steps):
        pinned_drafts.copy_(torch.from_numpy(e2e_rng[i * K_DRAFT:(i + 1) * K_DRAFT]))
        table[gen:gen + K_DRAFT].copy_(pinned_drafts, non_blocking=True)
        loop.replay()
        pinned_out[:K_DRAFT + 1].copy_(loop.committed[:K_DRAFT + 1], non_blocking=True)
        pinned_out[K_DRAFT + 1:].copy_(loop.n_commit[:1], non_blocking=True)
        s.synchronize()
        n = int(pinned_out[K_DRAFT + 1])
        gen += n
        e2e_committed += n
    e2e_s = time.perf_counter() - t0

    # latency against S = 1..17 (the verify-cost sweep), each S from the configured context: the
    # cache is rewound to CONTEXT positions first (a position rewind, pages past it released)
    sweep = {}
    if args.sweep:
        ctx_len = torch.full((1,), CONTEXT, dtype=torch.int32, device="cuda")
        for S in range(1, 18):
            v.rewind_cache(ctx_len, 1)
            lp = SpecLoop(v, B=1, max_span=S)
            lp.first.copy_(loop.committed[:1])       # continue from the current token
            lp.start([budget], k_init=S - 1)
            lp.capture(drafter=SDV_DRAFT_TABLE, table=table, table_stride=table_len, ngram=False)
            for _ in range(3):
                lp.replay()
            sweep[S] = round(timed_replays(lp, sweep_steps, s) / sweep_steps, 4)
        assert v.get_status() == 0
    ctx_end = cache_len()
    v.close()

    if world > 1:
        committed_all, ms_max, e2e_committed_all, e2e_max = aggregate_replicas(committed, ms, e2e_committed, e2e_s,
                                                                               "cuda")
    else:
        committed_all, ms_max, e2e_committed_all, e2e_max = committed, ms, e2e_committed, e2e_s

    mean_ctx = (ctx_start + ctx_start + committed) / 2
    S = K_DRAFT + 1
    L = shape.n_layers
    step_bytes = (L * (GEMM_BYTES_PER_LAYER + 10_752) + GEMM_BYTES["lm_head"] + 5120
                  + (mean_ctx + S) * KV_BYTES_PER_TOKEN * L / N_LAYERS + S * EMBED_BYTES_PER_ROW)
    peak, peak_kind = peaks()
    # dominant kernel: the weight-streaming GEMM; algorithmic bytes = the weight matrix each launch
    # streams; time = each launch's in-graph span from the device timeline, summed over the step
    gemm_bytes = L * GEMM_BYTES_PER_LAYER + GEMM_BYTES["lm_head"]
    gemm_ns = tr["gemm_ns"]
    n_gemm = 4 * L + 1
    achieved = gemm_bytes / (gemm_ns * 1e-9) / 1e9
    traffic = None
    if args.layers <= 0:
        traffic = round((L * sum(GEMM_TRAFFIC_MB[p] for p in PROJ) + GEMM_TRAFFIC_MB["lm_head"]) * 1e6 / n_gemm / 1e9, 5)
    prof_gemm_ms = sum(prof[p][0] for p in ("qkv_gemm", "o_gemm", "gateup_gemm", "down_gemm", "lmhead_gemm"))
    step_ms = ms_max / args.steps
    attn_launches = -(-S * 4 // 32)                   # query rows (heads x span rows) per launch: 32
    launches_per_step = 3 + L * (4 + attn_launches) + 1 + 2
    out = {
        "metric": "committed tok/s (4B-shape verify, K=7, b1)",
        "value": round(committed_all / (ms_max * 1e-3), 3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded random-init weights and tokens)",
        "config": {"workload": "qwen3-4b-shape verify, batch 1, 848-token context, K=7 (S=8), uniform drafts",
                   "model": "qwen3-4b-shape (random init)", "global_batch": world, "seq_len": CONTEXT,
                   "span": S, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (8.04 GB of weights streamed per step)",
                   "mean_context": round(mean_ctx, 1), "graph": True, "pdl": True},
        "verify_hbm_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
        "step_roofline_frac": round(step_bytes / (step_ms * 1e-3) / 1e9 / peak, 4),
        "step_bytes": int(step_bytes),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "traffic_unit": "GB per launch (ncu dram read + write, 2-layer capture scaled by launch)",
                     "algorithmic": round(gemm_bytes / n_gemm / 1e9, 5),
                     "kernel": "gemm_kernel (tcgen05 weight-streaming GEMM, all projections + LM head)",
                     "timing": ("in-graph, %globaltimer device timeline of the last of K traced steps: each "
                                "GEMM launch's exclusive window (its last CTA end minus the previous "
                                "launch's last CTA end), summed over the 145 GEMM launches"),
                     "peak_kind": f"{peak_kind} (copy bandwidth)",
                     "launches_per_step": n_gemm, "avg_launch_us": round(gemm_ns / n_gemm / 1e3, 2),
                     "gemm_ms_per_step": round(gemm_ns / 1e6, 4),
                     "traced_ms_per_step": round(traced_ms / args.steps, 4),
                     "achieved_serialised": round(gemm_bytes * args.steps / (prof_gemm_ms * 1e-3) / 1e9, 1)},
        "in_graph": {"exclusive_us_per_layer": tr["excl_us"],
                     "handoff_us": tr["handoff_us"],
                     "gemm_stream_us": tr["stream_us"],
                     "gemm_phases_us": tr["tail_us"],
                     "attention_ms_per_step": round(tr["attention_ns"] / 1e6, 4),
                     "traced_step_ms": round(tr["step_ns"] / 1e6, 4),
                     "note": ("exclusive window = a launch's end minus the previous launch's end; handoff "
                              "= first CTA past its wait minus the previous launch's end; stream = first "
                              "stage landed to last MMA issued; phases: first stage after the wait, partial "
                              "parked + cluster barrier after the last MMA, row epilogue, exit (medians "
                              "over layers, latest CTA of each); the row epilogue's first pass of four rows "
                              "per warp, split into summing the split partials and writing the rows "
                              "(medians over CTAs and layers)")},
        "phases_ms_per_step_serialised": {p: round(prof[p][0] / args.steps, 4) for p in prof},
        "e2e": {"value": round(e2e_committed_all / e2e_max, 3), "unit": "tok/s",
                "h2d_bytes_per_step": K_DRAFT * 4, "d2h_bytes_per_step": (K_DRAFT + 2) * 4},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "sweep_ms_per_step": sweep,
        "sweep_context": CONTEXT if args.sweep else None,
        "setup_s": round(setup_s, 1),
        "context_end": ctx_end,
    }
    return out


# ----------------------------------------------------------------------------- further workloads

def _greedy_streams(v, loop, B, first_lens, steps):
    """Run the plain greedy loop (one row per sequence and step) for `steps` steps, record each
    sequence's committed tokens, then rewind every cache to its length before the run."""
    import torch
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NONE
    streams = [[int(t)] for t in loop.first.cpu().tolist()]
    for _ in range(steps):
        loop.step(drafter=SDV_DRAFT_NONE, ngram=False)
        nc = loop.n_commit.cpu().numpy()
        cm = loop.committed.cpu().numpy().reshape(B, loop.max_span)
        for b in range(B):
            streams[b] += cm[b, :nc[b]].tolist()
    v.rewind_cache(torch.as_tensor(np.asarray(first_lens, dtype=np.int32)).cuda(), B)
    torch.cuda.synchronize()
    assert v.get_status() == 0
    return streams


def run_verify_workload(args, name, contexts, seed, dev, steps=None, warmup=None):
    """Verify steps over B sequences whose drafts are the target's own greedy continuation with
    each position replaced by a uniform token with probability 0.3 (mixed acceptance)."""
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_TABLE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    steps = steps or args.steps
    warmup = warmup or args.warmup
    shape = synth.QWEN3_4B if args.layers <= 0 else synth.QWEN3_4B.with_layers(args.layers)
    t_setup = time.time()
    B = len(contexts)
    gen_steps = (warmup + steps) * (K_DRAFT + 1) + 16
    max_ctx = max(len(c) for c in contexts) + gen_steps + 64
    n_pages = sum(-(-(len(c) + gen_steps + 64) // 16) for c in contexts) + 8 * B
    v = Verifier(shape, dev, page_size=16, n_pages=n_pages, max_batch=B, max_rows=128, max_span=128,
                 max_context=max_ctx)
    loop = SpecLoop(v, B=B, max_span=K_DRAFT + 1)
    loop.prefill(contexts, chunk=128)
    lens = [len(c) for c in contexts]
    loop.start([10_000_000] * B, k_init=0)
    streams = _greedy_streams(v, loop, B, lens, gen_steps)
    table_len = gen_steps + 64
    tables = np.stack([workloads.corrupt(seed, b, np.array((streams[b] + [0] * table_len)[:table_len]), 0.3,
                                         shape.vocab) for b in range(B)]).astype(np.int32)
    table = torch.as_tensor(tables.reshape(-1)).cuda()
    loop.start([10_000_000] * B, k_init=K_DRAFT)
    kw = dict(drafter=SDV_DRAFT_TABLE, table=table, table_stride=table_len, ngram=False)
    loop.capture(**kw)
    for _ in range(warmup):
        loop.replay()
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup
    lens_t = torch.zeros(B, dtype=torch.int32, device="cuda")

    def total_len():
        v.cache_seq_len(lens_t)
        torch.cuda.synchronize()
        return int(lens_t.sum().item())

    L0 = total_len()
    clocks = ClockSampler(None)
    clocks.start()
    s = torch.cuda.current_stream()
    ms = timed_replays(loop, steps, s)
    clk = clocks.stop()
    committed = total_len() - L0
    assert v.get_status() == 0
    # the device timeline of a few more steps (graph recaptured with the trace on; the last one read)
    trace_buf = torch.zeros((5 * shape.n_layers + 1) * TRACE_REGION_WORDS, dtype=torch.int64, device="cuda")
    v.fwd_trace(trace_buf)
    loop.capture(**kw)
    v.fwd_trace(None)
    for _ in range(3):
        loop.replay()
    timed_replays(loop, 3, s)
    tr = trace_launches(trace_buf, shape.n_layers)
    assert v.get_status() == 0
    del trace_buf
    v.profile_enable(True)  # per-phase device time (events around each launch group, eager steps)
    v.profile_read()
    n_prof = min(steps, 5)
    for _ in range(n_prof):
        loop.step(**kw)
    prof = v.profile_read()
    v.profile_enable(False)
    v.close()
    mean_ctx = (L0 + L0 + committed) / 2 / B
    step_ms = ms / steps
    S = K_DRAFT + 1
    L = shape.n_layers
    step_bytes = (L * (GEMM_BYTES_PER_LAYER + 10_752) + GEMM_BYTES["lm_head"] + 5120
                  + B * (mean_ctx + S) * KV_BYTES_PER_TOKEN * L / N_LAYERS + B * S * EMBED_BYTES_PER_ROW)
    peak, peak_kind = peaks()
    return {
        "metric": f"committed tok/s (4B-shape verify, K=7, {name})",
        "value": round(committed / (ms * 1e-3), 3), "unit": "tok/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "committed_per_step": round(committed / steps, 3),
        "dtype": "bf16", "data": "synthetic (seeded random-init weights and tokens)",
        "config": {"workload": name, "batch": B, "mean_context": round(mean_ctx, 1), "span": S,
                   "drafts": "greedy continuation, each position uniform-replaced with p=0.3", "graph": True},
        "verify_hbm_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
        "step_roofline_frac": round(step_bytes / (step_ms * 1e-3) / 1e9 / peak, 4),
        "step_bytes": int(step_bytes), "peak_kind": peak_kind, "clocks": clk, "setup_s": round(setup_s, 1),
        "phases_ms_per_step_serialised": {p: round(prof[p][0] / n_prof, 4) for p in prof},
        "in_graph": {"exclusive_us_per_layer": tr["excl_us"], "handoff_us": tr["handoff_us"],
                     "gemm_stream_us": tr["stream_us"], "gemm_phases_us": tr["tail_us"],
                     "attention_ms_per_step": round(tr["attention_ns"] / 1e6, 4),
                     "gemm_ms_per_step": round(tr["gemm_ns"] / 1e6, 4),
                     "traced_step_ms": round(tr["step_ns"] / 1e6, 4)},
    }


def b16_contexts(vocab):
    from synth import workloads
    lens = workloads.context_lengths(3, 16)
    return [workloads.uniform_context(3, int(n), vocab, name=f"b16.ctx.{b}") for b, n in enumerate(lens)]


def run_ngram_workload(args, dev):
    """End-to-end n-gram speculation: 8 prompts of 1024 tokens (32-token spans, half repeating an
    earlier span), 256 greedy tokens each, 2-gram prompt lookup with adaptive K (start 1, +2 on a
    fully accepted round, -1 on any rejection, cap 7), against the same loop without drafts."""
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NGRAM, SDV_DRAFT_NONE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    shape = synth.QWEN3_4B
    B, GEN = 8, 256
    prompts = [workloads.span_repeat_prompt(5 + b, n_spans=32, span=32, vocab=shape.vocab) for b in range(B)]
    out = {}
    for mode in ("spec_off", "spec_on"):
        v = Verifier(shape, dev, page_size=16, n_pages=B * ((1024 + GEN + 64) // 16 + 8), max_batch=B,
                     max_rows=128, max_span=128, max_context=1024 + GEN + 64, ngram_capacity=1024 + GEN + 64)
        loop = SpecLoop(v, B=B, max_span=8)
        loop.prefill(prompts, chunk=128, ngram=(mode == "spec_on"))
        loop.start([GEN] * B, k_init=1 if mode == "spec_on" else 0, adaptive=(mode == "spec_on"), k_max=7)
        kw = dict(drafter=SDV_DRAFT_NGRAM if mode == "spec_on" else SDV_DRAFT_NONE, ngram=(mode == "spec_on"))
        loop.capture(**kw)
        torch.cuda.synchronize()
        lens_t = torch.zeros(B, dtype=torch.int32, device="cuda")
        v.cache_seq_len(lens_t)
        torch.cuda.synchronize()
        L0 = int(lens_t.sum().item())
        s = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s)
        steps = 0
        while True:  # blocks of 16 steps until every sequence has its 256 tokens
            for _ in range(16):
                loop.replay()
            steps += 16
            v.cache_seq_len(lens_t)
            torch.cuda.synchronize()
            if int(lens_t.sum().item()) - L0 >= B * (GEN - 1) or steps > 4 * GEN:
                break
        e1.record(s)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1)
        gen = int(lens_t.sum().item()) - L0 + B      # + the first token of each sequence (from prefill)
        assert v.get_status() == 0
        out[mode] = {"tok_s": round(gen / (ms * 1e-3), 2), "ms": round(ms, 2), "steps": steps, "tokens": gen}
        v.close()
        del v, loop
        torch.cuda.empty_cache()
    return {"metric": "committed tok/s, n-gram spec on vs off (4B shape, b8, 1024-token repeat-heavy prompts, 256 tokens)",
            "value": out["spec_on"]["tok_s"], "unit": "tok/s", "spec_off": out["spec_off"], "spec_on": out["spec_on"],
            "speedup": round(out["spec_on"]["tok_s"] / out["spec_off"]["tok_s"], 3),
            "note": "steps run in blocks of 16 between host checks; idle steps after the budget count in the time"}


# ----------------------------------------------------------------------------- the oracle on the host cores

def _cores():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_verify_steps(n_steps, n_warmup):
    """The CPU oracle, as it stands, on the headline workload: whole S=8 verify steps of the
    36-layer 4B shape over an 848-token cache (synthetic cache contents; the weights are generated
    before timing). Each step is timed alone. Returns (seconds per timed step, cores)."""
    import oracle
    import synth
    from synth import workloads
    shape = synth.QWEN3_4B
    host = {n: synth.tensor(shape, SEED, n) for n in shape.tensor_shapes()}
    model = oracle.DenseDecoder(shape, lambda n: host[n], cache_weights=False)
    cache = oracle.SeqCache(shape, CONTEXT + 16)
    rng = np.random.default_rng(0)
    for l in range(shape.n_layers):
        cache.K[l][:CONTEXT] = rng.standard_normal(cache.K[l][:CONTEXT].shape)
        cache.V[l][:CONTEXT] = rng.standard_normal(cache.V[l][:CONTEXT].shape)
    span = workloads.uniform_drafts(SEED, 0, K_DRAFT + 1, shape.vocab)
    ts = []
    for i in range(n_warmup + n_steps):
        cache.length = CONTEXT
        t0 = time.perf_counter()
        model.forward([cache], [span])
        if i >= n_warmup:
            ts.append(time.perf_counter() - t0)
    return ts, _cores()


def oracle_tiny_generation():
    """Config 1 end to end in the oracle: the tiny decoder, a 128-token motif prompt, 2-gram
    drafts at fixed K = 4, 32 greedy tokens. Returns (seconds, committed tokens)."""
    import oracle
    import synth
    from synth import workloads
    shape = synth.TINY
    host = {n: synth.tensor(shape, 1, n) for n in shape.tensor_shapes()}
    model = oracle.DenseDecoder(shape, lambda n: host[n])
    t0 = time.perf_counter()
    streams, _, _ = oracle.generate(model, [workloads.motif_prompt(1)], 32, drafter="ngram", k=4)
    return time.perf_counter() - t0, len(streams[0])


def cpu_child(kind):
    """Entry of the child process that times the oracle (a fresh interpreter: no CUDA context,
    no torch thread pools competing with the BLAS threads)."""
    if kind == "verify":
        ts, cores = oracle_verify_steps(1, 0)
        print(json.dumps({"step_s": ts[0], "cores": cores}))
    elif kind == "tiny":
        s, n = oracle_tiny_generation()
        print(json.dumps({"seconds": s, "tokens": n, "cores": int(os.environ.get("OPENBLAS_NUM_THREADS", _cores()))}))


def spawn_cpu_child(kind, threads=None, timeout=900):
    env = dict(os.environ)
    if threads is not None:
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            env[k] = str(threads)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-child", kind], env=env,
                       capture_output=True, text=True, timeout=timeout)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline():
    """The oracle timed on the host cores, each figure in a fresh process."""
    step = spawn_cpu_child("verify")
    tiny_all = spawn_cpu_child("tiny")
    tiny_one = spawn_cpu_child("tiny", threads=1)
    out = {"unit": "tok/s", "kind": "oracle"}
    if "step_s" in step:
        out.update({"value": round(1.0 / step["step_s"], 6), "cores": step["cores"],
                    "sample": (f"one whole S=8 verify step of the 36-layer 4B shape over an 848-token cache "
                               f"(1 committed token at uniform drafts), timed alone in a fresh process: "
                               f"{step['step_s']:.2f} s; BLAS on {step['cores']} threads, the oracle's "
                               f"bf16-to-float64 weight conversion on one")})
    else:
        out.update({"value": None, "cores": _cores(), "sample": f"oracle step failed: {step['error']}"})
    if "seconds" in tiny_all and "seconds" in tiny_one:
        out["tiny_config_e2e"] = {"workload": "tiny decoder, 128-token motif prompt, 2-gram K=4, 32 tokens",
                                  "s_all_threads": round(tiny_all["seconds"], 3), "threads": tiny_all["cores"],
                                  "s_one_thread": round(tiny_one["seconds"], 3)}
    return out


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on the headline workload, W warm-up and K
    timed whole verify steps (36 layers, S = 8) on the host cores."""
    if rank != 0:
        return None
    ts, cores = oracle_verify_steps(args.steps, args.warmup)
    mean = sum(ts) / len(ts)
    value = 1.0 / mean               # uniform drafts: one committed token per verify step
    sample = (f"per step: one whole S=8 verify of the 36-layer 4B shape over an 848-token cache, each step "
              f"timed alone (min {min(ts):.2f} s, max {max(ts):.2f} s)")
    return {
        "impl": "reference",
        "metric": "committed tok/s (4B-shape verify, K=7, b1)",
        "value": round(value, 6), "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 1), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": "qwen3-4b-shape verify, batch 1, 848-token context, K=7 (S=8), uniform drafts"},
        "cpu_baseline": {"value": round(value, 6), "unit": "tok/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--no-extra", dest="extra", action="store_false",
                    help="skip the batch-16 and 32K-context sub-objects of the headline line")
    ap.add_argument("--workload", default="b1", choices=["b1", "b16", "ctx32k", "ngram"],
                    help="b1 (default, the headline line): batch 1, 848-token context; b16: 16 sequences with "
                         "contexts U[512, 4096]; ctx32k: batch 1, 32768-token context; ngram: end-to-end 2-gram "
                         "speculation against the same loop without drafts")
    ap.add_argument("--layers", type=int, default=0,
                    help="decoder layers (default: all 36); fewer only for small profiling cases")
    ap.add_argument("--cpu-child", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.cpu_child:
        cpu_child(args.cpu_child)
        return
    args.warmup = max(args.warmup, 3)
    rank, local, world = dist_env()

    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return

    import torch
    import synth
    torch.cuda.set_device(local)
    shape = synth.QWEN3_4B if args.layers <= 0 else synth.QWEN3_4B.with_layers(args.layers)
    if args.workload != "b1":
        if rank == 0:  # single-GPU measurement lines for the other workloads
            from synth import workloads
            dev = build_weights(shape, SEED)
            if args.workload == "b16":
                out = run_verify_workload(args, "qwen3-4b-shape verify, batch 16, contexts U[512, 4096], K=7",
                                          b16_contexts(shape.vocab), 3, dev)
            elif args.workload == "ctx32k":
                out = run_verify_workload(args, "qwen3-4b-shape verify, batch 1, 32768-token context, K=7",
                                          [workloads.uniform_context(4, 32768, shape.vocab)], 4, dev)
            else:
                out = run_ngram_workload(args, dev)
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = build_weights(shape, SEED)
    out = run_ours(args, rank, world, dev)
    if rank == 0 and world == 1 and args.extra:
        from synth import workloads
        steps, warm = min(args.steps, 20), 3
        for key, name, ctxs, seed in (
                ("b16", "qwen3-4b-shape verify, batch 16, contexts U[512, 4096], K=7", b16_contexts(shape.vocab), 3),
                ("ctx32k", "qwen3-4b-shape verify, batch 1, 32768-token context, K=7",
                 [workloads.uniform_context(4, 32768, shape.vocab)], 4)):
            r = run_verify_workload(args, name, ctxs, seed, dev, steps=steps, warmup=warm)
            out[key] = {k: r[k] for k in ("value", "unit", "ms_per_step", "committed_per_step", "steps", "warmup",
                                          "verify_hbm_gbs", "step_roofline_frac", "step_bytes", "clocks")}
            out[key]["config"] = r["config"]
            out[key]["phases_ms_per_step_serialised"] = r["phases_ms_per_step_serialised"]
            out[key]["in_graph"] = r["in_graph"]
            torch.cuda.empty_cache()
    if rank == 0:
        if args.cpu_baseline and world == 1:
            out["cpu_baseline"] = cpu_baseline()
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
