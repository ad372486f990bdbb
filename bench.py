#!/usr/bin/env python
"""Benchmark of the speculative-decoding verify transaction on one GB300.

Workload (default): Qwen3-4B-shaped decoder (36 layers, hidden 2560, 32/8 heads
of 128, FFN 9728, vocab 151936, bf16 weights N(0, 0.02) from seed 2), batch 1,
848 uniform-random context tokens prefilled into the paged KV (page 16), then
verify steps of S = K+1 = 8 rows with uniform-random drafts. A step is the
whole hot path: propose -> ensure_capacity -> spec_forward (verify) ->
accept_greedy -> rewind_cache, replayed as one CUDA graph.

Metric: committed tokens/s (whole job, all GPUs). Also reported: ms per step,
the per-S latency sweep (S = 1..17), the HBM roofline of the dominant kernel
(the tcgen05 weight-streaming GEMM), the end-to-end figure through host
buffers, and the CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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
WEIGHT_BYTES_PER_STEP = 8_044_936_192      # 36 layers + LM head + final norm (bf16)
KV_BYTES_PER_TOKEN = 147_456               # 2 (K,V) x 8 heads x 128 x 2 B x 36 layers
# DRAM bytes (read + write) that ncu measured per launch of the weight-streaming GEMM on the
# per-projection path, in a 2-layer case of the same shapes (every launch of two timed steps):
# QKV, O, gate/up, down per layer, then the LM head.
# A launch streams its own weights, so a 36-layer step is 36 layers of the first four plus one
# LM head; divided by the 145 launches it is the per-launch traffic beside `achieved`.
GEMM_TRAFFIC_MB = {"qkv": 31.6998, "o": 21.3698, "gate_up": 99.9877, "down": 50.5655, "lm_head": 778.2215}
GEMM_TRAFFIC_PER_LAUNCH = (36 * (GEMM_TRAFFIC_MB["qkv"] + GEMM_TRAFFIC_MB["o"] + GEMM_TRAFFIC_MB["gate_up"] +
                                 GEMM_TRAFFIC_MB["down"]) + GEMM_TRAFFIC_MB["lm_head"]) * 1e6 / 145
EMBED_BYTES_PER_ROW = 2560 * 2


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

    def __init__(self, gpu_index: int):
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


# ----------------------------------------------------------------------------- our implementation

def build_weights(shape, seed, device="cuda"):
    import synth
    from speculative_decoding_verify_02_gb300 import upload_bf16
    host, dev = {}, {}
    for name in shape.tensor_shapes():
        host[name] = synth.tensor(shape, seed, name)
        dev[name] = upload_bf16(host[name], device)
    return host, dev


def run_ours(args, rank, world):
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_TABLE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop

    dev_index = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev_index)
    shape = synth.QWEN3_4B if args.layers <= 0 else synth.QWEN3_4B.with_layers(args.layers)
    t_setup = time.time()
    host, dev = build_weights(shape, SEED)
    sweep_steps = 8 if args.sweep else 0
    total_steps = args.warmup + args.steps + 2 * args.steps + 17 * (sweep_steps + 3) + 16
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed")           # profilers can select the timed steps by this range
    e0.record(s)
    for _ in range(args.steps):
        loop.replay()
    e1.record(s)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    committed = cache_len() - L0
    assert v.get_status() == 0

    # live per-phase kernel timing (events around each launch group, same workload)
    v.profile_enable(True)
    v.profile_read()
    prof_ctx0 = cache_len()
    for _ in range(args.steps):
        loop.step(**step_kw)
    prof = v.profile_read()
    prof_ctx = (prof_ctx0 + cache_len()) / 2
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
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            for _ in range(sweep_steps):
                lp.replay()
            b.record(s)
            torch.cuda.synchronize()
            sweep[S] = round(a.elapsed_time(b) / sweep_steps, 4)
        assert v.get_status() == 0
    ctx_end = cache_len()

    # aggregate over ranks: tokens summed, time = max
    if world > 1:
        committed_all, ms_max, e2e_committed_all, e2e_max = aggregate_replicas(committed, ms, e2e_committed, e2e_s,
                                                                               "cuda")
    else:
        committed_all, ms_max, e2e_committed_all, e2e_max = committed, ms, e2e_committed, e2e_s

    mean_ctx = (ctx_start + ctx_start + committed) / 2
    S = K_DRAFT + 1
    step_bytes = WEIGHT_BYTES_PER_STEP + (mean_ctx + S) * KV_BYTES_PER_TOKEN + S * EMBED_BYTES_PER_ROW
    peak, peak_kind = peaks()
    # dominant kernel: the weight-streaming GEMM (every projection and the LM head)
    gemm_phases = ("qkv_gemm", "o_gemm", "gateup_gemm", "down_gemm", "lmhead_gemm")
    dom_ms = sum(prof[p][0] for p in gemm_phases)
    dom_launches = sum(prof[p][1] for p in gemm_phases)
    dom_bytes = WEIGHT_BYTES_PER_STEP * args.steps + S * 2560 * 2 * 5 * 36 * args.steps
    dom_name = "gemm_kernel (tcgen05 weight-streaming GEMM, all projections + LM head)"
    launches_per_step = 4 + 2 + 36 * (1 + 2 + 3)
    dom_traffic = None
    if args.layers <= 0 and dom_launches == 145 * args.steps:
        dom_traffic = round(GEMM_TRAFFIC_PER_LAUNCH / 1e9, 5)   # GB per launch, as `achieved` per second
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    step_ms = ms_max / args.steps
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
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": dom_traffic,
                     "traffic_unit": "GB per launch (ncu dram read + write)",
                     "algorithmic": round(dom_bytes / max(dom_launches, 1) / 1e9, 5),
                     "kernel": dom_name,
                     "peak_kind": f"{peak_kind} (burst copy; each launch timed alone)",
                     "launches": dom_launches, "avg_launch_us": round(dom_ms * 1e3 / max(dom_launches, 1), 2)},
        "phases_ms_per_step": {p: round(prof[p][0] / args.steps, 4) for p in prof},
        "e2e": {"value": round(e2e_committed_all / e2e_max, 3), "unit": "tok/s",
                "h2d_bytes_per_step": K_DRAFT * 4, "d2h_bytes_per_step": (K_DRAFT + 2) * 4},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
        "sweep_ms_per_step": sweep,
        "sweep_context": CONTEXT if args.sweep else None,
        "setup_s": round(setup_s, 1),
        "context_end": ctx_end,
    }
    return out, host


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


def run_verify_workload(args, name, contexts, seed):
    """Verify steps over B sequences whose drafts are the target's own greedy continuation with
    each position replaced by a uniform token with probability 0.3 (mixed acceptance)."""
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_TABLE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    shape = synth.QWEN3_4B if args.layers <= 0 else synth.QWEN3_4B.with_layers(args.layers)
    t_setup = time.time()
    host, dev = build_weights(shape, SEED)
    B = len(contexts)
    gen_steps = (args.warmup + args.steps) * (K_DRAFT + 1) + 16
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
    for _ in range(args.warmup):
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
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(args.steps):
        loop.replay()
    e1.record(s)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    committed = total_len() - L0
    assert v.get_status() == 0
    v.profile_enable(True)  # per-phase device time (events around each launch group, eager steps)
    v.profile_read()
    for _ in range(min(args.steps, 5)):
        loop.step(**kw)
    prof = v.profile_read()
    v.profile_enable(False)
    n_prof = min(args.steps, 5)
    mean_ctx = (L0 + L0 + committed) / 2 / B
    step_ms = ms / args.steps
    S = K_DRAFT + 1
    step_bytes = WEIGHT_BYTES_PER_STEP + B * (mean_ctx + S) * KV_BYTES_PER_TOKEN + B * S * EMBED_BYTES_PER_ROW
    peak, peak_kind = peaks()
    return {
        "metric": f"committed tok/s (4B-shape verify, K=7, {name})",
        "value": round(committed / (ms * 1e-3), 3), "unit": "tok/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "committed_per_step": round(committed / args.steps, 3),
        "dtype": "bf16", "data": "synthetic (seeded random-init weights and tokens)",
        "config": {"workload": name, "batch": B, "mean_context": round(mean_ctx, 1), "span": S,
                   "drafts": "greedy continuation, each position uniform-replaced with p=0.3", "graph": True},
        "verify_hbm_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
        "step_roofline_frac": round(step_bytes / (step_ms * 1e-3) / 1e9 / peak, 4),
        "step_bytes": int(step_bytes), "peak_kind": peak_kind, "clocks": clk, "setup_s": round(setup_s, 1),
        "phases_ms_per_step": {p: round(prof[p][0] / n_prof, 4) for p in prof},
    }


def run_ngram_workload(args):
    """End-to-end n-gram speculation: 8 prompts of 1024 tokens (32-token spans, half repeating an
    earlier span), 256 greedy tokens each, 2-gram prompt lookup with adaptive K (start 1, +2 on a
    fully accepted round, -1 on any rejection, cap 7), against the same loop without drafts."""
    import torch
    import synth
    from synth import workloads
    from speculative_decoding_verify_02_gb300 import SDV_DRAFT_NGRAM, SDV_DRAFT_NONE, Verifier
    from speculative_decoding_verify_02_gb300.runner import SpecLoop
    shape = synth.QWEN3_4B
    host, dev = build_weights(shape, SEED)
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
        del v, loop
        torch.cuda.empty_cache()
    return {"metric": "committed tok/s, n-gram spec on vs off (4B shape, b8, 1024-token repeat-heavy prompts, 256 tokens)",
            "value": out["spec_on"]["tok_s"], "unit": "tok/s", "spec_off": out["spec_off"], "spec_on": out["spec_on"],
            "speedup": round(out["spec_on"]["tok_s"] / out["spec_off"]["tok_s"], 3),
            "note": "steps run in blocks of 16 between host checks; idle steps after the budget count in the time"}


# ----------------------------------------------------------------------------- the oracle on the host cores

def oracle_step_sample(host=None, n_layers_sample=1):
    """Time the CPU oracle on a bounded sample of one S=8 verify step over an
    848-token cache: n_layers_sample decoder layers plus the final norm and LM
    head, with synthetic cache contents (timing only). The full step is
    estimated as 36 x (time per layer) + (LM-head time)."""
    import oracle
    import synth
    from synth import workloads
    shape = synth.QWEN3_4B
    sample_shape = shape.with_layers(n_layers_sample)
    if host is None:
        host = {}

    def get(n):
        if n not in host:
            host[n] = synth.tensor(shape, SEED, n)
        return host[n]

    model = oracle.DenseDecoder(sample_shape, get, cache_weights=False)
    cache = oracle.SeqCache(sample_shape, CONTEXT + 16)
    rng = np.random.default_rng(0)
    for l in range(n_layers_sample):
        cache.K[l][:CONTEXT] = rng.standard_normal(cache.K[l][:CONTEXT].shape)
        cache.V[l][:CONTEXT] = rng.standard_normal(cache.V[l][:CONTEXT].shape)
    cache.length = CONTEXT
    span = workloads.uniform_drafts(SEED, 0, K_DRAFT + 1, shape.vocab)
    t0 = time.perf_counter()
    model.forward([cache], [span])
    t_total = time.perf_counter() - t0
    # split the sample into layer time and head time
    y = np.zeros((K_DRAFT + 1, shape.hidden))
    t1 = time.perf_counter()
    oracle.rmsnorm(y, model.w("final_norm"), shape.rms_eps) @ model.w("lm_head").T
    t_head = time.perf_counter() - t1
    t_layer = max(t_total - t_head, 1e-6) / n_layers_sample
    t_step = shape.n_layers * t_layer + t_head
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    return t_step, t_total + t_head, cores


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle, as it stands, on the same workload."""
    if rank != 0:
        return None
    import synth
    ts = []
    host = {}
    for i in range(args.warmup + args.steps):
        t_step, _, cores = oracle_step_sample(host)
        if i >= args.warmup:
            ts.append(t_step)
    mean = sum(ts) / len(ts)
    value = 1.0 / mean               # uniform drafts: one committed token per verify step
    sample = (f"per step: one S=8 verify of the 4B shape over an 848-token cache, 1 decoder layer + final norm "
              f"+ LM head computed, full step = 36 x layer + head")
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
    ap.add_argument("--workload", default="b1", choices=["b1", "b16", "ctx32k", "ngram"],
                    help="b1 (default, the headline line): batch 1, 848-token context; b16: 16 sequences with "
                         "contexts U[512, 4096]; ctx32k: batch 1, 32768-token context; ngram: end-to-end 2-gram "
                         "speculation against the same loop without drafts")
    ap.add_argument("--layers", type=int, default=0,
                    help="decoder layers (default: all 36); fewer only for small profiling cases")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, local, world = dist_env()

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
        out = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(out), flush=True)
        return

    import torch
    if args.workload != "b1":
        if rank == 0:  # single-GPU measurement lines for the other workloads
            import synth
            from synth import workloads
            vocab = synth.QWEN3_4B.vocab
            if args.workload == "b16":
                lens = workloads.context_lengths(3, 16)
                ctxs = [workloads.uniform_context(3, int(n), vocab, name=f"b16.ctx.{b}") for b, n in enumerate(lens)]
                out = run_verify_workload(args, "qwen3-4b-shape verify, batch 16, contexts U[512, 4096], K=7", ctxs, 3)
            elif args.workload == "ctx32k":
                ctxs = [workloads.uniform_context(4, 32768, vocab)]
                out = run_verify_workload(args, "qwen3-4b-shape verify, batch 1, 32768-token context, K=7", ctxs, 4)
            else:
                out = run_ngram_workload(args)
            print(json.dumps(out), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    out, host = run_ours(args, rank, world)
    if rank == 0:
        if args.cpu_baseline and world == 1:
            t_step, spent, cores = oracle_step_sample(host)
            out["cpu_baseline"] = {"value": round(1.0 / t_step, 6), "unit": "tok/s", "cores": cores, "kind": "oracle",
                                   "sample": (f"one S=8 verify of the 4B shape over an 848-token cache: 1 decoder "
                                              f"layer + final norm + LM head computed in {spent:.1f} s, full step "
                                              f"estimated as 36 x layer + head = {t_step:.1f} s")}
        print(json.dumps(out), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
