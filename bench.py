"""Benchmark of one CSA2 layer step on GB300.

A step is one pass of the whole hot path over one batch: compress of the
groups that close at this step, index scores over every visible compressed
entry, top-512 selection, and the two-source attention with sink. The
headline workload is decode at batch 32 with 65,536-token contexts
(ratio 4 -> 16,384 compressed entries per sequence), bf16, seeded synthetic
inputs. Units are query tokens: tokens/s = 32 * steps / time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

Under torchrun each rank runs its own batch (data-parallel over sequences,
no collective on the data path); the line reports the whole-job rate over the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import PRESETS, make_inputs  # noqa: E402

METRIC = "CSA2 decode tokens/s and HBM GB/s (% of ~8 TB/s) at 64K and 1M context"
N_COPIES = 4  # rotating input copies: each step's working set is evicted from L2 by the other three
# dram bytes read + written by one index_score launch on decode_64k_b32, from the
# ncu capture summarised in profiles/index_score_decode_64k_b32.md (same kernel)
INDEX_TRAFFIC_BYTES = 134_319_616 + 3_283_456


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        t0, t1 = (self.marks[0], self.marks[1]) if len(self.marks) >= 2 else (0, 1e30)
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        use = inside if inside else self.samples
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, line in use:
            parts = [p.strip() for p in line.split(",")]
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except Exception:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(use), "in_timed_region": bool(inside)}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device):
    if pg is not None:
        if device.type == "cuda":
            pg.barrier(device_ids=[device.index])
        else:
            pg.barrier()


def aggregate_value(world: int, units_per_step: int, steps: int, ms_max: float) -> float:
    """Whole-job throughput under weak scaling: every rank processed its own
    units_per_step each step; the job took the slowest rank's time."""
    return world * units_per_step * steps / (ms_max / 1000.0)


def max_over_ranks(pg, x: float, device) -> float:
    if pg is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device if device.type == "cuda" else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workload bytes

# bytes of one stored row (codes + scales) per storage format code
_ROW_BYTES = {0: 1024, 1: 512 + 16, 2: 256 + 32}     # 512-channel rows: bf16, fp8 (ue8m0 / 32), fp4 (e4m3 / 16)
_KEY_BYTES = {0: 256, 1: 128 + 4, 3: 64 + 4}         # 128-channel keys: bf16, fp8, mxfp4 (e8m0 / 32)


def row_bytes(wl):
    """(window row, pool row, index key) bytes; an fp4 pool keeps an fp8 window."""
    win = _ROW_BYTES[1] if wl.kv_fp8 else _ROW_BYTES[0]
    return win, _ROW_BYTES[wl.kv_format], _KEY_BYTES[wl.idx_key_format]


def algorithmic_bytes(wl, has_compress=True):
    """Minimal HBM bytes of one step: every visible index key once, the gathered
    window and selected rows once, q/q^I/w in, the output out, and the closing
    groups' raw tokens and gates in plus their stored entries out."""
    wrow, prow, key = row_bytes(wl)
    total = 0
    for b in range(wl.n_seq):
        n = wl.ctx_len[b]
        for i in range(wl.n_query_per_seq):
            t = n - wl.n_query_per_seq + i
            nv = (t + 1) // wl.m
            win = min(wl.window, t + 1)
            total += nv * key + win * wrow + min(wl.topk, nv) * prow
            total += wl.n_heads * wl.head_dim * 2 * 2 + wl.idx_heads * wl.idx_dim * 2 + wl.idx_heads * 4
        if has_compress and n % wl.m == 0:
            total += wl.m * wl.head_dim * (2 + 4) + prow + key
    return total


def kv_format_name(wl):
    if not wl.kv_fp8:
        return "bf16"
    pool = "fp4_e2m1_e4m3_b16 pool, fp8 window" if wl.pool_fp4 else "fp8_e4m3_ue8m0_b32"
    keys = "mxfp4_e2m1_ue8m0_b32 keys" if wl.key_fp4 else ("fp8 keys" if wl.idx_fp8 else "bf16 keys")
    return f"{pool}; {keys}"


def index_bytes(wl):
    key = row_bytes(wl)[2]
    tot = 0
    for b in range(wl.n_seq):
        n = wl.ctx_len[b]
        for i in range(wl.n_query_per_seq):
            t = n - wl.n_query_per_seq + i
            nv = (t + 1) // wl.m
            tot += nv * (key + 4) + wl.idx_heads * wl.idx_dim * 2 + wl.idx_heads * 4
    return tot


# ----------------------------------------------------------------------------- GPU arm

class Copy:
    """One resident copy of a step's inputs and outputs."""

    def __init__(self, ctx, wl, seed_offset, device):
        from compressed_sparse_attention_gb300 import binding
        wlc = wl.scaled(seed=wl.seed + 1000 * seed_offset)
        inp = make_inputs(wlc, device)

        def store(x, fmt):
            dim = x.shape[1]
            blk = 16 if fmt == binding.KV_FP4 else 32
            codes = torch.empty((x.shape[0], dim if fmt == binding.KV_FP8 else dim // 2), dtype=torch.uint8,
                                device=device)
            sc = torch.empty((x.shape[0], dim // blk), dtype=torch.uint8, device=device)
            for i in range(0, x.shape[0], 1 << 20):
                ctx.store_rows(x[i:i + (1 << 20)], None, fmt, codes[i:i + (1 << 20)], sc[i:i + (1 << 20)])
            return codes, sc

        if wl.kv_fp8:
            inp["win_kv"], inp["win_scale"] = store(inp.pop("win_kv_f32"), binding.KV_FP8)
            inp["pool_kv"], inp["pool_scale"] = store(inp.pop("pool_kv_f32"), wl.kv_format)
        if wl.idx_fp8:
            inp["idx_keys"], inp["idx_key_scale"] = store(inp.pop("idx_keys_f32"), wl.idx_key_format)
        torch.cuda.synchronize()
        self.inp = inp
        Q = wl.n_query
        self.max_vis = int(inp["n_vis"].max())
        self.out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=device)
        self.idx = torch.empty((Q, wl.topk), dtype=torch.int32, device=device)
        self.ws = binding.workspace(ctx.step_workspace_size(Q, self.max_vis), device)
        self.scores = torch.empty((Q, self.max_vis), dtype=torch.float32, device=device)
        self.wl = wl

    def step_kwargs(self, q=None, raw=None, gate=None, out=None):
        i = self.inp
        return dict(q=i["q"] if q is None else q, q_pos=i["q_pos"], seq_of_q=i["seq_of_q"], n_vis=i["n_vis"],
                    sink=i["sink"], win_kv=i["win_kv"], win_scale=i.get("win_scale"), win_off=i["win_off"],
                    pool_kv=i["pool_kv"], pool_scale=i.get("pool_scale"), pool_off=i["pool_off"],
                    topk_idx=self.idx, out=self.out if out is None else out, workspace=self.ws, q_idx=i["q_idx"],
                    w_heads=i["w_heads"], idx_keys=i["idx_keys"], idx_key_scale=i.get("idx_key_scale"),
                    raw=i["raw"] if raw is None else raw, gate=i["gate"] if gate is None else gate,
                    tok_off=i["tok_off"], first_pos=i["first_pos"], norm_w=i["norm_w"], w_idx=i["w_idx"],
                    k_norm_w=i["k_norm_w"])

    def step(self, ctx, q=None, raw=None, gate=None, out=None):
        ctx.step(0, self.wl.n_seq, self.max_vis, **self.step_kwargs(q, raw, gate, out))

    def step_as(self, ctx, mode, cand_role=0, cand=None):
        """A Full or Reindex step of this copy, optionally as the hierarchical
        indexer's candidate source (cand_role 1) or pool reader (2)."""
        i = self.inp
        full = mode == 0
        ctx.step(mode, self.wl.n_seq, self.max_vis, q=i["q"], q_pos=i["q_pos"], seq_of_q=i["seq_of_q"],
                 n_vis=i["n_vis"], sink=i["sink"], win_kv=i["win_kv"], win_scale=i.get("win_scale"),
                 win_off=i["win_off"], pool_kv=i["pool_kv"], pool_scale=i.get("pool_scale"), pool_off=i["pool_off"],
                 topk_idx=self.idx, out=self.out, workspace=self.ws, q_idx=i["q_idx"], w_heads=i["w_heads"],
                 idx_keys=i["idx_keys"], idx_key_scale=i.get("idx_key_scale"), raw=i["raw"] if full else None,
                 gate=i["gate"] if full else None, tok_off=i["tok_off"] if full else None,
                 first_pos=i["first_pos"] if full else None, norm_w=i["norm_w"] if full else None,
                 w_idx=i["w_idx"] if full else None, k_norm_w=i["k_norm_w"] if full else None, cand_role=cand_role,
                 cand=cand)

    def attend_only(self, ctx, ws):
        """Attention alone on this copy's last selection (decode or prefill)."""
        i = self.inp
        ctx.attend(self.wl.n_seq, i["q"], i["q_pos"], i["seq_of_q"], i["win_kv"], i.get("win_scale"), i["win_off"],
                   None, i["pool_kv"], i.get("pool_scale"), i["pool_off"], self.idx, i["sink"], self.out, None, ws)

    def index_only(self, ctx):
        i = self.inp
        ctx.index_score(self.wl.n_seq, i["q_idx"], i["w_heads"], i["idx_keys"], i.get("idx_key_scale"),
                        i["pool_off"], i["seq_of_q"], i["n_vis"], self.max_vis, self.scores)


def run_gpu_workload(args, wl, rank, pg, device, peaks, sampler=None):
    from compressed_sparse_attention_gb300 import binding, build
    build.build()
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads, kv_format=wl.kv_format,
                          idx_key_format=wl.idx_key_format)
    copies = [Copy(ctx, wl, rank * N_COPIES + c, device) for c in range(N_COPIES)]
    stream = torch.cuda.Stream(device=device)
    # launches per step
    with torch.cuda.stream(stream):
        copies[0].step(ctx)
    launches_per_step = ctx.last_launch_count
    torch.cuda.synchronize()
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the bench workload")
    # one CUDA graph per copy, and one that runs the N_COPIES steps in turn
    # (as a serving loop captures consecutive layers): the timed region
    # replays the latter, so the graph launch cost is shared by four steps
    graphs = []
    for c in copies:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            c.step(ctx)
        graphs.append(g)
    g_all = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_all, stream=stream):
        for c in copies:
            c.step(ctx)
    torch.cuda.synchronize()
    for i in range(max(args.warmup, 3)):
        graphs[i % N_COPIES].replay()
    torch.cuda.synchronize()
    # ---- timed region: exactly K steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(pg, device)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps // N_COPIES):
            g_all.replay()
        for i in range(args.steps % N_COPIES):
            graphs[i].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark()
    barrier(pg, device)
    ms = e0.elapsed_time(e1)
    ms_max = max_over_ranks(pg, ms, device)
    # ---- the same region's replays timed one by one: median per step
    n_rep = 64
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record(stream)
            g_all.replay()
            b.record(stream)
    torch.cuda.synchronize()
    rep_ms = sorted(a.elapsed_time(b) / N_COPIES for a, b in ev)
    ms_median = statistics.median(rep_ms)
    # ---- dominant kernel (index score) timed alone, on its launch stream
    n_idx = max(args.steps, 20)
    with torch.cuda.stream(stream):
        for i in range(3):
            copies[i % N_COPIES].index_only(ctx)
        torch.cuda.synchronize()
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for i in range(n_idx):
            copies[i % N_COPIES].index_only(ctx)
        k1.record(stream)
    torch.cuda.synchronize()
    idx_ms = k0.elapsed_time(k1) / n_idx
    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, ctx, copies, stream, device, wl)
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} after timing")
    return dict(ms=ms, ms_max=ms_max, launches=launches_per_step, idx_ms=idx_ms, e2e=e2e, ms_median=ms_median,
                n_rep=n_rep)


def attention_flops(wl) -> float:
    """QK^T + PV flops of one step: per query, 2 x rows x 64 heads x 512 dims
    for each product, rows = window rows + selected entries."""
    tot = 0
    for b in range(wl.n_seq):
        for i in range(wl.n_query_per_seq):
            t = wl.ctx_len[b] - wl.n_query_per_seq + i
            rows = min(wl.window, t + 1) + min(wl.topk, (t + 1) // wl.m)
            tot += 2 * 2 * rows * wl.n_heads * wl.head_dim
    return float(tot)


def run_prefill_extra(args, device, bf16_peak):
    """The chunked-prefill workload: the whole step (graph), and the attention
    alone (its QK^T and PV contractions against the bf16 tensor peak)."""
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS["prefill_4k_after_8k"]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads)
    copies = [Copy(ctx, wl, c, device) for c in range(2)]  # q alone is 256 MB per copy, > L2
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        for c in copies:
            c.step(ctx)
    torch.cuda.synchronize()
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the prefill workload")
    ws = [binding.workspace(ctx.attend_workspace_size(wl.n_query), device) for _ in copies]
    steps = max(3, min(args.steps, 20))

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                fn(i)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_step = timed(lambda i: copies[i % 2].step(ctx))
    ms_att = timed(lambda i: copies[i % 2].attend_only(ctx, ws[i % 2]))
    flops = attention_flops(wl)
    tf = flops / (ms_att / 1000.0) / 1e12
    return {"workload": wl.name, "queries": wl.n_query, "tokens_per_s": wl.n_query / (ms_step / 1000.0),
            "ms_per_step": ms_step, "attend_ms": ms_att, "attend_flops": flops,
            "roofline_attend": {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s",
                                "frac": tf / bf16_peak, "peak_kind": "bf16 dense, burst (kernel timed alone)"}}


def run_tiny_extra(args, device):
    """Latency of one CSA2 layer step on the tiny decode workload (batch 1,
    4,096 context, ratio 4 -> 1,024 entries): one CUDA graph per step, each
    replay timed alone, median and spread. Its ~1 MB working set stays in L2,
    as it would from step to step of a real decode."""
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS["tiny_decode"]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads)
    c = Copy(ctx, wl, 0, device)
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        c.step(ctx)
    torch.cuda.synchronize()
    launches = ctx.last_launch_count
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the tiny workload")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        c.step(ctx)
    n = 200
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    with torch.cuda.stream(stream):
        for _ in range(10):
            g.replay()
        for a, b in ev:
            a.record(stream)
            g.replay()
            b.record(stream)
    torch.cuda.synchronize()
    us = sorted(1000.0 * a.elapsed_time(b) for a, b in ev)
    return {"workload": wl.name, "us_per_step_median": statistics.median(us), "us_p10": us[n // 10],
            "us_p90": us[(9 * n) // 10], "replays": n, "launches_per_step": launches,
            "tokens_per_s": 1e6 / statistics.median(us),
            "timing": "one graph replay per step, each timed alone with CUDA events (L2-resident inputs)"}


def run_hier_extra(args, device):
    """The hierarchical sparse indexer at 1M (fp8): a Reindex step scoring the
    whole pool against one scoring only the candidate pool of 2,048 blocks of
    8 that a Full candidate-source step left (and that source step itself)."""
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS["decode_1m_b8_fp8"]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads, kv_format=wl.kv_format,
                          idx_key_format=wl.idx_key_format)
    copies = [Copy(ctx, wl, c, device) for c in range(2)]  # 280 MB of keys and rows each, > L2
    cands = [torch.full((wl.n_query, int(ctx.cfg.cand_keep)), -1, dtype=torch.int32, device=device) for _ in copies]
    stream = torch.cuda.Stream(device=device)
    steps = max(5, min(args.steps, 100))

    def timed(fn):
        with torch.cuda.stream(stream):
            for i in range(3):
                fn(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(steps):
                fn(i)
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms_source = timed(lambda i: copies[i % 2].step_as(ctx, 0, 1, cands[i % 2]))
    ms_full = timed(lambda i: copies[i % 2].step_as(ctx, 0))
    ms_reindex = timed(lambda i: copies[i % 2].step_as(ctx, 1))
    ms_pool = timed(lambda i: copies[i % 2].step_as(ctx, 1, 2, cands[i % 2]))
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the hierarchical workload")
    pool = int(ctx.cfg.cand_keep) * int(ctx.cfg.cand_block)
    return {"workload": wl.name, "pool_entries": pool, "entries_per_query": int(copies[0].max_vis),
            "ms_full_step": ms_full, "ms_full_step_as_candidate_source": ms_source,
            "ms_reindex_step": ms_reindex, "ms_reindex_step_in_pool": ms_pool,
            "reindex_speedup": ms_reindex / ms_pool}


def run_sharded_extra(args, device):
    """The pool-sharded step at 1M (fp8) for G = 2 and 4 shards of every
    sequence's pool, with every shard's kernels run on this one GPU, one
    shard at a time. Phase 1 is the shard's visible count, scan, local top-k
    and (score, entry) pairs; phase 2 the merge of the G pair lists and the
    partial attention; phase 3 the combine. Each phase of each shard is one
    captured CUDA graph, replayed after an L2 flush and timed alone with CUDA
    events. On G GPUs the G shards run each phase at once, so the step's
    compute is the sum over the phases of the slowest shard. The two
    all-gathers between the phases are not timed (one GPU); their payloads
    per shard are reported."""
    from compressed_sparse_attention_gb300 import binding, sharded
    wl = PRESETS["decode_1m_b8_fp8"]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads, kv_format=wl.kv_format,
                          idx_key_format=wl.idx_key_format)
    base = Copy(ctx, wl, 0, device)
    ops = sharded.ContextOps(ctx)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=device)  # > the 129 MB L2
    stream = torch.cuda.Stream(device=device)
    reps = max(3, min(args.steps, 20))
    res = {"workload": wl.name, "timing": "per phase and shard: one graph replay after an L2 flush, CUDA events",
           "exchanges": "not timed (one GPU)"}
    with torch.cuda.stream(stream):
        for G in (2, 4):
            shards = [sharded.shard_inputs(base.inp, wl.n_seq, G, g) for g in range(G)]
            gens = [sharded.shard_step(ops, s, wl.topk) for s in shards]
            graphs, payload = [[], [], []], None
            for ph in range(3):
                outs = []
                for g in range(G):
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=stream):
                        try:
                            outs.append(next(gens[g]) if ph == 0 else gens[g].send(payload))
                        except StopIteration as stop:
                            outs.append(stop.value)
                    gr.replay()
                    graphs[ph].append(gr)
                torch.cuda.synchronize()
                if ph < 2:
                    payload = tuple(torch.stack([o[i] for o in outs]) for i in range(len(outs[0])))
                if ph == 0:
                    pairs = payload
            # the merge of phase 2 alone, on the same gathered pairs
            sel_m = torch.empty((wl.n_query, wl.topk), dtype=torch.int32, device=device)
            gm = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gm, stream=stream):
                ctx.topk_merge(pairs[0], pairs[1], wl.topk, sel_m)
            ms_merge = 0.0
            ms = [[0.0] * G for _ in range(3)]
            for _ in range(reps):
                for ph in range(3):
                    for g in range(G):
                        flush.zero_()
                        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        graphs[ph][g].replay()
                        e1.record(stream)
                        torch.cuda.synchronize()
                        ms[ph][g] += e0.elapsed_time(e1) / reps
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                gm.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                ms_merge += e0.elapsed_time(e1) / reps
            worst = [max(m) for m in ms]
            step = sum(worst)
            pairs_b = wl.n_query * wl.topk * 8
            part_b = wl.n_query * 64 * (512 + 2) * 4
            res[f"g{G}"] = {"ms_phase1_scan_topk": worst[0], "ms_phase2_merge_attend": worst[1],
                            "ms_phase3_combine": worst[2], "ms_step_compute": step, "ms_merge_alone": ms_merge,
                            "tokens_per_s_compute": wl.n_query / (step / 1000.0),
                            "ms_phase1_per_shard": ms[0], "ms_phase2_per_shard": ms[1],
                            "exchange_bytes_per_shard": [pairs_b, part_b]}
            del graphs, gens, shards, payload, pairs, gm
            torch.cuda.synchronize()
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the sharded workload")
    return res


def reuse_bytes(wl):
    """Minimal HBM bytes of one Reuse layer: the borrowed selection, the
    gathered window and selected rows once, q in and the output out."""
    wrow, prow, _ = row_bytes(wl)
    total = 0
    for b in range(wl.n_seq):
        n = wl.ctx_len[b]
        for i in range(wl.n_query_per_seq):
            t = n - wl.n_query_per_seq + i
            nv = (t + 1) // wl.m
            total += min(wl.window, t + 1) * wrow + min(wl.topk, nv) * prow
            total += wl.topk * 4 + wl.n_heads * wl.head_dim * 2 * 2
    return total


def run_mixed_extra(args, device, hbm):
    """The mixed serving batch: 64 decode sequences of log-uniform length
    1K..256K, compress ratio 1. One Reindex layer scores every visible entry
    and selects; three Reuse layers, each with its own q, window and sink,
    attend over the borrowed pool and selection. The four layers are one CUDA
    graph, timed back to back (the scan's 0.8 GB evicts L2 between groups)."""
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS["mixed_reuse_b64"]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads)
    base = Copy(ctx, wl, 0, device)
    shared = {k: base.inp[k] for k in ("n_vis", "pool_kv", "pool_off", "q_idx", "w_heads", "idx_keys")}
    layers = []
    for layer in (1, 2, 3):
        li = make_inputs(wl.scaled(seed=wl.seed), device, layer=layer, with_compress=False)
        layers.append((li, torch.empty_like(base.out)))
    stream = torch.cuda.Stream(device=device)

    def reindex():
        base.step_as(ctx, binding.MODE_REINDEX)

    def reuse(li, out):
        ctx.step(binding.MODE_REUSE, wl.n_seq, base.max_vis, q=li["q"], q_pos=li["q_pos"], seq_of_q=li["seq_of_q"],
                 sink=li["sink"], win_kv=li["win_kv"], win_off=li["win_off"], topk_idx=base.idx, out=out,
                 workspace=base.ws, **shared)

    def group():
        reindex()
        for li, out in layers:
            reuse(li, out)

    reps = max(5, min(args.steps, 100))

    def timed(fn):
        with torch.cuda.stream(stream):
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    ms_group = timed(group)
    ms_reindex = timed(reindex)
    ms_reuse = timed(lambda: reuse(*layers[0]))
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x} on the mixed workload")
    b_reindex = algorithmic_bytes(wl, has_compress=False)
    b_reuse = reuse_bytes(wl)
    b_group = b_reindex + 3 * b_reuse
    return {"workload": wl.name, "layers": "1 Reindex + 3 Reuse", "entries": int(base.inp["n_vis"].sum()),
            "ms_per_group": ms_group, "layer_tokens_per_s": 4 * wl.n_query / (ms_group / 1000.0),
            "ms_reindex_layer": ms_reindex, "ms_reuse_layer": ms_reuse,
            "group_algorithmic_bytes": b_group, "hbm_gbs": b_group / (ms_group / 1000.0) / 1e9,
            "hbm_frac": b_group / (ms_group / 1000.0) / 1e9 / hbm}


def run_e2e(args, ctx, copies, stream, device, wl):
    """The step through its host-buffer entry points, with the step's inputs
    (q, and the closing groups' raw tokens and gates) and its output in pinned
    host memory; the caches (window, pool, index keys) stay resident. Timed two
    ways: one csa2_step_graph_launch per step (the host step captured once per
    input copy) and one csa2_step_host call per step. Inside, q is staged by a
    kernel on a copy stream as the index scan retires, compress reads the raw
    tokens and gates in place, and the merge writes the output into host memory. The argument
    block of each input copy is prepared once, as a serving loop that reuses
    its buffers would."""
    steps = max(10, min(args.steps, 200))
    hosts = []
    for c in copies:
        i = c.inp
        hosts.append(dict(q=i["q"].cpu().pin_memory(), raw=i["raw"].cpu().pin_memory(),
                          gate=i["gate"].cpu().pin_memory()))
    dq = torch.empty_like(copies[0].inp["q"])
    draw = torch.empty_like(copies[0].inp["raw"])
    dgate = torch.empty_like(copies[0].inp["gate"])
    dout = torch.empty_like(copies[0].out)
    hout = torch.empty(dout.shape, dtype=dout.dtype).pin_memory()
    h2d = (dq.numel() * dq.element_size() + draw.numel() * draw.element_size() + dgate.numel() * dgate.element_size())
    d2h = dout.numel() * dout.element_size()

    prepared = [ctx.prepare_step(0, wl.n_seq, c.max_vis, **c.step_kwargs(q=dq, raw=draw, gate=dgate, out=dout))
                for c in copies]
    # each step one csa2_step_graph_launch: the copies in, the step, the copy out
    with torch.cuda.stream(stream):
        graphs = [p.host_graph(q=h["q"], raw=h["raw"], gate=h["gate"], out=hout) for p, h in zip(prepared, hosts)]

    def direct(i):
        h = hosts[i % N_COPIES]
        prepared[i % N_COPIES].run_host(q=h["q"], raw=h["raw"], gate=h["gate"], out=hout)

    def one(i):
        graphs[i % N_COPIES].launch()

    with torch.cuda.stream(stream):
        for i in range(3):
            one(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            one(i)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    with torch.cuda.stream(stream):
        for i in range(3):
            direct(i)
        torch.cuda.synchronize()
        e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e2.record(stream)
        for i in range(steps):
            direct(i)
        e3.record(stream)
    torch.cuda.synchronize()
    return dict(ms_per_step=ms / steps, steps=steps, h2d=h2d, d2h=d2h, direct_ms=e2.elapsed_time(e3) / steps)


def profile_kernel(args):
    """A small case for an ncu capture of one kernel: one input copy of the
    workload (the 1M decodes hold ~1.4 GB, still larger than L2), one full
    step to make the selection, then five calls of csa2_index_score or
    csa2_attend on the same inputs."""
    from compressed_sparse_attention_gb300 import binding, build
    build.build()
    device = torch.device("cuda:0")
    torch.cuda.set_device(device)
    wl = PRESETS[args.workload]
    ctx = binding.Context(compress_ratio=wl.m, idx_heads=wl.idx_heads, kv_format=wl.kv_format,
                          idx_key_format=wl.idx_key_format)
    c = Copy(ctx, wl, 0, device)
    c.step(ctx)
    ws = binding.workspace(ctx.attend_workspace_size(wl.n_query), device)
    for _ in range(5):
        if args.profile_kernel == "index":
            c.index_only(ctx)
        else:
            c.attend_only(ctx, ws)
    torch.cuda.synchronize()
    flags, _ = ctx.check()
    if flags:
        raise RuntimeError(f"device error word 0x{flags:x}")
    print(json.dumps({"profile_kernel": args.profile_kernel, "workload": wl.name, "calls": 5}))


# ----------------------------------------------------------------------------- CPU oracle arm

class OracleSample:
    """The CPU oracle on whole decode queries of the workload's first sequence
    (a bounded sample of the same workload); inputs are prepared once."""

    def __init__(self, wl):
        import numpy as np
        from oracle import csa2_oracle as O
        from oracle import formats as F
        self.O = O
        self.geom = O.Geometry(compress_ratio=wl.m, idx_heads=wl.idx_heads, topk=wl.topk, window=wl.window)
        g = self.geom
        self.f = O.yarn_inv_freq(64, g.rope_theta, g.yarn_factor, g.yarn_orig_len, g.yarn_beta_fast, g.yarn_beta_slow)
        one = wl.scaled(n_seq=1, ctx_len=wl.ctx_len[:1])
        inp = make_inputs(one, "cpu")

        def bf(t):
            return F.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))

        def fp8(t):
            return F.fp8_block_dequantize(*F.fp8_block_quantize(t.double().numpy()))

        def fp4(t):
            return F.fp4_block_dequantize(*F.fp4_block_quantize(t.double().numpy()))

        def mxfp4(t):
            return F.mxfp4_block_dequantize(*F.mxfp4_block_quantize(t.double().numpy()))

        if wl.idx_fp8:
            self.keys = (mxfp4 if wl.key_fp4 else fp8)(inp["idx_keys_f32"])
        else:
            self.keys = bf(inp["idx_keys"])
        if wl.kv_fp8:
            self.pool = (fp4 if wl.pool_fp4 else fp8)(inp["pool_kv_f32"])
            self.win = fp8(inp["win_kv_f32"])
        else:
            self.pool, self.win = bf(inp["pool_kv"]), bf(inp["win_kv"])
        self.q = bf(inp["q"][0])
        self.qi, self.w = bf(inp["q_idx"][0]), inp["w_heads"][0].double().numpy()
        self.sink = inp["sink"].double().numpy()
        self.t = int(inp["q_pos"][0])
        self.wl = wl

    def run_one(self):
        cap = self.win.shape[0]
        win = self.win
        self.O.step_query(self.O.MODE_REINDEX, self.geom, self.f, q=self.q, t=self.t,
                          win_rows_by_pos=lambda p: win[p % cap], comp_rows=self.pool, sink=self.sink,
                          q_idx=self.qi, w_heads=self.w, idx_keys=self.keys)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() in ("Model name", "Model"):
                v = line.split(":", 1)[1].strip()
                if v and not v.isdigit():
                    return v
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith(("model name", "cpu model")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _cpu_baseline_child(name, budget_s, threads):
    """Runs in a child process whose BLAS thread count was fixed by its
    environment (and whose affinity is cut to `threads` cores): times whole
    decode queries of the workload through the oracle for about budget_s."""
    if hasattr(os, "sched_setaffinity"):
        cpus = sorted(os.sched_getaffinity(0))
        os.sched_setaffinity(0, set(cpus[:threads]))
    wl = PRESETS[name]
    s = OracleSample(wl)
    done = 0
    t0 = time.perf_counter()
    while True:
        s.run_one()
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    print(json.dumps({"done": done, "seconds": el}))


def cpu_baseline(wl, budget_s):
    """The oracle, as it stands, on the host's cores: whole decode queries of
    the workload's first sequence, timed twice in child processes, once with
    the BLAS thread count and the affinity at every core of this process and
    once at one core. The line's value is the all-core run."""
    n_all = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    runs = {}
    for threads in (n_all, 1):
        env = dict(os.environ)
        for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS",
                  "VECLIB_MAXIMUM_THREADS", "NUMEXPR_NUM_THREADS"):
            env[k] = str(threads)
        code = (f"import sys; sys.path.insert(0, {ROOT!r}); import bench; "
                f"bench._cpu_baseline_child({wl.name!r}, {float(budget_s)!r}, {threads})")
        try:
            r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                               timeout=budget_s * 4 + 180)
            d = json.loads(r.stdout.strip().splitlines()[-1])
            runs[threads] = d["done"] / d["seconds"], d["done"], d["seconds"]
        except Exception as ex:  # reported, never silently dropped
            runs[threads] = None, 0, repr(ex)[:200]
    v_all, n_done, el = runs[n_all]
    v_one = runs[1][0]
    return {"value": v_all, "unit": "tokens/s", "cores": n_all, "kind": "oracle",
            "value_1_core": v_one, "cpu_model": cpu_model(),
            "sample": f"{n_done} decode queries of {wl.name} (one sequence, {wl.ctx_len[0]} context) through the "
                      f"float64 NumPy oracle (score, top-k, attend) in {el if isinstance(el, str) else f'{el:.1f} s'}, "
                      f"BLAS threads and affinity at {n_all} cores; again at 1 core for value_1_core"}


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="decode_64k_b32", choices=sorted(PRESETS))
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-extra", action="store_true", help="skip the 1M-context line item")
    ap.add_argument("--profile-kernel", choices=["index", "attend"], default=None,
                    help="for an ncu capture on a small case: one input copy of --workload, one step, then five "
                         "calls of that kernel's entry point; prints one line and exits (no timing)")
    args = ap.parse_args()
    if args.profile_kernel:
        profile_kernel(args)
        return

    world, rank, local, pg = dist_setup(args)
    wl = PRESETS[args.workload]
    units_per_step = wl.n_query

    if args.impl == "reference":
        if rank != 0:
            return
        sample = OracleSample(wl)
        for _ in range(args.warmup):
            sample.run_one()
        t0 = time.perf_counter()
        n_done = 0
        for _ in range(args.steps):
            sample.run_one()
            n_done += 1
        el = time.perf_counter() - t0
        val = n_done / el
        line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s", "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * el / args.steps,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": wl.name, "batch": wl.n_seq, "context": wl.ctx_len[0],
                           "compress_ratio": wl.m, "topk": wl.topk, "window": wl.window,
                           "step_sample": "one decode query per step (a bounded sample of the batch)"},
                "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                 "sample": f"{args.steps} single-query steps of {wl.name} through the float64 "
                                           "NumPy oracle"},
                "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for the gb300 arm")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    hbm, bf16_burst, bf16_sus, peak_src = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    r = run_gpu_workload(args, wl, rank, pg, device, (hbm, bf16_burst))
    sampler.stop()
    clocks = sampler.summary()
    ms_step = r["ms_max"] / args.steps
    value = aggregate_value(world, units_per_step, args.steps, r["ms_max"])
    step_bytes = algorithmic_bytes(wl)
    gbs = step_bytes / (ms_step / 1000.0) / 1e9
    idx_b = index_bytes(wl)
    idx_gbs = idx_b / (r["idx_ms"] / 1000.0) / 1e9
    e2e = r["e2e"]
    # the two public host-buffer paths, each the slowest rank's time; the
    # faster of the two is the end-to-end figure
    e2e_graph = max_over_ranks(pg, e2e["ms_per_step"], device)
    e2e_direct = max_over_ranks(pg, e2e["direct_ms"], device)
    e2e_ms = min(e2e_graph, e2e_direct)
    e2e_api = ("csa2_step_graph_launch per step" if e2e_graph <= e2e_direct else "csa2_step_host per step")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": wl.name, "batch": wl.n_seq, "context": wl.ctx_len[0], "compress_ratio": wl.m,
                   "topk": wl.topk, "window": wl.window, "heads": "64x512", "indexer": f"{wl.idx_heads}x128",
                   "kv": kv_format_name(wl),
                   "l2": f"{N_COPIES} rotating input copies ({N_COPIES * step_bytes / 1e6:.0f} MB > 129 MB L2)",
                   "graph": f"one CUDA graph per {N_COPIES} consecutive steps (one per input copy)"},
        "hbm_gbs": gbs, "hbm_frac": gbs / hbm, "step_algorithmic_bytes": step_bytes,
        "roofline": {"kernel": "index_score", "bound": "hbm", "achieved": idx_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": idx_gbs / hbm,
                     "traffic": INDEX_TRAFFIC_BYTES if wl.name == "decode_64k_b32" else None,
                     "peak_source": peak_src,
                     "bytes_per_launch": idx_b, "ms_per_launch": r["idx_ms"]},
        "e2e": {"value": world * units_per_step / (e2e_ms / 1000.0), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e_ms, "steps": e2e["steps"],
                "api": e2e_api + " (pinned host q, raw tokens, gates and out: q staged by a kernel on a copy "
                                 "stream as the index scan retires, raw tokens and gates read in place by "
                                 "compress, out written by the merge over the host link)",
                "ms_per_step_csa2_step_graph_launch": e2e_graph, "ms_per_step_csa2_step_host": e2e_direct},
        "ms_per_step_median": max_over_ranks(pg, r["ms_median"], device),
        "ms_per_step_median_how": f"median over {r['n_rep']} replays of the {N_COPIES}-step graph, each timed "
                                  f"alone with CUDA events, divided by {N_COPIES}",
        "gpu_launches": r["launches"] * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_extra and wl.name == "decode_64k_b32" and world == 1:
        for key, name in (("extra_1m", "decode_1m_b8_fp8"), ("extra_1m_fp4", "decode_1m_b8_fp4")):
            try:
                wl4 = PRESETS[name]
                a2 = argparse.Namespace(**vars(args))
                a2.steps = min(args.steps, 500)
                r4 = run_gpu_workload(a2, wl4, rank, None, device, (hbm, bf16_burst))
                ms4 = r4["ms"] / a2.steps
                b4 = algorithmic_bytes(wl4)
                line[key] = {"workload": wl4.name, "kv": kv_format_name(wl4),
                             "tokens_per_s": wl4.n_query / (ms4 / 1000.0), "ms_per_step": ms4,
                             "hbm_gbs": b4 / (ms4 / 1000.0) / 1e9, "hbm_frac": b4 / (ms4 / 1000.0) / 1e9 / hbm,
                             "step_algorithmic_bytes": b4,
                             "index_gbs": index_bytes(wl4) / (r4["idx_ms"] / 1000.0) / 1e9}
            except Exception as ex:  # reported, never silently dropped
                line[key] = {"error": repr(ex)[:300]}
        try:
            line["extra_tiny"] = run_tiny_extra(args, device)
        except Exception as ex:  # reported, never silently dropped
            line["extra_tiny"] = {"error": repr(ex)[:300]}
        try:
            line["extra_hier"] = run_hier_extra(args, device)
        except Exception as ex:  # reported, never silently dropped
            line["extra_hier"] = {"error": repr(ex)[:300]}
        try:
            line["extra_prefill"] = run_prefill_extra(args, device, bf16_burst)
        except Exception as ex:  # reported, never silently dropped
            line["extra_prefill"] = {"error": repr(ex)[:300]}
        try:
            line["extra_mixed_reuse"] = run_mixed_extra(args, device, hbm)
        except Exception as ex:  # reported, never silently dropped
            line["extra_mixed_reuse"] = {"error": repr(ex)[:300]}
        try:
            line["extra_sharded"] = run_sharded_extra(args, device)
        except Exception as ex:  # reported, never silently dropped
            line["extra_sharded"] = {"error": repr(ex)[:300]}
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget)
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
