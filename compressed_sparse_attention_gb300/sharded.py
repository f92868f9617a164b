"""A CSA2 layer step with each sequence's compressed pool split over shards.

Shard g of G holds entries [lo_g, hi_g) of every sequence's pool (its rows at
pool_off[b] + j - lo_g of its own arrays), its index keys alike, and a copy
of the batch's queries; one shard also holds the window rows. The selection
is the unsharded one ("Reading Notes of DeepSeek-V4.1-Flash", section 3f,
C2 step 2: the 512 best entries of the whole pool). The pages' own
multi-rank form splits the heads and all-reduces the indexer's scores
(PocketLLM "DeepSeek-V4.1-Flash", "The CSA2 attention layers"); here the pool
is split instead, and two exchanges carry 512 (score, entry) pairs and one
(m, l, O) partial per query and shard:

  1. the shard's visible count (csa2_shard_visible), its scan and local
     top-k over its own entries, as (score, global entry) pairs
     (csa2_topk_pairs);
  -- exchange 1: all-gather of the G pair lists --
  2. the global top-k (csa2_topk_merge; ties to the lower entry), then the
     partial attention over the selected entries that lie in this shard, plus
     the window on the shard that holds it (csa2_attend_partial);
  -- exchange 2: all-gather of the G partials --
  3. the log-sum-exp combine with the sink counted once (csa2_attend_combine).

`shard_step` is one shard's part, written as a generator that yields its
payload at each exchange and receives the gathered payloads (stacked in
shard order). `run_distributed` drives it on one rank per shard through
torch.distributed all-gathers; `run_local` drives all shards of one process
in lockstep, the gather being a stack. Every step of the arithmetic runs in
the library's kernels; this module only allocates outputs and moves tensors.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import binding


def shard_range(n_entries: int, n_shards: int, shard: int) -> tuple[int, int]:
    """Entries [lo, hi) of shard `shard` when n_entries are split as evenly as
    ceil division allows (the last shards may be shorter or empty)."""
    if n_shards < 1 or not 0 <= shard < n_shards:
        raise ValueError("shard out of range")
    per = -(-max(n_entries, 0) // n_shards)
    lo = min(n_entries, shard * per)
    return lo, min(n_entries, lo + per)


@dataclass
class ShardInputs:
    """One shard's view of a step: the batch's queries (the same on every
    shard), this shard's slice of the pools and keys, and the window on the
    shard that attends to it."""
    lo: int
    hi: int
    with_window: bool
    n_seq: int
    q: torch.Tensor          # [Q, 64, 512] bf16
    q_pos: torch.Tensor      # [Q] int64
    seq_of_q: torch.Tensor   # [Q] int32
    n_vis: torch.Tensor      # [Q] int32, visible entries of the whole pool
    q_idx: torch.Tensor      # [Q, H_I, 128] bf16
    w_heads: torch.Tensor    # [Q, H_I] fp32
    sink: torch.Tensor       # [64] fp32
    pool_off: torch.Tensor   # [B+1] int64, this shard's rows of each sequence
    pool_kv: torch.Tensor
    idx_keys: torch.Tensor
    pool_scale: Optional[torch.Tensor] = None
    idx_key_scale: Optional[torch.Tensor] = None
    win_kv: Optional[torch.Tensor] = None
    win_scale: Optional[torch.Tensor] = None
    win_off: Optional[torch.Tensor] = None
    win_lo: Optional[torch.Tensor] = None


def shard_inputs(inp: dict, n_seq: int, n_shards: int, shard: int, window_shard: int = 0) -> ShardInputs:
    """Shard `shard`'s view of a resident batch `inp` (the step's arguments by
    name, as csa2_step takes them): entries [lo, hi) of every sequence's pool,
    lo and hi from the longest pool, copied out as one contiguous slice per
    sequence (rows, scales, index keys and their scales alike), and the window
    on shard `window_shard` only."""
    poff = inp["pool_off"].tolist()
    longest = max(poff[b + 1] - poff[b] for b in range(n_seq))
    lo, hi = shard_range(longest, n_shards, shard)
    spans = [(poff[b] + lo, max(poff[b] + lo, min(poff[b + 1], poff[b] + hi))) for b in range(n_seq)]
    off = [0]
    for a, e in spans:
        off.append(off[-1] + e - a)

    def rows(t):
        if t is None:
            return None
        if off[-1] == 0:  # no entries here: one row keeps the arrays addressable
            return t[:1].clone()
        return torch.cat([t[a:e] for a, e in spans if e > a]).contiguous()

    win = shard == window_shard
    dev = inp["q"].device
    return ShardInputs(
        lo=lo, hi=hi, with_window=win, n_seq=n_seq, q=inp["q"], q_pos=inp["q_pos"], seq_of_q=inp["seq_of_q"],
        n_vis=inp["n_vis"], q_idx=inp["q_idx"], w_heads=inp["w_heads"], sink=inp["sink"],
        pool_off=torch.tensor(off, dtype=torch.int64, device=dev), pool_kv=rows(inp["pool_kv"]),
        pool_scale=rows(inp.get("pool_scale")), idx_keys=rows(inp["idx_keys"]),
        idx_key_scale=rows(inp.get("idx_key_scale")), win_kv=inp["win_kv"] if win else None,
        win_scale=inp.get("win_scale") if win else None, win_off=inp["win_off"] if win else None,
        win_lo=inp.get("win_lo") if win else None)


def shard_step(ctx, s: ShardInputs, k: int):
    """One shard's part of the step (a generator; see the module notes).
    Returns (out [Q, 64, 512] bf16, lse [Q, 64] fp32, selection [Q, k] int32)."""
    dev = s.q.device
    n_q = s.q.shape[0]
    width = max(1, s.hi - s.lo)
    n_vis_local = torch.empty(n_q, dtype=torch.int32, device=dev)
    ctx.shard_visible(s.n_vis, s.lo, s.hi, n_vis_local)
    scores = torch.empty((n_q, width), dtype=torch.float32, device=dev)
    ctx.index_score(s.n_seq, s.q_idx, s.w_heads, s.idx_keys, s.idx_key_scale, s.pool_off, s.seq_of_q, n_vis_local,
                    width, scores)
    local = torch.empty((n_q, k), dtype=torch.int32, device=dev)
    ctx.topk(scores, n_vis_local, width, k, local, ctx.topk_workspace(n_q, width))
    pair_score = torch.empty((n_q, k), dtype=torch.float32, device=dev)
    pair_idx = torch.empty((n_q, k), dtype=torch.int32, device=dev)
    ctx.topk_pairs(scores, local, s.lo, pair_score, pair_idx)
    all_score, all_idx = yield (pair_score, pair_idx)
    sel = torch.empty((n_q, k), dtype=torch.int32, device=dev)
    ctx.topk_merge(all_score, all_idx, k, sel)
    part_o = torch.empty((n_q, 64, 512), dtype=torch.float32, device=dev)
    part_m = torch.empty((n_q, 64), dtype=torch.float32, device=dev)
    part_l = torch.empty((n_q, 64), dtype=torch.float32, device=dev)
    ctx.attend_partial(s.n_seq, s.q, s.q_pos, s.seq_of_q, s.with_window, s.win_kv, s.win_scale, s.win_off, s.win_lo,
                       s.pool_kv, s.pool_scale, s.pool_off, sel, s.lo, s.hi, part_o, part_m, part_l)
    all_o, all_m, all_l = yield (part_o, part_m, part_l)
    out = torch.empty((n_q, 64, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((n_q, 64), dtype=torch.float32, device=dev)
    ctx.attend_combine(all_o, all_m, all_l, s.q_pos, s.sink, out, lse)
    return out, lse, sel


def run_local(gens):
    """All shards in one process: each generator runs to its next exchange,
    then every one receives the payloads stacked in shard order."""
    payloads = [next(g) for g in gens]
    while True:
        gathered = tuple(torch.stack([p[i] for p in payloads]) for i in range(len(payloads[0])))
        results, nxt = [], []
        for g in gens:
            try:
                nxt.append(g.send(gathered))
            except StopIteration as stop:
                results.append(stop.value)
        if results:
            if len(results) != len(gens):
                raise RuntimeError("shards disagree on the number of exchanges")
            return results
        payloads = nxt


def all_gather_stacked(t: torch.Tensor, group=None) -> torch.Tensor:
    """[world, *t.shape]: every rank's tensor in rank order (torch.distributed)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    parts = [torch.empty_like(t) for _ in range(world)]
    dist.all_gather(parts, t.contiguous(), group=group)
    return torch.stack(parts)


def run_distributed(gen, group=None):
    """One shard on this rank: each exchange is an all-gather over the group
    (NCCL between GPUs, gloo between CPU processes)."""
    payload = next(gen)
    while True:
        gathered = tuple(all_gather_stacked(t, group) for t in payload)
        try:
            payload = gen.send(gathered)
        except StopIteration as stop:
            return stop.value


class ContextOps:
    """The calls shard_step makes, on a binding.Context (the CUDA library)."""

    def __init__(self, ctx: "binding.Context"):
        self.ctx = ctx

    def __getattr__(self, name):
        return getattr(self.ctx, name)

    def topk_workspace(self, n_query: int, max_vis: int) -> torch.Tensor:
        n = int(self.ctx.lib.csa2_topk_workspace_size(self.ctx.h, n_query, max_vis))
        return binding.workspace(n, self.ctx.device)
