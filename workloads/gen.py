"""Workload presets and seeded input generation.

Layouts produced (row-major, last axis contiguous; B sequences, Q queries):

  q          [Q, H, D]     bf16   per-query attention query (unrotated)
  q_pos      [Q]           int64  position t of each query
  seq_of_q   [Q]           int32  sequence of each query
  n_vis      [Q]           int32  compressed entries visible to each query
  q_idx      [Q, HI, DI]   bf16   indexer query
  w_heads    [Q, HI]       fp32   indexer head weights
  sink       [H]           fp32   per-head sink logit
  win_off    [B+1]         int64  window-buffer row offsets (capacity per sequence)
  win_kv     [sum cap, D]  bf16   stored window rows; position p of sequence b is
                                  row win_off[b] + p % cap_b
  pool_off   [B+1]         int64  compressed-pool row offsets
  pool_kv    [sum P, D]    bf16   stored compressed rows
  idx_keys   [sum P, DI]   bf16   index keys
  raw, gate  [T, D]        bf16 / fp32  tokens to compress (whole groups)
  tok_off    [B+1]         int64  token offsets of each sequence's segment
  first_pos  [B]           int64  position of each segment's first token
  norm_w [D], k_norm_w [DI] fp32, w_idx [DI, D] bf16  compressor weights

For the fp8 workloads the window rows, pool rows and index keys are drawn as
fp32 values (keys *_f32); each side stores them in its own fp8 format.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    n_seq: int
    ctx_len: tuple            # tokens seen per sequence (decode: the query is the last one)
    m: int                    # compress ratio
    seed: int
    n_query_per_seq: int = 1  # prefill: queries appended at the end of each sequence
    window: int = 128
    topk: int = 512
    n_heads: int = 64
    head_dim: int = 512
    idx_heads: int = 8
    idx_dim: int = 128
    kv_fp8: bool = False      # window and pool drawn in fp32 and stored quantised (fp8 unless pool_fp4)
    idx_fp8: bool = False     # index keys drawn in fp32 and stored quantised (fp8 unless key_fp4)
    pool_fp4: bool = False    # pool rows stored fp4 e2m1 with an e4m3 scale per 16 (needs kv_fp8)
    key_fp4: bool = False     # index keys stored mxfp4 with an e8m0 scale per 32 (needs idx_fp8)
    value_std: float = 1.0    # q and KV element std
    outlier_frac: float = 0.0  # fraction of KV rows scaled by outlier_scale
    outlier_scale: float = 8.0
    n_layers: int = 1         # >1: one Reindex layer then Reuse layers sharing pool and idx
    win_linear: bool = False  # window buffer holds every position (prefill) instead of a ring

    @property
    def kv_format(self) -> int:
        """The library's kv_format code: 0 bf16, 1 fp8, 2 fp4 pool + fp8 window."""
        return 2 if self.pool_fp4 else int(self.kv_fp8)

    @property
    def idx_key_format(self) -> int:
        """The library's idx_key_format code: 0 bf16, 1 fp8, 3 mxfp4."""
        return 3 if self.key_fp4 else int(self.idx_fp8)

    @property
    def n_query(self) -> int:
        return self.n_seq * self.n_query_per_seq

    def pool_len(self, b: int) -> int:
        return self.ctx_len[b] // self.m

    def win_cap(self, b: int) -> int:
        return self.ctx_len[b] if self.win_linear else self.window

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


def _log_uniform_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    g = torch.Generator().manual_seed(seed + 1000)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    vals = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return tuple(int(v) for v in torch.floor(vals).tolist())


PRESETS = {
    # tiny decode: batch 1, context 4,096, ratio 4 -> 1,024 entries, q/KV ~ N(0,1)/sqrt(512)
    "tiny_decode": Workload("tiny_decode", 1, (4096,), 4, seed=0, value_std=1.0 / math.sqrt(512.0)),
    # decode batch 32 at 65,536 context, ratio 4 -> 16,384 entries, 1% outlier rows x8
    "decode_64k_b32": Workload("decode_64k_b32", 32, (65536,) * 32, 4, seed=1, outlier_frac=0.01),
    # chunked prefill: 4,096 causal queries after an 8,192-token prefix, ratio 2
    "prefill_4k_after_8k": Workload("prefill_4k_after_8k", 1, (12288,), 2, seed=2,
                                    n_query_per_seq=4096, win_linear=True),
    # long-context decode batch 8 at 1,048,576, ratio 4 -> 262,144 entries, fp8 KV and keys
    "decode_1m_b8_fp8": Workload("decode_1m_b8_fp8", 8, (1 << 20,) * 8, 4, seed=3,
                                 kv_fp8=True, idx_fp8=True),
    # the same decode with fp4 pool rows (e4m3 scale per 16), an fp8 window and
    # mxfp4 index keys: 256 + 32 B per pool entry and 64 + 4 B per key
    "decode_1m_b8_fp4": Workload("decode_1m_b8_fp4", 8, (1 << 20,) * 8, 4, seed=5,
                                 kv_fp8=True, idx_fp8=True, pool_fp4=True, key_fp4=True),
    # mixed serving batch: 64 sequences, lengths log-uniform 1K-256K, ratio 1,
    # one Reindex layer then three Reuse layers
    "mixed_reuse_b64": Workload("mixed_reuse_b64", 64, _log_uniform_lengths(64, 1024, 262144, 4),
                                1, seed=4, n_layers=4),
}


def _randn(shape, g, device, std=1.0):
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std


def _kv_rows(n, d, g, device, std, outlier_frac, outlier_scale):
    x = _randn((n, d), g, device, std)
    if outlier_frac > 0 and n > 0:
        n_out = max(1, int(round(outlier_frac * n)))
        rows = torch.randperm(n, generator=g, device=device)[:n_out]
        x[rows] *= outlier_scale
    return x


def make_inputs(wl: Workload, device="cpu", layer: int = 0, with_compress: bool = True) -> dict:
    """Draw one layer's inputs for workload `wl` (layer > 0: a Reuse layer's own q/window/sink)."""
    device = torch.device(device)
    g = torch.Generator(device=device).manual_seed(wl.seed * 7919 + layer * 104729)
    H, D, HI, DI, B = wl.n_heads, wl.head_dim, wl.idx_heads, wl.idx_dim, wl.n_seq
    Q = wl.n_query
    out = {}
    # queries
    q_pos, seq_of_q, n_vis = [], [], []
    for b in range(B):
        n = wl.ctx_len[b]
        for i in range(wl.n_query_per_seq):
            t = n - wl.n_query_per_seq + i
            q_pos.append(t)
            seq_of_q.append(b)
            n_vis.append((t + 1) // wl.m)
    out["q_pos"] = torch.tensor(q_pos, dtype=torch.int64, device=device)
    out["seq_of_q"] = torch.tensor(seq_of_q, dtype=torch.int32, device=device)
    out["n_vis"] = torch.tensor(n_vis, dtype=torch.int32, device=device)
    out["q"] = _randn((Q, H, D), g, device, wl.value_std).to(torch.bfloat16)
    out["sink"] = _randn((H,), g, device)
    # window buffer
    caps = [wl.win_cap(b) for b in range(B)]
    win_off = [0]
    for c in caps:
        win_off.append(win_off[-1] + c)
    out["win_off"] = torch.tensor(win_off, dtype=torch.int64, device=device)
    win = _kv_rows(win_off[-1], D, g, device, wl.value_std, wl.outlier_frac, wl.outlier_scale)
    if wl.kv_fp8:
        out["win_kv_f32"] = win
    else:
        out["win_kv"] = win.to(torch.bfloat16)
    del win
    if layer > 0:
        return out
    # indexer query
    out["q_idx"] = _randn((Q, HI, DI), g, device).to(torch.bfloat16)
    out["w_heads"] = torch.rand((Q, HI), generator=g, device=device, dtype=torch.float32)
    # compressed pool and index keys
    plen = [wl.pool_len(b) for b in range(B)]
    pool_off = [0]
    for p in plen:
        pool_off.append(pool_off[-1] + p)
    out["pool_off"] = torch.tensor(pool_off, dtype=torch.int64, device=device)
    pool = _kv_rows(pool_off[-1], D, g, device, wl.value_std, wl.outlier_frac, wl.outlier_scale)
    if wl.kv_fp8:
        out["pool_kv_f32"] = pool
    else:
        out["pool_kv"] = pool.to(torch.bfloat16)
    del pool
    keys = _randn((pool_off[-1], DI), g, device)
    if wl.idx_fp8:
        out["idx_keys_f32"] = keys
    else:
        out["idx_keys"] = keys.to(torch.bfloat16)
    del keys
    if with_compress:
        # the tokens of the groups that close at this step: decode closes at most one
        # group per sequence; prefill closes every group of the appended chunk
        tok_off, first_pos = [0], []
        for b in range(B):
            n = wl.ctx_len[b]
            start = n - wl.n_query_per_seq
            first = (start // wl.m) * wl.m
            closed_end = (n // wl.m) * wl.m
            cnt = max(0, closed_end - first)
            first_pos.append(first)
            tok_off.append(tok_off[-1] + cnt)
        out["tok_off"] = torch.tensor(tok_off, dtype=torch.int64, device=device)
        out["first_pos"] = torch.tensor(first_pos, dtype=torch.int64, device=device)
        T = tok_off[-1]
        out["raw"] = _randn((T, D), g, device).to(torch.bfloat16)
        out["gate"] = _randn((T, D), g, device)
        out["norm_w"] = 0.5 + torch.rand((D,), generator=g, device=device)
        out["w_idx"] = _randn((DI, D), g, device, 1.0 / math.sqrt(D)).to(torch.bfloat16)
        out["k_norm_w"] = 0.5 + torch.rand((DI,), generator=g, device=device)
    return out


def make_selection(wl: Workload, n_vis: torch.Tensor, seed: int, device="cpu") -> torch.Tensor:
    """A valid top-k index set per query: min(k, n_vis) distinct visible entries,
    ascending, padded with -1 (drawn at random, not from any score)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    nv = n_vis.cpu().tolist()
    out = torch.full((len(nv), wl.topk), -1, dtype=torch.int32)
    for i, n in enumerate(nv):
        k = min(wl.topk, n)
        if k:
            pick = torch.randperm(n, generator=g)[:k]
            out[i, :k] = torch.sort(pick).values.to(torch.int32)
    return out.to(device)


def make_topk_scores(n_query: int, n: int, seed: int, tie_levels: int = 0, device="cpu") -> torch.Tensor:
    """fp32 scores [n_query, n]; tie_levels > 0 draws from that many distinct values
    so that many scores tie; also plants -0.0 and +0.0 together."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    if tie_levels > 0:
        lv = torch.randn(tie_levels, generator=g, dtype=torch.float32)
        s = lv[torch.randint(0, tie_levels, (n_query, n), generator=g)]
    else:
        s = torch.randn((n_query, n), generator=g, dtype=torch.float32)
    if n >= 4:
        s[:, 1] = -0.0
        s[:, 3] = 0.0
    return s.to(device)
