"""CPU oracle of the CSA2 compressed-sparse-attention step (float64, NumPy).

TEST INFRASTRUCTURE ONLY. The oracle is what the CUDA path is checked
against. Only the tests, the smoke check and the benchmark's CPU-baseline /
reference leg may import it; the product path (the C-ABI library and its
Python binding) never calls it and shares no code, header, table or helper
with it. It computes each step in plain float64, one query at a time, in the
order the method is written, with no blocking or fusion.

Sources (pages are cited by title and section):

* R  = "Reading Notes of DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache
       Compression", section 3a (the attention formula and its worked
       example) and section 3f, component C2 (CSA2 steps 1-4: compress,
       index, attend, the three sharing modes), C5 (window bounds).
* W  = "DeepSeek-V4.1-Flash on WASTE", section "What is new", item 1 (CSA2:
       the compressor, the two-level indexer, the attention sink, the output
       de-rotation, the two RoPE schedules) and "The shape" (64 heads x 512,
       one 512-wide KV per token, RoPE on 64 dims, YaRN factor 16 over 65,536).
* P  = "DeepSeek-V4.1-Flash" (PocketLLM), section "The CSA2 attention layers"
       (compressor in fp32, index key from the unrotated latent, RoPE of a
       compressed latent at the first token of its group, -1 padding) and
       section "The op layer" (the finite score floor so an all-invalid row
       yields zeros).

Readings where the pages leave a step open, each taken as the plainest one
that the rest of the pages support:

* Gate logits are per channel: g has the same shape as the raw KV c and the
  softmax runs over the m tokens of a group, channel by channel (R, C2 step 1
  writes the softmax elementwise with the Hadamard product).
* The compressor output is RMS-normalised with a learned weight after
  pooling, at every ratio including m = 1 (W, item 1: "then RMS-normed").
* The index key is RMSNorm_{k_norm}(c_hat @ W_I^T), taken from the normed,
  unrotated latent (P, "The CSA2 attention layers"); neither q^I nor k^I is
  rotated.
* The indexer weights omega are caller inputs used as they are.
* Top-k keeps the K largest scores, ties broken toward the lower index, and
  returns the chosen indices in ascending order, padded with -1.
* Entry j of a sequence is visible to the query at position t iff its whole
  group has been seen: (j + 1) * m - 1 <= t.
* The window of the query at t is positions [max(lo, t - w + 1), t],
  including t itself (R, C5 gives [max(s, i - w + 1), i]); lo defaults to 0.
* Key and value are the same stored row (W, "one 512-wide KV per token").
* The sink is a logit: the denominator gains exp(sink_h), unscaled by tau.
* tau = 1/sqrt(512) multiplies q.k; no YaRN attention-scale factor.
* RoPE rotates adjacent pairs of the last rope_dim dims by angle pos*f_i,
  with the YaRN ramp of DeepSeek-V3 (W, "What the engine already has").
* An empty row set with the sink at -inf yields a zero output (the finite
  floor of P, "The op layer").
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from . import formats as F


# ----------------------------------------------------------------------------
# Geometry
# ----------------------------------------------------------------------------

@dataclass(frozen=True)
class Geometry:
    """Shape constants of one CSA2 layer (W, "The shape"; P geometry table)."""
    n_heads: int = 64
    head_dim: int = 512
    rope_dim: int = 64
    window: int = 128
    compress_ratio: int = 4
    idx_heads: int = 8
    idx_dim: int = 128
    topk: int = 512
    softmax_scale: float = 1.0 / math.sqrt(512.0)
    norm_eps: float = 1e-20
    rope_theta: float = 160000.0
    yarn_factor: float = 16.0
    yarn_orig_len: float = 65536.0
    yarn_beta_fast: float = 32.0
    yarn_beta_slow: float = 1.0


# ----------------------------------------------------------------------------
# RoPE with the YaRN frequency ramp
# ----------------------------------------------------------------------------

def yarn_inv_freq(rope_dim: int, theta: float, factor: float, orig_len: float,
                  beta_fast: float, beta_slow: float) -> np.ndarray:
    """Per-pair rotation frequencies f_i, i < rope_dim/2 (float64).

    Plain RoPE gives f_i = theta^(-2i/rope_dim). YaRN ("NTK-by-parts", Peng et
    al. 2023, in the DeepSeek-V3 form that W names) keeps f_i for the pairs
    that turn more than beta_fast times over the original context, divides f_i
    by the factor for the pairs that turn fewer than beta_slow times, and
    blends linearly in the pair index between the two boundary indices.
    """
    half = rope_dim // 2
    i = np.arange(half, dtype=np.float64)
    base = theta ** (-(2.0 * i) / rope_dim)
    if factor is None or factor <= 1.0:
        return base

    def boundary_index(turns: float) -> float:
        # pair index whose wavelength fits `turns` times into orig_len:
        # orig_len / (2*pi*theta^(2i/d)) = turns  <=>  i = d*ln(L/(2*pi*turns)) / (2 ln theta)
        return rope_dim * math.log(orig_len / (turns * 2.0 * math.pi)) / (2.0 * math.log(theta))

    lo = max(math.floor(boundary_index(beta_fast)), 0)
    hi = min(math.ceil(boundary_index(beta_slow)), rope_dim - 1)
    if hi == lo:
        hi = hi + 0.001
    ramp = np.clip((i - lo) / (hi - lo), 0.0, 1.0)  # 0 keeps f_i, 1 divides by factor
    keep = 1.0 - ramp
    return base / factor * (1.0 - keep) + base * keep


def rope_rotate(x: np.ndarray, pos, inv_freq: np.ndarray, inverse: bool = False) -> np.ndarray:
    """Rotate the last 2*len(inv_freq) entries of x's last axis at position(s) pos.

    Pair i is (x[o+2i], x[o+2i+1]), o = D - 2*len(inv_freq); it turns by the
    angle pos*f_i (by -pos*f_i when inverse). pos is a scalar or has the shape
    of x without its last axis.
    """
    x = np.array(x, dtype=np.float64, copy=True)
    half = inv_freq.shape[0]
    if half == 0:
        return x
    d = x.shape[-1]
    o = d - 2 * half
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq  # [..., half]
    if inverse:
        ang = -ang
    c, s = np.cos(ang), np.sin(ang)
    x0 = x[..., o::2].copy()
    x1 = x[..., o + 1::2].copy()
    x[..., o::2] = x0 * c - x1 * s
    x[..., o + 1::2] = x0 * s + x1 * c
    return x


# ----------------------------------------------------------------------------
# a1. Compressor (R, C2 step 1; W item 1; P "The CSA2 attention layers")
# ----------------------------------------------------------------------------

def rms_norm(x: np.ndarray, weight: np.ndarray, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * weight along the last axis."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * weight


def compress(raw: np.ndarray, gate, m: int, first_pos: int, norm_w: np.ndarray,
             eps: float, inv_freq: np.ndarray, w_idx=None, k_norm_w=None):
    """Pool m consecutive raw KV vectors into one entry per group.

    raw [T, D] and gate [T, D] (T a multiple of m; gate unused at m = 1) hold
    the tokens at positions first_pos .. first_pos+T-1, first_pos a multiple
    of m. For group j (global index first_pos/m + i):
      weights  w_u = softmax over the group's m tokens of g_u (per channel),
      pooled   c_bar = sum_u w_u * c_u,
      normed   c_hat = RMSNorm_norm_w(c_bar),
      index key k_I = RMSNorm_k_norm_w(c_hat @ w_idx^T)   (unrotated c_hat),
      stored   kv   = RoPE at position j*m on the last rope dims of c_hat.
    Returns (kv_rotated [G, D], c_hat [G, D], k_I [G, idx_dim] or None).
    """
    raw = np.asarray(raw, dtype=np.float64)
    t_len, d = raw.shape
    if t_len % m or first_pos % m:
        raise ValueError("tokens must cover whole groups")
    g_cnt = t_len // m
    blocks = raw.reshape(g_cnt, m, d)
    if m == 1:
        pooled = blocks[:, 0, :]
    else:
        g = np.asarray(gate, dtype=np.float64).reshape(g_cnt, m, d)
        g = g - g.max(axis=1, keepdims=True)
        e = np.exp(g)
        w = e / e.sum(axis=1, keepdims=True)
        pooled = (w * blocks).sum(axis=1)
    c_hat = rms_norm(pooled, np.asarray(norm_w, dtype=np.float64), eps)
    k_idx = None
    if w_idx is not None:
        k_lin = c_hat @ np.asarray(w_idx, dtype=np.float64).T
        k_idx = rms_norm(k_lin, np.asarray(k_norm_w, dtype=np.float64), eps)
    group_pos = (first_pos // m + np.arange(g_cnt)) * m
    kv = rope_rotate(c_hat, group_pos, inv_freq)
    return kv, c_hat, k_idx


# ----------------------------------------------------------------------------
# Hierarchical sparse indexer (R, section 3f, C3; P, "The container",
# select_candidate_blocks)
# ----------------------------------------------------------------------------

def candidate_blocks(scores: np.ndarray, block: int = 8, n_keep: int = 2048) -> np.ndarray:
    """First level: the candidate source's pool of blocks.

    The n = len(scores) visible entries fall into blocks of `block`
    consecutive entries; a block scores the largest index score among its
    entries (R, C3: score(beta) = max over j in beta of sigma(j)). The block
    holding the newest entry n-1 is still filling and is kept whatever its
    score (P, "The container": pinned rather than ranked). The n_keep best
    blocks, by score and then by the lower block index, form the pool.
    Returns their block indices in ascending order."""
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    nb = -(-n // block)
    bs = np.array([s[b * block:min((b + 1) * block, n)].max() for b in range(nb)])
    bs[nb - 1] = np.inf
    order = np.lexsort((np.arange(nb), -bs))
    return np.sort(order[:n_keep]).astype(np.int64)


def pool_entries(cand: np.ndarray, n_vis: int, block: int = 8) -> np.ndarray:
    """The entries of the pool (R, C3: P_t, the union of the kept blocks),
    those below n_vis, ascending."""
    j = (np.asarray(cand, dtype=np.int64)[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return j[j < n_vis]


def pool_topk(scores: np.ndarray, cand: np.ndarray, k: int, block: int = 8) -> np.ndarray:
    """Second level: a Reindex layer's own top-k inside the pool (R, C3:
    S = TopK over j in P of sigma^(l)(j)); same order and tie rule as
    topk_select, entry indices ascending, -1 padded."""
    s = np.asarray(scores, dtype=np.float64)
    P = pool_entries(cand, s.shape[0], block)
    sel = topk_select(s[P], k)
    return np.where(sel >= 0, P[np.maximum(sel, 0)], -1).astype(np.int64)


class CompressorState:
    """The compressor with its open group carried between calls.

    During decode an entry is emitted only once every m = compress_ratio
    tokens, and the partial group waits in state (R, section 3f, C2 "the
    compressor"; P, "The container": a step at a non-flush position writes
    nothing). Tokens of one sequence are fed in order, in chunks of any size;
    every group a chunk completes is compressed by `compress` above on its m
    tokens, so the result cannot depend on the chunking.
    """

    def __init__(self, m: int, norm_w, eps: float, inv_freq, w_idx=None, k_norm_w=None):
        self.m, self.norm_w, self.eps, self.inv_freq = m, norm_w, eps, inv_freq
        self.w_idx, self.k_norm_w = w_idx, k_norm_w
        self.next_pos = 0
        self.raw, self.gate = [], []

    def pending(self) -> int:
        return len(self.raw)

    def feed(self, raw, gate, first_pos: int):
        """raw / gate [n, D]: the tokens at positions first_pos .. first_pos+n-1.
        Returns [(j, kv_rotated, c_hat, k_idx)] for each group completed."""
        if first_pos != self.next_pos:
            raise ValueError("tokens must be fed in order")
        raw = np.asarray(raw, dtype=np.float64)
        gate = None if gate is None else np.asarray(gate, dtype=np.float64)
        out = []
        for i in range(raw.shape[0]):
            self.raw.append(raw[i])
            self.gate.append(None if gate is None else gate[i])
            if len(self.raw) == self.m:
                p0 = first_pos + i + 1 - self.m
                g = None if self.m == 1 else np.stack(self.gate)
                kv, c_hat, k_idx = compress(np.stack(self.raw), g, self.m, p0, self.norm_w, self.eps,
                                            self.inv_freq, self.w_idx, self.k_norm_w)
                out.append((p0 // self.m, kv[0], c_hat[0], None if k_idx is None else k_idx[0]))
                self.raw, self.gate = [], []
        self.next_pos = first_pos + raw.shape[0]
        return out


# ----------------------------------------------------------------------------
# Global KV bytes per token (R, section 3c, the B_glob formula; C2 "Resulting
# memory")
# ----------------------------------------------------------------------------

def global_kv_bytes_per_token(layers) -> float:
    """B_glob = sum over cache-producing layers of (main + index bytes) / m.

    layers: iterable of (bytes_main_entry, bytes_index_entry, m).
    """
    return float(sum((bm + bi) / m for bm, bi, m in layers))


def entry_bytes(dim: int, fmt: str) -> int:
    """Bytes of one stored row of `dim` channels in a storage format.

    'bf16': 2 bytes a channel; 'fp8_b32': one e4m3 byte a channel plus one
    ue8m0 byte per 32 channels; 'fp4_e4m3_b16': half a byte a channel plus one
    E4M3 scale byte per 16 channels (R, C2 "Resulting memory"); 'mxfp4_b32':
    half a byte a channel plus one E8M0 byte per 32 channels.
    """
    if fmt == "bf16":
        return 2 * dim
    if fmt == "fp8_b32":
        return dim + dim // 32
    if fmt == "fp4_e4m3_b16":
        return dim // 2 + dim // 16
    if fmt == "mxfp4_b32":
        return dim // 2 + dim // 32
    raise ValueError(fmt)


# ----------------------------------------------------------------------------
# Visibility and window bounds
# ----------------------------------------------------------------------------

def n_visible(t: int, m: int) -> int:
    """Number of compressed entries j with (j+1)*m - 1 <= t."""
    return (t + 1) // m


def window_positions(t: int, w: int, lo: int = 0) -> np.ndarray:
    """Raw-KV positions the query at t attends to: [max(lo, t-w+1), t]."""
    return np.arange(max(lo, t - w + 1), t + 1, dtype=np.int64)


# ----------------------------------------------------------------------------
# a2. Lightning indexer score (R, C2 step 2)
# ----------------------------------------------------------------------------

def index_scores(q_idx: np.ndarray, w_heads: np.ndarray, keys: np.ndarray) -> np.ndarray:
    """sigma(j) = sum_h w_h * max(0, q_h . k_j) for every row j of keys.

    q_idx [H_I, d_I], w_heads [H_I], keys [n, d_I]; returns float64 [n].
    """
    dots = np.asarray(keys, dtype=np.float64) @ np.asarray(q_idx, dtype=np.float64).T  # [n, H_I]
    return np.maximum(dots, 0.0) @ np.asarray(w_heads, dtype=np.float64)


# ----------------------------------------------------------------------------
# a3. Top-k selection (R, C2 step 2, S_t = TopK sigma_t)
# ----------------------------------------------------------------------------

def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest scores (ties to the lower index), ascending, -1 padded."""
    scores = np.asarray(scores)
    n = scores.shape[0]
    j = np.arange(n)
    # -0.0 and +0.0 are the same score
    key = np.where(scores == 0, 0.0, scores).astype(np.float64)
    order = np.lexsort((j, -key))  # primary: score descending; then index ascending
    chosen = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[:chosen.shape[0]] = chosen
    return out


# ----------------------------------------------------------------------------
# a4. Two-source attention with sink (R, 3a and C2 step 3; W item 1)
# ----------------------------------------------------------------------------

def attention_weights(q: np.ndarray, t: int, rows: np.ndarray, sink: np.ndarray, scale: float,
                      inv_freq: np.ndarray):
    """Softmax weights p[h, r] = e^{s_r} / (sum_r' e^{s_r'} + e^{sink_h}) and the log-denominator.

    q [H, D] (unrotated), rows [R, D], sink [H]; s_r = scale * RoPE_t(q_h) . row_r.
    A head whose logits and sink are all -inf gets zero weights and lse -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    rows = np.asarray(rows, dtype=np.float64).reshape(-1, q.shape[1])
    sink = np.asarray(sink, dtype=np.float64)
    qr = rope_rotate(q, t, inv_freq)
    s = scale * (qr @ rows.T)  # [H, R]
    mx = np.max(np.concatenate([s, sink[:, None]], axis=1), axis=1)  # [H]
    p = np.zeros_like(s)
    lse = np.full(q.shape[0], -np.inf)
    finite = np.isfinite(mx)
    if finite.any():
        e = np.exp(s[finite] - mx[finite, None])
        den = e.sum(axis=1) + np.exp(sink[finite] - mx[finite])
        p[finite] = e / den[:, None]
        lse[finite] = mx[finite] + np.log(den)
    return p, lse


def attend(q: np.ndarray, t: int, rows: np.ndarray, sink: np.ndarray, scale: float,
           inv_freq: np.ndarray):
    """One query over the concatenated rows (window rows then selected entries).

    q [H, D] (unrotated), rows [R, D] stored rows (already rotated at their own
    positions), sink [H]. Computes, per head h:
      q~ = RoPE_t(q_h);  s_r = scale * q~ . row_r;
      o_h = sum_r e^{s_r} row_r / (sum_r e^{s_r} + e^{sink_h});
      out_h = RoPE_{-t} applied to the rope dims of o_h.
    Returns (out [H, D] float64, lse [H] = log(sum_r e^{s_r} + e^{sink_h})).
    """
    rows = np.asarray(rows, dtype=np.float64).reshape(-1, np.asarray(q).shape[1])
    p, lse = attention_weights(q, t, rows, sink, scale, inv_freq)
    out = rope_rotate(p @ rows, t, inv_freq, inverse=True)
    return out, lse


def gather_rows(t: int, geom: Geometry, win_rows_by_pos, comp_rows: np.ndarray,
                sel: np.ndarray, win_lo: int = 0) -> np.ndarray:
    """Window rows at [max(lo, t-w+1), t] followed by comp_rows[sel[sel >= 0]]."""
    wp = window_positions(t, geom.window, win_lo)
    parts = [np.asarray(win_rows_by_pos(wp), dtype=np.float64).reshape(len(wp), -1)]
    sel = np.asarray(sel)
    sel = sel[sel >= 0]
    if sel.size:
        parts.append(np.asarray(comp_rows, dtype=np.float64)[sel])
    return np.concatenate(parts, axis=0)


# ----------------------------------------------------------------------------
# a5. One layer step per query under the three modes (R, C2 step 4)
# ----------------------------------------------------------------------------

MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2


def step_query(mode: int, geom: Geometry, inv_freq: np.ndarray, *, q, t, win_rows_by_pos,
               comp_rows, sink, q_idx=None, w_heads=None, idx_keys=None, sel=None,
               win_lo: int = 0):
    """One query of one layer.

    Full and Reindex score the visible entries with their own indexer query
    and select their own top-k; Reuse takes `sel` from the layer it borrows
    from. (Full additionally writes its compressed entries first; that is the
    compress() call, which the caller makes before this one.) All three then
    attend with their own q and window. Returns (out, lse, sel, scores).
    """
    scores = None
    if mode in (MODE_FULL, MODE_REINDEX):
        nv = n_visible(t, geom.compress_ratio)
        scores = index_scores(q_idx, w_heads, np.asarray(idx_keys)[:nv])
        sel = topk_select(scores, geom.topk)
    elif sel is None:
        raise ValueError("Reuse needs the borrowed selection")
    rows = gather_rows(t, geom, win_rows_by_pos, comp_rows, sel, win_lo)
    out, lse = attend(q, t, rows, sink, geom.softmax_scale, inv_freq)
    return out, lse, sel, scores
