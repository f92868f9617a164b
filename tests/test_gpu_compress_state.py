"""The compressor with its open group carried in device state
(csa2_compress_append, and csa2_step with append), against the oracle.

* Fed all at once, token by token, or in random chunks, the compressed pool
  rows and index keys come out bit-identical (the same arithmetic on the same
  values), and the open group's tokens sit in their state slots.
* A chunked prefill and the same positions decoded token by token, with the
  top-k untruncated (k >= every n_vis), leave bit-identical pool rows, keys
  and selections; their attention outputs agree with the oracle and with each
  other within the attention tolerance (the two forms group the attention
  sums differently: decode splits a query's tiles over CTAs and merges them).
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import (FMT_BF16, SCALE_BLOCK, assert_attention_close, assert_rows_close_stored, attention_bound,
                        bf16_np, code_bytes, context, f32_np, geometry, inv_freq, require_gpu)
from oracle import csa2_oracle as O

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buffers(rows, dim, fmt):
    if fmt == FMT_BF16:
        return torch.zeros((rows, dim), dtype=torch.bfloat16, device=DEV), None
    return (torch.zeros((rows, code_bytes(dim, fmt)), dtype=torch.uint8, device=DEV),
            torch.zeros((rows, dim // SCALE_BLOCK[fmt]), dtype=torch.uint8, device=DEV))


def _weights(g):
    norm_w = 0.5 + torch.rand(512, generator=g, device=DEV)
    w_idx = (torch.randn((128, 512), generator=g, device=DEV) / math.sqrt(512)).to(torch.bfloat16)
    k_norm_w = 0.5 + torch.rand(128, generator=g, device=DEV)
    return norm_w, w_idx, k_norm_w


class _Cache:
    def __init__(self, n_seq, m, cap, kv_fmt, key_fmt):
        self.pool, self.psc = _buffers(n_seq * cap, 512, kv_fmt)
        self.keys, self.ksc = _buffers(n_seq * cap, 128, key_fmt)
        self.st_raw = torch.zeros((n_seq, m, 512), dtype=torch.bfloat16, device=DEV)
        self.st_gate = torch.zeros((n_seq, m, 512), dtype=torch.float32, device=DEV)
        self.pool_off = torch.arange(0, n_seq + 1, dtype=torch.int64, device=DEV) * cap

    def same(self, other):
        pairs = [(self.pool, other.pool), (self.keys, other.keys)]
        pairs += [(a, b) for a, b in ((self.psc, other.psc), (self.ksc, other.ksc)) if a is not None]
        return all(torch.equal(a, b) for a, b in pairs)


def _feed(ctx, cache, seqs, chunks, weights):
    """seqs: per sequence (raw [L,512] bf16, gate [L,512] fp32); chunks: a list
    of calls, each a list of per-sequence token counts."""
    pos = [0] * len(seqs)
    for counts in chunks:
        raw = torch.cat([seqs[b][0][pos[b]:pos[b] + c] for b, c in enumerate(counts)])
        gate = torch.cat([seqs[b][1][pos[b]:pos[b] + c] for b, c in enumerate(counts)])
        tok_off = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64, device=DEV)
        first = torch.tensor(pos, dtype=torch.int64, device=DEV)
        ctx.compress_append(raw.contiguous(), gate.contiguous(), len(seqs), tok_off, first, cache.pool_off,
                            *weights, cache.pool, cache.psc, cache.keys, cache.ksc, cache.st_raw, cache.st_gate)
        pos = [p + c for p, c in zip(pos, counts)]
    assert ctx.check()[0] == 0


@pytest.mark.parametrize("m", [2, 4])
@pytest.mark.parametrize("fmts", [(0, 0), (1, 1), (2, 3)], ids=["bf16", "fp8", "fp4_mxfp4"])
def test_compress_append_chunking_is_bit_identical(m, fmts):
    require_gpu()
    kv_fmt, key_fmt = fmts
    ctx = context(compress_ratio=m, kv_format=kv_fmt, idx_key_format=key_fmt)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    g = torch.Generator(device=DEV).manual_seed(70 + m + 10 * kv_fmt)
    lens = [61, 18, 37]
    seqs = [(torch.randn((L, 512), generator=g, device=DEV).to(torch.bfloat16),
             torch.randn((L, 512), generator=g, device=DEV) * 2) for L in lens]
    weights = _weights(g)
    cap = max(lens) // m + 2
    one, each, rand = (_Cache(3, m, cap, kv_fmt, key_fmt) for _ in range(3))
    _feed(ctx, one, seqs, [lens], weights)
    _feed(ctx, each, seqs, [[1 if i < L else 0 for L in lens] for i in range(max(lens))], weights)
    rng = np.random.default_rng(m)
    left, calls = list(lens), []
    while any(left):
        c = [int(min(x, rng.integers(0, 6))) for x in left]
        calls.append(c)
        left = [x - y for x, y in zip(left, c)]
    _feed(ctx, rand, seqs, calls, weights)
    assert one.same(each) and one.same(rand), "chunked and one-shot compress differ"
    for b, L in enumerate(lens):
        done = (L // m) * m
        # open group in the state, slot pos mod m
        for p in range(done, L):
            assert torch.equal(one.st_raw[b, p % m], seqs[b][0][p])
            assert torch.equal(one.st_gate[b, p % m], seqs[b][1][p])
        # complete groups against the oracle
        kv, _, kidx = O.compress(bf16_np(seqs[b][0][:done]), f32_np(seqs[b][1][:done]), m, 0, f32_np(weights[0]),
                                 geom.norm_eps, f, bf16_np(weights[1]), f32_np(weights[2]))
        rows = slice(b * cap, b * cap + L // m)
        assert_rows_close_stored(one.pool[rows], None if one.psc is None else one.psc[rows], kv, kv_fmt, f"kv {b}")
        assert_rows_close_stored(one.keys[rows], None if one.ksc is None else one.ksc[rows], kidx, key_fmt,
                                 f"key {b}")
        # rows past the last complete group are untouched
        assert float(one.pool[b * cap + L // m:(b + 1) * cap].float().abs().sum()) == 0.0


def test_prefill_equals_token_by_token_decode_untruncated():
    """600 prefix tokens compressed, then positions 600..899 either as one
    chunked-prefill Full step (300 queries, 300 new tokens) or as 300 decode
    Full steps of one query and one new token each; k = 512 >= n_vis <= 225."""
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    m, N, P = 4, 900, 600
    ctx = context(compress_ratio=m)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    g = torch.Generator(device=DEV).manual_seed(77)
    raw = torch.randn((N, 512), generator=g, device=DEV).to(torch.bfloat16)
    gate = torch.randn((N, 512), generator=g, device=DEV) * 2
    win = (torch.randn((N, 512), generator=g, device=DEV) / math.sqrt(512)).to(torch.bfloat16)
    Qn = N - P
    q = (torch.randn((Qn, 64, 512), generator=g, device=DEV) / 22.6).to(torch.bfloat16)
    q_idx = torch.randn((Qn, 8, 128), generator=g, device=DEV).to(torch.bfloat16)
    w_heads = torch.rand((Qn, 8), generator=g, device=DEV)
    sink = torch.randn(64, generator=g, device=DEV)
    weights = _weights(g)
    cap = N // m
    win_off = torch.tensor([0, N], dtype=torch.int64, device=DEV)
    zero1 = torch.zeros(1, dtype=torch.int64, device=DEV)

    a = _Cache(1, m, cap, FMT_BF16, FMT_BF16)
    _feed(ctx, a, [(raw[:P], gate[:P])], [[P]], weights)
    b = _Cache(1, m, cap, FMT_BF16, FMT_BF16)
    for dst, src in ((b.pool, a.pool), (b.keys, a.keys), (b.st_raw, a.st_raw), (b.st_gate, a.st_gate)):
        dst.copy_(src)

    def step(cache, t0, t1, out, idx):
        n_q = t1 - t0
        pos = torch.arange(t0, t1, dtype=torch.int64, device=DEV)
        n_vis = ((pos + 1) // m).to(torch.int32)
        max_vis = int((t1) // m)
        ws = binding.workspace(ctx.step_workspace_size(n_q, max_vis), DEV)
        ctx.step(binding.MODE_FULL, 1, max_vis, q=q[t0 - P:t1 - P], q_pos=pos,
                 seq_of_q=torch.zeros(n_q, dtype=torch.int32, device=DEV), n_vis=n_vis, sink=sink, win_kv=win,
                 win_off=win_off, pool_kv=cache.pool, pool_off=cache.pool_off, topk_idx=idx, out=out,
                 workspace=ws, q_idx=q_idx[t0 - P:t1 - P], w_heads=w_heads[t0 - P:t1 - P], idx_keys=cache.keys,
                 raw=raw[t0:t1], gate=gate[t0:t1],
                 tok_off=torch.tensor([0, n_q], dtype=torch.int64, device=DEV), first_pos=zero1 + t0,
                 norm_w=weights[0], w_idx=weights[1], k_norm_w=weights[2], append=True, state_raw=cache.st_raw,
                 state_gate=cache.st_gate)

    out_a = torch.empty((Qn, 64, 512), dtype=torch.bfloat16, device=DEV)
    idx_a = torch.empty((Qn, 512), dtype=torch.int32, device=DEV)
    step(a, P, N, out_a, idx_a)
    assert ctx.check() == (0, 0)
    out_b = torch.empty_like(out_a)
    idx_b = torch.empty_like(idx_a)
    for t in range(P, N):
        step(b, t, t + 1, out_b[t - P:t - P + 1], idx_b[t - P:t - P + 1])
    assert ctx.check() == (0, 0)

    assert a.same(b), "prefill and token-by-token decode left different compressed caches"
    assert torch.equal(idx_a, idx_b)
    for t in (P, P + 1, P + 3, 777, N - 1):
        nv = (t + 1) // m
        sel = idx_a[t - P].cpu().numpy()
        assert np.array_equal(sel[:nv], np.arange(nv)) and np.all(sel[nv:] == -1)
    # the oracle on sampled queries: every visible entry plus the window
    kv, _, _ = O.compress(bf16_np(raw), f32_np(gate), m, 0, f32_np(weights[0]), geom.norm_eps, f,
                          bf16_np(weights[1]), f32_np(weights[2]))
    pool_np = bf16_np(a.pool[:cap])
    assert np.all(np.abs(pool_np - kv) <= np.abs(kv) * 2.0 ** -7 + 1e-6)
    win_np = bf16_np(win)
    for t in (P, P + 3, 777, N - 1):
        nv = (t + 1) // m
        rows = O.gather_rows(t, geom, lambda p_: win_np[p_], pool_np[:nv], np.arange(nv))
        qv = bf16_np(q[t - P])
        ref, _ = O.attend(qv, t, rows, f32_np(sink), geom.softmax_scale, f)
        bnd = attention_bound(qv, t, rows, f32_np(sink), geom.softmax_scale, f)
        assert_attention_close(bf16_np(out_a[t - P]), ref, bnd, f"prefill t={t}")
        assert_attention_close(bf16_np(out_b[t - P]), ref, bnd, f"decode t={t}")
    oa, ob = bf16_np(out_a), bf16_np(out_b)
    rel = np.linalg.norm(oa - ob) / np.linalg.norm(oa)
    assert rel <= 1e-2 and np.abs(oa - ob).max() <= 2e-2
