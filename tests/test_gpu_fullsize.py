"""Full-size parity: the CSA2 layer step on each workload at its real size, in
the launch configuration the benchmark times (csa2_step over the whole
batch), checked on sampled queries that the float64 oracle recomputes one by
one from the same generator inputs.

Per sampled query:
  - the compressed entry written at this step (Full mode) against the
    oracle's compress of the same tokens;
  - index scores over every visible entry (score tolerance);
  - the selection: equal to the oracle's, or differing only among entries
    whose oracle scores tie with the threshold within the score tolerance;
  - attention: the step's own output when the selections are equal, and in
    every case csa2_attend run on the oracle's selection (oracle -> GPU).
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import (FMT_BF16, FMT_FP8, SCALE_BLOCK, assert_attention_close, assert_rows_close_stored,
                        attention_bound, bf16_np, check_topk_valid, code_bytes, context, f32_np, geometry, inv_freq,
                        oracle_stored, require_gpu, score_tolerance, storage_bound)
from oracle import csa2_oracle as O
from workloads import PRESETS, make_inputs

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"


def _to_stored(ctx, x, dim, fmt):
    """fp32 generator rows stored by csa2_store_rows in format `fmt` (codes, scales)."""
    codes = torch.empty((x.shape[0], code_bytes(dim, fmt)), dtype=torch.uint8, device=DEV)
    sc = torch.empty((x.shape[0], dim // SCALE_BLOCK[fmt]), dtype=torch.uint8, device=DEV)
    step = 1 << 20
    for i in range(0, x.shape[0], step):
        ctx.store_rows(x[i:i + step], None, fmt, codes[i:i + step], sc[i:i + step])
    return codes, sc


class Case:
    """GPU inputs of one layer of a workload, stored in the context's formats."""

    def __init__(self, ctx, wl, layer=0, base=None):
        inp = make_inputs(wl, DEV, layer=layer, with_compress=(layer == 0))
        if base is not None:  # a Reuse layer borrows the pool, keys and visibility
            for k in ("pool_off", "pool_kv", "pool_scale", "pool_kv_f32", "idx_keys", "idx_key_scale",
                      "idx_keys_f32", "n_vis", "q_idx", "w_heads"):
                if k in base.inp:
                    inp[k] = base.inp[k]
        if wl.kv_fp8:
            inp["win_kv"], inp["win_scale"] = _to_stored(ctx, inp["win_kv_f32"], 512, FMT_FP8)
            if base is None:
                inp["pool_kv"], inp["pool_scale"] = _to_stored(ctx, inp["pool_kv_f32"], 512, wl.kv_format)
        if wl.idx_fp8 and base is None:
            inp["idx_keys"], inp["idx_key_scale"] = _to_stored(ctx, inp["idx_keys_f32"], 128, wl.idx_key_format)
        torch.cuda.synchronize()
        self.inp, self.wl = inp, wl


def _step(ctx, case, mode, topk_idx):
    from compressed_sparse_attention_gb300 import binding
    i, wl = case.inp, case.wl
    Q = wl.n_query
    max_vis = int(i["n_vis"].max())
    out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = binding.workspace(ctx.step_workspace_size(Q, max_vis), DEV)
    full = mode == binding.MODE_FULL
    ctx.step(mode, wl.n_seq, max_vis, q=i["q"], q_pos=i["q_pos"], seq_of_q=i["seq_of_q"], n_vis=i["n_vis"],
             sink=i["sink"], win_kv=i["win_kv"], win_scale=i.get("win_scale"), win_off=i["win_off"],
             pool_kv=i["pool_kv"], pool_scale=i.get("pool_scale"), pool_off=i["pool_off"], topk_idx=topk_idx,
             out=out, workspace=ws, q_idx=i.get("q_idx"), w_heads=i.get("w_heads"), idx_keys=i.get("idx_keys"),
             idx_key_scale=i.get("idx_key_scale"), raw=i["raw"] if full else None,
             gate=i["gate"] if full else None, tok_off=i["tok_off"] if full else None,
             first_pos=i["first_pos"] if full else None, norm_w=i["norm_w"] if full else None,
             w_idx=i["w_idx"] if full else None, k_norm_w=i["k_norm_w"] if full else None)
    flags, st = ctx.check()
    assert flags == 0 and st == 0, f"device error word 0x{flags:x}"
    scores = ws[: Q * max_vis * 4].view(torch.float32).view(Q, max_vis)
    return out, scores


def _oracle_rows(src_f32, src_bf16, fmt):
    """The oracle's own copy of stored rows from the generator values (bf16
    rows are drawn as bf16; the scaled formats from fp32 values)."""
    if fmt == FMT_BF16:
        return bf16_np(src_bf16)
    return oracle_stored(f32_np(src_f32), fmt)


def _check_query(ctx, case, qi, geom, f, out_step, scores_step, sel_step, oracle_state, tag, borrowed=None):
    """Score / selection / attention checks of one sampled query. A Reuse layer
    passes `borrowed` = (the oracle's own selection of the layer it borrows
    from, whether the GPU's selection matched it). Returns (selection, same)."""
    i, wl = case.inp, case.wl
    b = int(i["seq_of_q"][qi])
    t = int(i["q_pos"][qi])
    nv = int(i["n_vis"][qi])
    # the generator's visibility against the oracle's own rule (entry j is
    # visible at t iff its group has closed), so that a wrong rule in the
    # generator cannot pass on both sides
    assert nv == O.n_visible(t, wl.m), f"{tag} q{qi}: n_vis {nv} but the oracle's rule gives {O.n_visible(t, wl.m)}"
    keys, pool, new_rng, key_step = oracle_state(b)
    woff = i["win_off"].cpu().numpy()
    cap = int(woff[b + 1] - woff[b])
    win_rows = _oracle_rows(i.get("win_kv_f32", None)[woff[b]:woff[b + 1]] if wl.kv_fp8 else None,
                            i["win_kv"][woff[b]:woff[b + 1]] if not wl.kv_fp8 else None, int(wl.kv_fp8))
    q = bf16_np(i["q"][qi])
    sink = f32_np(i["sink"])
    if scores_step is not None:
        qv, w = bf16_np(i["q_idx"][qi]), f32_np(i["w_heads"][qi])
        ref_s = O.index_scores(qv, w, keys[:nv])
        tol = score_tolerance(ref_s, qv, w, keys[:nv])
        # entries compressed at this step: the GPU's stored key may sit one
        # storage step (key_step, per element) from the oracle's
        j0, j1 = new_rng
        j1 = min(j1, nv)
        if j1 > j0:
            tol[j0:j1] += (np.abs(w)[None, :] * (key_step[j0:j1] @ np.abs(qv).T)).sum(axis=1)
        got_s = f32_np(scores_step[qi, :nv])
        bad = np.abs(got_s - ref_s) > tol
        assert not bad.any(), f"{tag} q{qi}: {int(bad.sum())} scores off"
        sel_ref = O.topk_select(ref_s, geom.topk)
        same = check_topk_valid(sel_step[qi], sel_ref, ref_s, tol)
    else:
        sel_ref, same = borrowed
    chosen = sel_ref[sel_ref >= 0]
    pool_rows = pool[chosen]  # only the selected rows, read on demand
    rows = O.gather_rows(t, geom, lambda p: win_rows[p % cap], pool_rows, np.arange(chosen.shape[0]))
    ref, _ = O.attend(q, t, rows, sink, geom.softmax_scale, f)
    bnd = attention_bound(q, t, rows, sink, geom.softmax_scale, f)
    if same:
        assert_attention_close(bf16_np(out_step[qi]), ref, bnd, f"{tag} q{qi} (step)")
    # csa2_attend on the oracle's selection, same buffers
    from compressed_sparse_attention_gb300 import binding
    sel_t = torch.tensor(sel_ref[None, :], dtype=torch.int32, device=DEV)
    o1 = torch.empty((1, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = binding.workspace(ctx.attend_workspace_size(1), DEV)
    ctx.attend(wl.n_seq, i["q"][qi:qi + 1].contiguous(), i["q_pos"][qi:qi + 1].contiguous(),
               i["seq_of_q"][qi:qi + 1].contiguous(), i["win_kv"], i.get("win_scale"), i["win_off"], None,
               i["pool_kv"], i.get("pool_scale"), i["pool_off"], sel_t, i["sink"], o1, None, ws)
    assert ctx.check()[0] == 0
    assert_attention_close(bf16_np(o1[0]), ref, bnd, f"{tag} q{qi} (oracle selection)")
    return sel_ref, same


def _full_state(ctx, case, geom, f):
    """Per sequence: the oracle's keys and pool, with the groups compressed at this step."""
    i, wl = case.inp, case.wl
    poff = i["pool_off"].cpu().numpy()
    tok_off = i["tok_off"].cpu().numpy()
    kfmt, pfmt = wl.idx_key_format, wl.kv_format
    cache = {}

    def state(b):
        if b in cache:
            return cache[b]
        r0, r1 = int(poff[b]), int(poff[b + 1])
        keys = _oracle_rows(i.get("idx_keys_f32", None)[r0:r1] if wl.idx_fp8 else None,
                            i["idx_keys"][r0:r1] if not wl.idx_fp8 else None, kfmt)
        pool_src = i.get("pool_kv_f32") if wl.kv_fp8 else i["pool_kv"]
        t0, t1 = int(tok_off[b]), int(tok_off[b + 1])
        j0 = int(i["first_pos"][b]) // wl.m
        g = (t1 - t0) // wl.m
        new_rows, key_step = None, None
        if g:
            kv, _, kidx = O.compress(bf16_np(i["raw"][t0:t1]), f32_np(i["gate"][t0:t1]), wl.m,
                                     int(i["first_pos"][b]), f32_np(i["norm_w"]), geom.norm_eps, f,
                                     bf16_np(i["w_idx"]), f32_np(i["k_norm_w"]))
            # the GPU's stored forms of the new entries against the exact values,
            # and the oracle's own stored forms in the state it scores with
            new = slice(r0 + j0, r0 + j0 + g)
            k_sc = i.get("idx_key_scale")[new] if kfmt != FMT_BF16 else None
            p_sc = i.get("pool_scale")[new] if pfmt != FMT_BF16 else None
            assert_rows_close_stored(i["idx_keys"][new], k_sc, kidx, kfmt, f"keys seq {b}")
            assert_rows_close_stored(i["pool_kv"][new], p_sc, kv, pfmt, f"kv seq {b}")
            keys[j0:j0 + g] = oracle_stored(kidx, kfmt)
            new_rows = oracle_stored(kv, pfmt)
            # the GPU's stored key and the oracle's each lie within one bound of
            # the exact key
            key_step = np.zeros_like(keys)
            key_step[j0:j0 + g] = 2.0 * storage_bound(kidx, k_sc, kfmt)
        pool = _LazyPool(pool_src, r0, r1, pfmt, j0, new_rows)
        cache[b] = (keys, pool, (j0, j0 + g), key_step)
        return cache[b]

    return state


class _LazyPool:
    """The oracle's view of one sequence's pool rows, read from the generator
    values on demand (a 1M-context pool is 256K rows), with this step's new
    entries in the oracle's own stored form."""

    def __init__(self, src, r0, r1, fmt, j0, new_rows):
        self.src, self.r0, self.n, self.fmt, self.j0, self.new = src, r0, r1 - r0, fmt, j0, new_rows

    def __getitem__(self, idx):
        idx = np.asarray(idx)
        rows = self.src[torch.as_tensor(self.r0 + idx, device=self.src.device)]
        vals = _oracle_rows(rows, rows, self.fmt)
        if self.new is not None:
            hit = (idx >= self.j0) & (idx < self.j0 + self.new.shape[0])
            vals[hit] = self.new[idx[hit] - self.j0]
        return vals


def _run_full(preset, sample):
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS[preset]
    ctx = context(compress_ratio=wl.m, idx_heads=wl.idx_heads, kv_format=wl.kv_format,
                  idx_key_format=wl.idx_key_format)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    case = Case(ctx, wl)
    idx = torch.empty((wl.n_query, wl.topk), dtype=torch.int32, device=DEV)
    out, scores = _step(ctx, case, binding.MODE_FULL, idx)
    sel = idx.cpu().numpy()
    state = _full_state(ctx, case, geom, f)
    return [_check_query(ctx, case, qi, geom, f, out, scores, sel, state, preset)[1] for qi in sample]


def test_fullsize_tiny_decode():
    """Batch 1 at 4,096 context, ratio 4 (1,024 entries), q and KV ~ N(0,1)/sqrt(512),
    seed 0: the one query of the batch, through csa2_step as the benchmark
    runs it."""
    same = _run_full("tiny_decode", [0])
    assert all(same), "the tiny decode's selection differs from the oracle's"


def test_fullsize_decode_64k_b32():
    same = _run_full("decode_64k_b32", [0, 13, 31])
    assert sum(same) >= 2


def test_fullsize_decode_1m_b8_fp8():
    same = _run_full("decode_1m_b8_fp8", [0, 7])
    assert sum(same) >= 1


def test_fullsize_decode_1m_b8_fp4():
    """fp4 pool rows, an fp8 window and mxfp4 keys at 1M context."""
    same = _run_full("decode_1m_b8_fp4", [0, 7])
    assert sum(same) >= 1


def test_fullsize_prefill_4k_after_8k():
    same = _run_full("prefill_4k_after_8k", [0, 1, 2047, 4095])
    assert sum(same) >= 3


def test_fullsize_mixed_reindex_then_reuse():
    """One Reindex layer, then three Reuse layers with their own q, window and
    sink, borrowing the pool and the Reindex layer's selection."""
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    wl = PRESETS["mixed_reuse_b64"]
    ctx = context(compress_ratio=wl.m, idx_heads=wl.idx_heads)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    lens = np.array(wl.ctx_len)
    sample = [int(np.argmax(lens)), int(np.argmin(lens)), 17]
    print(f"mixed batch: {wl.n_seq} sequences, {int(lens.sum())} entries, sampled lengths {lens[sample].tolist()}")
    base = Case(ctx, wl)
    idx = torch.empty((wl.n_query, wl.topk), dtype=torch.int32, device=DEV)
    out, scores = _step(ctx, base, binding.MODE_REINDEX, idx)
    sel = idx.cpu().numpy()
    poff = base.inp["pool_off"].cpu().numpy()

    def state(b):
        r0, r1 = int(poff[b]), int(poff[b + 1])
        keys = bf16_np(base.inp["idx_keys"][r0:r1])
        return keys, _LazyPool(base.inp["pool_kv"], r0, r1, False, 0, None), (0, 0), None

    oracle_sel = {qi: _check_query(ctx, base, qi, geom, f, out, scores, sel, state, "reindex") for qi in sample}
    for layer in (1, 2, 3):
        reuse = Case(ctx, wl, layer=layer, base=base)
        out_l, _ = _step(ctx, reuse, binding.MODE_REUSE, idx)
        for qi in sample:
            _check_query(ctx, reuse, qi, geom, f, out_l, None, sel, state, f"reuse{layer}", borrowed=oracle_sel[qi])
    assert sum(s for _, s in oracle_sel.values()) >= 2
