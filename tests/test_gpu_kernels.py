"""GPU parity of each CSA2 kernel against the float64 oracle on identical seeded inputs.

Sizes here are ones the oracle finishes in seconds while still spanning
several tiles and ragged tails; full-size checks are in test_gpu_fullsize.py.
"""
import math

import numpy as np
import pytest
import torch

from gpu_common import (FMT_BF16, SCALE_BLOCK, assert_attention_close, attention_bound, assert_rows_close_bf16, lse_bound,
                        assert_rows_close_fp8, assert_rows_close_stored, bf16_np, check_topk_valid, code_bytes,
                        context, f32_np, geometry, inv_freq, oracle_fp8_rows, require_gpu, rope_sanity,
                        score_tolerance)
from oracle import csa2_oracle as O
from oracle import formats as F
from workloads import Workload, make_inputs, make_selection, make_topk_scores

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(autouse=True)
def _gpu():
    require_gpu()


# ----------------------------------------------------------------------------- storage / rope

@pytest.mark.parametrize("dim", [512, 128])
def test_store_rows_bf16_and_fp8_bit_exact_without_rope(dim):
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn((333, dim), generator=g, device=DEV) * torch.exp(torch.randn((333, 1), generator=g, device=DEV) * 3)
    x[7] = 0.0
    x[9, :32] = 0.0
    out = torch.empty((333, dim), dtype=torch.bfloat16, device=DEV)
    ctx.store_rows(x, None, binding.KV_BF16, out)
    ref = F.f64_to_bf16_bits(f32_np(x))
    assert np.array_equal(out.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    codes = torch.empty((333, dim), dtype=torch.uint8, device=DEV)
    sc = torch.empty((333, dim // 32), dtype=torch.uint8, device=DEV)
    ctx.store_rows(x, None, binding.KV_FP8, codes, sc)
    rc, re_, _ = oracle_fp8_rows(f32_np(x))
    assert np.array_equal(sc.cpu().numpy(), re_)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert ctx.check()[0] == 0


def test_store_rows_rope_matches_oracle():
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    rope_sanity(ctx)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    g = torch.Generator(device=DEV).manual_seed(6)
    x = torch.randn((200, 512), generator=g, device=DEV)
    pos = torch.randint(0, 1 << 20, (200,), generator=g, device=DEV)
    pos[0] = 0
    pos[1] = (1 << 20) - 1
    out = torch.empty((200, 512), dtype=torch.bfloat16, device=DEV)
    ctx.store_rows(x, pos, binding.KV_BF16, out)
    ref = O.rope_rotate(f32_np(x), pos.cpu().numpy(), f)
    assert_rows_close_bf16(bf16_np(out), ref, "rope store bf16")
    codes = torch.empty((200, 512), dtype=torch.uint8, device=DEV)
    sc = torch.empty((200, 16), dtype=torch.uint8, device=DEV)
    ctx.store_rows(x, pos, binding.KV_FP8, codes, sc)
    got = F.fp8_block_dequantize(codes.cpu().numpy(), sc.cpu().numpy())
    assert_rows_close_fp8(got, ref, F.ue8m0_to_f64(sc.cpu().numpy()), "rope store fp8")


# ----------------------------------------------------------------------------- attention

def _attend_case(wl, ctx, fp8=False, win_lo=None, sel_seed=11, layer=0):
    """Run csa2_attend on workload wl with a random valid selection; return (gpu out, lse, oracle refs)."""
    from compressed_sparse_attention_gb300 import binding
    inp = make_inputs(wl, DEV, layer=layer, with_compress=False)
    if layer > 0:
        base = make_inputs(wl, DEV, layer=0, with_compress=False)
        for k in ("pool_off", "pool_kv", "pool_kv_f32", "n_vis"):
            if k in base:
                inp[k] = base[k]
    sel = make_selection(wl, inp["n_vis"], sel_seed, DEV)
    B, Q = wl.n_seq, wl.n_query
    if fp8:
        win = torch.empty(inp["win_kv_f32"].shape, dtype=torch.uint8, device=DEV)
        win_sc = torch.empty((win.shape[0], 16), dtype=torch.uint8, device=DEV)
        ctx.store_rows(inp["win_kv_f32"], None, binding.KV_FP8, win, win_sc)
        pool = torch.empty(inp["pool_kv_f32"].shape, dtype=torch.uint8, device=DEV)
        pool_sc = torch.empty((pool.shape[0], 16), dtype=torch.uint8, device=DEV)
        ctx.store_rows(inp["pool_kv_f32"], None, binding.KV_FP8, pool, pool_sc)
    else:
        win, win_sc, pool, pool_sc = inp["win_kv"], None, inp["pool_kv"], None
    lo_t = None if win_lo is None else torch.tensor(win_lo, dtype=torch.int64, device=DEV)
    out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
    ws = binding.workspace(ctx.attend_workspace_size(Q), DEV)
    ctx.attend(B, inp["q"], inp["q_pos"], inp["seq_of_q"], win, win_sc, inp["win_off"], lo_t, pool, pool_sc,
               inp["pool_off"], sel, inp["sink"], out, lse, ws)
    flags, _ = ctx.check()
    assert flags == 0
    # oracle on the same inputs
    if fp8:
        win_np = oracle_fp8_rows(f32_np(inp["win_kv_f32"]))[2]
        pool_np = oracle_fp8_rows(f32_np(inp["pool_kv_f32"]))[2]
    else:
        win_np, pool_np = bf16_np(win), bf16_np(pool)
    return dict(inp=inp, sel=sel.cpu().numpy(), out=bf16_np(out), lse=f32_np(lse), win_np=win_np, pool_np=pool_np,
                win_lo=win_lo)


def _oracle_attend(case, geom, f, qi):
    inp = case["inp"]
    b = int(inp["seq_of_q"][qi])
    t = int(inp["q_pos"][qi])
    woff = inp["win_off"].cpu().numpy()
    poff = inp["pool_off"].cpu().numpy()
    cap = woff[b + 1] - woff[b]
    lo = 0 if case["win_lo"] is None else max(0, case["win_lo"][b])
    rows = O.gather_rows(t, geom, lambda p: case["win_np"][woff[b] + (p % cap)], case["pool_np"][poff[b]:poff[b + 1]],
                         case["sel"][qi], lo)
    q = bf16_np(inp["q"][qi])
    out, lse = O.attend(q, t, rows, f32_np(inp["sink"]), geom.softmax_scale, f)
    case["lse_bound"] = lse_bound(q, t, rows, geom.softmax_scale, f)
    return out, lse, attention_bound(q, t, rows, f32_np(inp["sink"]), geom.softmax_scale, f)


def test_attend_softmax_worked_example():
    """q = 1, k = (0, ln 3), v = (10, 20) gives 17.5 (the reading notes' worked example)."""
    from compressed_sparse_attention_gb300 import binding
    ctx = context(rope_dim=0, softmax_scale=1.0)
    win = torch.zeros((128, 512), dtype=torch.float32, device=DEV)
    t = 200
    win[(t - 1) % 128, 1] = 10.0
    win[t % 128, 0] = math.log(3.0)
    win[t % 128, 1] = 20.0
    # every other window position holds a row whose key is very negative
    other = [p for p in range(t - 127, t - 1)]
    for p in other:
        win[p % 128, 0] = -1000.0
    win_bf = torch.empty((128, 512), dtype=torch.bfloat16, device=DEV)
    ctx.store_rows(win, None, binding.KV_BF16, win_bf)
    q = torch.zeros((1, 64, 512), dtype=torch.bfloat16, device=DEV)
    q[0, :, 0] = 1.0
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device=DEV)
    sink = torch.full((64,), -math.inf, device=DEV)
    ctx.attend(1, q, torch.tensor([t], device=DEV), torch.zeros(1, dtype=torch.int32, device=DEV), win_bf, None,
               torch.tensor([0, 128], device=DEV), None, None, None, None, None, sink, out, None, None)
    assert ctx.check()[0] == 0
    o = bf16_np(out)[0]  # [64 heads, 512 channels]
    # ln 3 is stored as bf16 (1.1015625) and the output is rounded to bf16 (step 0.125 near 17.5)
    assert np.all(np.abs(o[:, 1] - 17.5) <= 0.07)
    assert np.all(np.abs(o[:, 0] - 0.75 * math.log(3.0)) <= 0.01)
    assert np.all(np.abs(o[:, 2:]) == 0)


@pytest.mark.parametrize("fp8", [False, True])
def test_attend_decode_ragged(fp8):
    ctx = context(kv_format=1 if fp8 else 0)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    wl = Workload("attend_ragged", 4, (300, 4100, 40, 2051), 4, seed=21, kv_fp8=fp8, outlier_frac=0.02)
    lo = [0, 4000, 0, 1990]
    case = _attend_case(wl, ctx, fp8=fp8, win_lo=lo)
    for qi in range(wl.n_query):
        ref, lse, bnd = _oracle_attend(case, geom, f, qi)
        assert_attention_close(case["out"][qi], ref, bnd, f"query {qi}")
        assert np.all(np.abs(case["lse"][qi] - lse) <= case["lse_bound"])


def test_attend_many_queries_single_split_rescale():
    """Prefill-shaped: 200 causal queries on one sequence with a linear window
    buffer -> one CTA per query runs all five tiles with the running max."""
    ctx = context(compress_ratio=2)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    wl = Workload("attend_prefill", 1, (2300,), 2, seed=22, n_query_per_seq=200, win_linear=True,
                  outlier_frac=0.05, outlier_scale=16.0)
    case = _attend_case(wl, ctx)
    for qi in (0, 1, 57, 123, 199):
        ref, _, bnd = _oracle_attend(case, geom, f, qi)
        assert_attention_close(case["out"][qi], ref, bnd, f"query {qi}")


@pytest.mark.parametrize("window_only", [False, True])
def test_attend_persistent_many_queries_ragged_and_invalid(window_only):
    """More queries than SMs over three sequences of different lengths: one
    CTA per SM takes queries c, c + SMs, c + 2 SMs, ... and prefetches each
    next query while it stores the current one. The shortest sequence's
    selections are -1 padded (fewer than 512 visible entries); one query's
    sequence index is out of range: its flag is raised, its output is the
    sink-only zero, and the queries after it on the same CTA are unaffected.
    Window-only: no selection, so every query is a single tile."""
    from compressed_sparse_attention_gb300 import binding
    ctx = context(compress_ratio=2)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = Workload("attend_persist", 3, (700, 1500, 2600), 2, seed=31, n_query_per_seq=120, win_linear=True)
    inp = make_inputs(wl, DEV, with_compress=False)
    sel = None if window_only else make_selection(wl, inp["n_vis"], 13, DEV)
    Q = wl.n_query
    bad = 40
    seq_of_q = inp["seq_of_q"].clone()
    seq_of_q[bad] = wl.n_seq + 2
    out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
    ws = binding.workspace(ctx.attend_workspace_size(Q), DEV)
    ctx.attend(wl.n_seq, inp["q"], inp["q_pos"], seq_of_q, inp["win_kv"], None, inp["win_off"], None,
               None if window_only else inp["pool_kv"], None, None if window_only else inp["pool_off"], sel,
               inp["sink"], out, lse, ws)
    flags, _ = ctx.check()
    assert flags == binding.FLAG_BAD_QUERY
    assert torch.count_nonzero(out[bad]) == 0
    sel_np = np.full((Q, 512), -1, dtype=np.int32) if window_only else sel.cpu().numpy()
    assert window_only or (sel_np[:120] == -1).any()  # padded selections in the short sequence
    case = dict(inp=inp, sel=sel_np, out=bf16_np(out), lse=f32_np(lse), win_np=bf16_np(inp["win_kv"]),
                pool_np=bf16_np(inp["pool_kv"]), win_lo=None)
    # the bad query's CTA mates, both ends of each sequence, and a second-round query
    for qi in sorted({bad - 1, bad + 1, bad + n_sm, bad + 2 * n_sm, 0, 119, 120, 239, 240, Q - 1, n_sm + 3}):
        if qi >= Q or qi == bad:
            continue
        ref, ref_lse, bnd = _oracle_attend(case, geom, f, qi)
        assert_attention_close(case["out"][qi], ref, bnd, f"query {qi}")
        assert np.all(np.abs(case["lse"][qi] - ref_lse) <= case["lse_bound"]), f"lse of query {qi}"


def test_attend_reports_bad_index_and_skips_row():
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    wl = Workload("attend_bad", 1, (4096,), 4, seed=23)
    inp = make_inputs(wl, DEV, with_compress=False)
    sel = make_selection(wl, inp["n_vis"], 1, DEV)
    sel[0, 3] = 1024  # == pool length: out of range
    out = torch.empty((1, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = binding.workspace(ctx.attend_workspace_size(1), DEV)
    ctx.attend(1, inp["q"], inp["q_pos"], inp["seq_of_q"], inp["win_kv"], None, inp["win_off"], None,
               inp["pool_kv"], None, inp["pool_off"], sel, inp["sink"], out, None, ws)
    flags, st = ctx.check()
    assert flags & binding.FLAG_BAD_TOPK_INDEX and st == 4
    assert torch.isfinite(out.float()).all()


# ----------------------------------------------------------------------------- indexer

@pytest.mark.parametrize("idx_heads", [8, 16, 32])
@pytest.mark.parametrize("fp8", [False, True])
def test_index_score(idx_heads, fp8):
    from compressed_sparse_attention_gb300 import binding
    ctx = context(idx_heads=idx_heads, idx_key_format=1 if fp8 else 0)
    wl = Workload("idx", 3, (4000, 148, 10404), 4, seed=31 + idx_heads, idx_heads=idx_heads, idx_fp8=fp8,
                  n_query_per_seq=2)
    inp = make_inputs(wl, DEV, with_compress=False)
    Q = wl.n_query
    nv = inp["n_vis"].clone()
    nv[1] = 7      # ragged, shorter than the pool
    nv[2] = 0      # nothing visible
    max_vis = int(nv.max())
    if fp8:
        keys = torch.empty(inp["idx_keys_f32"].shape, dtype=torch.uint8, device=DEV)
        ksc = torch.empty((keys.shape[0], 4), dtype=torch.uint8, device=DEV)
        ctx.store_rows(inp["idx_keys_f32"], None, binding.KV_FP8, keys, ksc)
        keys_np = oracle_fp8_rows(f32_np(inp["idx_keys_f32"]))[2]
    else:
        keys, ksc = inp["idx_keys"], None
        keys_np = bf16_np(keys)
    ld = max_vis + 5
    scores = torch.full((Q, ld), float("nan"), device=DEV)
    ctx.index_score(wl.n_seq, inp["q_idx"], inp["w_heads"], keys, ksc, inp["pool_off"], inp["seq_of_q"], nv,
                    max_vis, scores)
    assert ctx.check()[0] == 0
    s = f32_np(scores)
    poff = inp["pool_off"].cpu().numpy()
    for qi in range(Q):
        b = int(inp["seq_of_q"][qi])
        n = int(nv[qi])
        qv = bf16_np(inp["q_idx"][qi])
        w = f32_np(inp["w_heads"][qi])
        kk = keys_np[poff[b]:poff[b] + n]
        ref = O.index_scores(qv, w, kk)
        tol = score_tolerance(ref, qv, w, kk)
        assert np.all(np.abs(s[qi, :n] - ref) <= tol), f"query {qi}"
        assert np.all(np.isnan(s[qi, n:])), "entries past n_vis must stay untouched"


@pytest.mark.parametrize("idx_heads", [8, 16, 32])
@pytest.mark.parametrize("interleave", [False, True])
def test_index_score_many_queries(idx_heads, interleave):
    """Many queries per sequence take the tensor-core indexer: query blocks of
    256 / H_I queries against 128-key tiles. Interleaving two sequences makes
    every block mixed, which is scored on the CUDA cores instead."""
    ctx = context(idx_heads=idx_heads)
    n_seq = 2 if interleave else 1
    wl = Workload("idx_many", n_seq, (3000,) * n_seq if not interleave else (3000, 2200), 2,
                  seed=77 + idx_heads, idx_heads=idx_heads, n_query_per_seq=300 if not interleave else 160)
    inp = make_inputs(wl, DEV, with_compress=False)
    Q = wl.n_query
    perm = torch.randperm(Q, generator=torch.Generator().manual_seed(5)) if interleave else torch.arange(Q)
    perm = perm.to(DEV)
    q_idx, w, seq, nv = inp["q_idx"][perm].contiguous(), inp["w_heads"][perm].contiguous(), \
        inp["seq_of_q"][perm].contiguous(), inp["n_vis"][perm].clone()
    nv[5] = 0      # nothing visible
    nv[7] = 3      # ragged inside the first tile
    nv[40] = 129   # one key into the second tile
    max_vis = int(nv.max())
    ld = max_vis + 3
    scores = torch.full((Q, ld), float("nan"), device=DEV)
    ctx.index_score(wl.n_seq, q_idx, w, inp["idx_keys"], None, inp["pool_off"], seq, nv, max_vis, scores)
    assert ctx.check()[0] == 0
    s = f32_np(scores)
    keys_np = bf16_np(inp["idx_keys"])
    poff = inp["pool_off"].cpu().numpy()
    for qi in range(Q):
        b = int(seq[qi])
        n = int(nv[qi])
        qv = bf16_np(q_idx[qi])
        wv = f32_np(w[qi])
        kk = keys_np[poff[b]:poff[b] + n]
        ref = O.index_scores(qv, wv, kk)
        tol = score_tolerance(ref, qv, wv, kk)
        assert np.all(np.abs(s[qi, :n] - ref) <= tol), f"query {qi}"
        assert np.all(np.isnan(s[qi, n:])), "entries past n_vis must stay untouched"


# ----------------------------------------------------------------------------- top-k

@pytest.mark.parametrize("n,tie_levels,k", [(3000, 0, 512), (3000, 3, 512), (20000, 2, 512), (5000, 0, 2048),
                                            (777, 0, 1), (262144, 0, 512), (262144, 40, 512), (100, 0, 512),
                                            (20000, 1, 512), (40000, 0, 64), (300000, 0, 512), (300000, 7, 512),
                                            (16384, 0, 512), (16384, 1, 512), (16384, 6, 512), (8192, 2, 2048),
                                            (2047, 0, 512), (6001, 0, 100)])
def test_topk_bit_exact(n, tie_levels, k):
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    Q = 4
    sc = make_topk_scores(Q, n, seed=n + tie_levels + k, tie_levels=tie_levels)
    nv = torch.tensor([n, max(0, n - 1), min(n, k - 1 if k > 1 else 1), 0], dtype=torch.int32)
    scores = sc.to(DEV)
    out = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.topk_workspace_size(Q, n), DEV)
    ctx.topk(scores, nv.to(DEV), n, k, out, ws)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    s = sc.numpy()
    for qi in range(Q):
        ref = O.topk_select(s[qi, :int(nv[qi])], k)
        assert np.array_equal(got[qi], ref), f"query {qi}"


def _floats_from_keys(keys):
    """float32 scores whose order-preserving keys are `keys` (the inverse of
    the map the selection orders by: positive floats have the top key bit
    set, negative ones are inverted)."""
    keys = np.asarray(keys, dtype=np.uint32)
    bits = np.where(keys & 0x80000000, keys & 0x7FFFFFFF, ~keys).astype(np.uint32)
    return bits.view(np.float32)


@pytest.mark.parametrize("case", ["normal", "huge_max", "bin_exact", "threshold_ties", "negative", "all_equal"])
def test_topk_decode_row_paths(case):
    """Rows of 8,193 .. 16,384 scores (the decode form, 1,024 threads a row),
    shaped to take each path of its search: the two relative levels
    (normal), the fallback radix search when the k largest reach more than
    2^24 key steps below the largest (huge_max), a first-level bin that holds
    exactly the keys still needed (bin_exact), many ties at the threshold
    value (threshold_ties, all_equal), and negative scores. Bit-exact against
    the oracle's selection on the same scores."""
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    k, n = 512, 16384
    lens = [16384, 12000, 8193]
    rng = np.random.default_rng({"normal": 1, "huge_max": 2, "bin_exact": 3, "threshold_ties": 4,
                                 "negative": 5, "all_equal": 6}[case])
    rows = []
    for r in range(len(lens)):
        x = rng.standard_normal(n).astype(np.float32)
        if case == "huge_max":
            x[rng.integers(0, lens[r])] = 1e30
        elif case == "bin_exact":
            top = np.uint32(0x80000000 | np.float32(50.0).view(np.uint32))
            keys = (top - np.uint32(1 << 25) - rng.integers(0, 1 << 20, n).astype(np.uint32)).astype(np.uint32)
            pos = rng.permutation(lens[r])[:k]
            keys[pos] = top - (np.arange(k, dtype=np.uint32) << np.uint32(12))
            x = _floats_from_keys(keys)
        elif case == "threshold_ties":
            x = np.abs(x)
            pos = rng.permutation(lens[r])
            x[pos[:400]] = 10.0
            x[pos[400:700]] = 9.0
        elif case == "negative":
            x = -np.abs(x) - 5.0
        elif case == "all_equal":
            x[:] = 3.25
        rows.append(x)
    sc = torch.from_numpy(np.stack(rows))
    nv = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((len(lens), k), dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.topk_workspace_size(len(lens), n), DEV)
    ctx.topk(sc.to(DEV), nv.to(DEV), n, k, out, ws)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    for qi, ln in enumerate(lens):
        ref = O.topk_select(rows[qi][:ln].astype(np.float64), k)
        assert np.array_equal(got[qi], ref), f"row {qi} (n {ln})"


@pytest.mark.parametrize("n", [100000, 262144])
@pytest.mark.parametrize("case", ["normal", "huge_max", "bin_exact", "rank", "threshold_ties", "negative",
                                  "all_equal"])
def test_topk_cluster_row_paths(case, n):
    """Rows of 100,000 and 262,144 scores (one cluster of 7 or 8 CTAs a row),
    shaped to take each path of the cluster search: the two relative levels
    (normal), the digit levels from the top bit when the k largest reach
    more than 2^24 key steps below the largest (huge_max), a first-level bin
    that holds exactly the keys still needed (bin_exact), at most 256 keys at
    the threshold ranked directly (rank), more ties at the threshold value
    (threshold_ties, all_equal), and negative scores. Bit-exact against the
    oracle's selection on the same scores."""
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    k = 512
    lens = [n, n - 12345, n // 2 + 7]
    rng = np.random.default_rng({"normal": 11, "huge_max": 12, "bin_exact": 13, "rank": 14, "threshold_ties": 15,
                                 "negative": 16, "all_equal": 17}[case] + n)
    rows = []
    for r in range(len(lens)):
        x = rng.standard_normal(n).astype(np.float32)
        if case == "huge_max":
            x[rng.integers(0, lens[r])] = 1e30
        elif case == "bin_exact":
            top = np.uint32(0x80000000 | np.float32(50.0).view(np.uint32))
            keys = (top - np.uint32(1 << 25) - rng.integers(0, 1 << 20, n).astype(np.uint32)).astype(np.uint32)
            pos = rng.permutation(lens[r])[:k]
            keys[pos] = top - (np.arange(k, dtype=np.uint32) << np.uint32(12))
            x = _floats_from_keys(keys)
        elif case in ("rank", "threshold_ties"):
            x = np.abs(x)
            pos = rng.permutation(lens[r])
            n_top = 450 if case == "rank" else 400
            x[pos[:n_top]] = 10.0
            x[pos[n_top:n_top + (100 if case == "rank" else 300)]] = 9.0
        elif case == "negative":
            x = -np.abs(x) - 5.0
        elif case == "all_equal":
            x[:] = 3.25
        rows.append(x)
    sc = torch.from_numpy(np.stack(rows))
    nv = torch.tensor(lens, dtype=torch.int32)
    out = torch.empty((len(lens), k), dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.topk_workspace_size(len(lens), n), DEV)
    ctx.topk(sc.to(DEV), nv.to(DEV), n, k, out, ws)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    for qi, ln in enumerate(lens):
        ref = O.topk_select(rows[qi][:ln].astype(np.float64), k)
        assert np.array_equal(got[qi], ref), f"row {qi} (n {ln})"


@pytest.mark.parametrize("n_lists,order", [(4, "ranges"), (16, "ranges"), (4, "shuffled"), (16, "shuffled")])
def test_topk_merge_lists(n_lists, order):
    """csa2_topk_merge over n_lists lists of 512 (score, entry) pairs per
    query, -1 padded at the ends, scores with ties: lists over ascending
    disjoint entry ranges (as shards and slices give them), and the same
    entries shuffled across and within the lists. The selection is the
    oracle's top-k over the union (entries mapped to a dense row in
    ascending order, so that ties still go to the lower entry), ascending,
    -1 padded; bit-exact."""
    ctx = context()
    k, k_in, Q = 512, 512, 3
    rng = np.random.default_rng(900 + n_lists + (order == "shuffled"))
    score = np.full((n_lists, Q, k_in), -np.inf, dtype=np.float32)
    idx = np.full((n_lists, Q, k_in), -1, dtype=np.int32)
    expect = []
    for q in range(Q):
        n_valid = [k_in - (rng.integers(0, 200) if (l + q) % 3 == 0 else 0) for l in range(n_lists)]
        span = 3000
        ents = np.concatenate([np.sort(rng.choice(span, n_valid[l], replace=False)) + l * span
                               for l in range(n_lists)]).astype(np.int32)
        sc = (np.round(rng.standard_normal(ents.shape[0]) * 8) / 8).astype(np.float32)  # many ties
        if order == "shuffled":
            perm = rng.permutation(ents.shape[0])
            ents, sc = ents[perm], sc[perm]
        pos = 0
        for l in range(n_lists):
            idx[l, q, :n_valid[l]] = ents[pos:pos + n_valid[l]]
            score[l, q, :n_valid[l]] = sc[pos:pos + n_valid[l]]
            pos += n_valid[l]
        o = np.argsort(ents, kind="stable")
        dense = O.topk_select(sc[o].astype(np.float64), k)
        expect.append(np.where(dense >= 0, ents[o][np.maximum(dense, 0)], -1))
    out = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ctx.topk_merge(torch.from_numpy(score).to(DEV), torch.from_numpy(idx).to(DEV), k, out)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    for q in range(Q):
        assert np.array_equal(got[q], expect[q]), f"query {q}"


@pytest.mark.parametrize("tie_levels", [0, 2])
def test_topk_many_queries_mixed_lengths(tie_levels):
    """More queries than the GPU holds top-k clusters for at once, with row
    lengths spread log-uniformly from 100 to 262,144 (and the edges: empty,
    k - 1, exactly the one-CTA limit and one past it): the selections are
    bit-exact against the oracle's, whichever path takes them."""
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    Q, n, k = 48, 262144, 512
    sc = make_topk_scores(Q, n, seed=4242 + tie_levels, tie_levels=tie_levels)
    rng = np.random.default_rng(7)
    lens = np.exp(rng.uniform(np.log(100), np.log(n), Q)).astype(np.int32)
    lens[:6] = [n, 0, k - 1, 16384, 16385, 100]
    scores = sc.to(DEV)
    out = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.topk_workspace_size(Q, n), DEV)
    ctx.topk(scores, torch.from_numpy(lens).to(DEV), n, k, out, ws)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    s = sc.numpy()
    for qi in range(Q):
        ref = O.topk_select(s[qi, :int(lens[qi])], k)
        assert np.array_equal(got[qi], ref), f"query {qi} (n_vis {lens[qi]})"


# ----------------------------------------------------------------------------- compressor

@pytest.mark.parametrize("m", [1, 2, 4])
@pytest.mark.parametrize("fmts", [(0, 0), (1, 1), (2, 3)], ids=["bf16", "fp8", "fp4_mxfp4"])
def test_compress(m, fmts):
    """Compressed entries and their index keys stored in each format pair
    (pool kv_format, index idx_key_format) against the oracle's exact values."""
    kv_fmt, key_fmt = fmts
    ctx = context(compress_ratio=m, kv_format=kv_fmt, idx_key_format=key_fmt)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    g = torch.Generator(device=DEV).manual_seed(40 + m)
    seg_groups = [3, 1, 5]
    first_group = [0, 17, 1000]
    T = sum(seg_groups) * m
    raw = torch.randn((T, 512), generator=g, device=DEV).to(torch.bfloat16)
    gate = torch.randn((T, 512), generator=g, device=DEV) * 2
    norm_w = 0.5 + torch.rand(512, generator=g, device=DEV)
    w_idx = (torch.randn((128, 512), generator=g, device=DEV) / math.sqrt(512)).to(torch.bfloat16)
    k_norm_w = 0.5 + torch.rand(128, generator=g, device=DEV)
    tok_off = torch.tensor(np.concatenate([[0], np.cumsum(seg_groups) * m]), dtype=torch.int64, device=DEV)
    first_pos = torch.tensor([x * m for x in first_group], dtype=torch.int64, device=DEV)
    plen = [first_group[i] + seg_groups[i] + 2 for i in range(3)]
    pool_off = torch.tensor(np.concatenate([[0], np.cumsum(plen)]), dtype=torch.int64, device=DEV)
    P = int(pool_off[-1])

    def buffers(dim, fmt):
        if fmt == FMT_BF16:
            return torch.zeros((P, dim), dtype=torch.bfloat16, device=DEV), None
        return (torch.zeros((P, code_bytes(dim, fmt)), dtype=torch.uint8, device=DEV),
                torch.zeros((P, dim // SCALE_BLOCK[fmt]), dtype=torch.uint8, device=DEV))

    pool, psc = buffers(512, kv_fmt)
    keys, ksc = buffers(128, key_fmt)
    ctx.compress(raw, gate if m > 1 else None, 3, tok_off, first_pos, pool_off, norm_w, w_idx, k_norm_w,
                 pool, psc, keys, ksc)
    assert ctx.check()[0] == 0
    raw_np, gate_np = bf16_np(raw), f32_np(gate)
    for b in range(3):
        t0, t1 = int(tok_off[b]), int(tok_off[b + 1])
        kv, c_hat, kidx = O.compress(raw_np[t0:t1], gate_np[t0:t1], m, int(first_pos[b]), f32_np(norm_w),
                                     geom.norm_eps, f, bf16_np(w_idx), f32_np(k_norm_w))
        r0 = int(pool_off[b]) + first_group[b]
        rows = slice(r0, r0 + seg_groups[b])
        assert_rows_close_stored(pool[rows], None if psc is None else psc[rows], kv, kv_fmt, f"kv seq {b}")
        assert_rows_close_stored(keys[rows], None if ksc is None else ksc[rows], kidx, key_fmt, f"key seq {b}")
        # rows outside the written groups stay untouched
        assert float(pool[int(pool_off[b]) + first_group[b] + seg_groups[b]].float().abs().sum()) == 0.0


@pytest.mark.parametrize("fmts", [(0, 0), (1, 1), (2, 3)], ids=["bf16", "fp8", "fp4_mxfp4"])
def test_compress_many_groups_equals_per_group(fmts):
    """A call with more than four groups an SM takes the compressor form that
    loads the index-key weights where it uses them (two CTAs an SM); the same
    groups compressed in calls of at most 300 groups take the form that holds
    them in registers. Both must store bit-identical pool rows and index keys
    (the same arithmetic in the same order), and the rows must match the
    oracle."""
    kv_fmt, key_fmt = fmts
    m = 2
    ctx = context(compress_ratio=m, kv_format=kv_fmt, idx_key_format=key_fmt)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    g = torch.Generator(device=DEV).manual_seed(77)
    seg_groups = [4 * n_sm + 37, 211, 5]
    first_group = [0, 3000, 17]
    T = sum(seg_groups) * m
    raw = torch.randn((T, 512), generator=g, device=DEV).to(torch.bfloat16)
    gate = torch.randn((T, 512), generator=g, device=DEV) * 2
    norm_w = 0.5 + torch.rand(512, generator=g, device=DEV)
    w_idx = (torch.randn((128, 512), generator=g, device=DEV) / math.sqrt(512)).to(torch.bfloat16)
    k_norm_w = 0.5 + torch.rand(128, generator=g, device=DEV)
    tok_off = np.concatenate([[0], np.cumsum(seg_groups) * m])
    plen = [first_group[i] + seg_groups[i] for i in range(3)]
    pool_off = torch.tensor(np.concatenate([[0], np.cumsum(plen)]), dtype=torch.int64, device=DEV)
    P = int(pool_off[-1])

    def buffers(dim, fmt):
        if fmt == FMT_BF16:
            return torch.zeros((P, dim), dtype=torch.bfloat16, device=DEV), None
        return (torch.zeros((P, code_bytes(dim, fmt)), dtype=torch.uint8, device=DEV),
                torch.zeros((P, dim // SCALE_BLOCK[fmt]), dtype=torch.uint8, device=DEV))

    def run(chunks):
        """chunks: per sequence, the group counts of successive calls"""
        pool, psc = buffers(512, kv_fmt)
        keys, ksc = buffers(128, key_fmt)
        done = [0, 0, 0]
        for step in range(max(len(c) for c in chunks)):
            # one call over every sequence, each with its groups of this step (maybe none)
            r_parts, g_parts, offs, firsts = [], [], [0], []
            for b in range(3):
                n = chunks[b][step] if step < len(chunks[b]) else 0
                t0 = int(tok_off[b]) + done[b] * m
                r_parts.append(raw[t0:t0 + n * m])
                g_parts.append(gate[t0:t0 + n * m])
                firsts.append((first_group[b] + done[b]) * m)
                offs.append(offs[-1] + n * m)
                done[b] += n
            ctx.compress(torch.cat(r_parts), torch.cat(g_parts), 3, torch.tensor(offs, dtype=torch.int64, device=DEV),
                         torch.tensor(firsts, dtype=torch.int64, device=DEV), pool_off, norm_w, w_idx, k_norm_w,
                         pool, psc, keys, ksc)
        assert ctx.check()[0] == 0
        return pool, psc, keys, ksc

    whole = run([[n] for n in seg_groups])
    small = run([[min(300, n - i) for i in range(0, n, 300)] for n in seg_groups])
    for a, b in zip(whole, small):
        if a is not None:
            assert torch.equal(a, b)
    pool, psc, keys, ksc = whole
    raw_np, gate_np = bf16_np(raw), f32_np(gate)
    for b in range(3):
        t0, t1 = int(tok_off[b]), int(tok_off[b + 1])
        kv, c_hat, kidx = O.compress(raw_np[t0:t1], gate_np[t0:t1], m, first_group[b] * m, f32_np(norm_w),
                                     geom.norm_eps, f, bf16_np(w_idx), f32_np(k_norm_w))
        r0 = int(pool_off[b]) + first_group[b]
        rows = slice(r0, r0 + seg_groups[b])
        assert_rows_close_stored(pool[rows], None if psc is None else psc[rows], kv, kv_fmt, f"kv seq {b}")
        assert_rows_close_stored(keys[rows], None if ksc is None else ksc[rows], kidx, key_fmt, f"key seq {b}")


def test_compress_rejects_misaligned_segment():
    from compressed_sparse_attention_gb300 import binding
    ctx = context(compress_ratio=4)
    raw = torch.zeros((8, 512), dtype=torch.bfloat16, device=DEV)
    gate = torch.zeros((8, 512), device=DEV)
    pool = torch.zeros((10, 512), dtype=torch.bfloat16, device=DEV)
    ctx.compress(raw, gate, 1, torch.tensor([0, 8], device=DEV), torch.tensor([2], device=DEV),
                 torch.tensor([0, 10], device=DEV), torch.ones(512, device=DEV), None, None, pool, None, None, None)
    flags, st = ctx.check()
    assert flags & binding.FLAG_BAD_SEGMENT and st == 4
    assert float(pool.float().abs().sum()) == 0.0
