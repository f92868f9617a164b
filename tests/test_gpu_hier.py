"""The hierarchical sparse indexer on the GPU against the oracle
("Reading Notes of DeepSeek-V4.1-Flash", 3f C3; PocketLLM "The container").

* csa2_candidate_pool: bit-exact block pools on identical fp32 scores (ties
  between blocks, the pinned newest block, short and empty rows, rows that
  need the cluster top-k over block scores).
* csa2_index_score_pool: pool-only scores against the oracle's on the same
  pool; n_pool exact.
* csa2_topk_pool: bit-exact entry indices on identical fp32 pool scores.
* A Full step as candidate source followed by a Reindex step reading the
  pool: the pool against the oracle's own (equal up to near-tied blocks), the
  Reindex selection and attention against the oracle.
"""
import numpy as np
import pytest
import torch

from gpu_common import (assert_attention_close, attention_bound, bf16_np, check_topk_valid, context, f32_np,
                        geometry, inv_freq, oracle_stored, require_gpu, score_tolerance)
from oracle import csa2_oracle as O
from workloads import Workload, make_inputs, make_topk_scores

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("n,tie_levels,keep", [(1000, 0, 2048), (16384, 0, 2048), (40000, 0, 2048),
                                               (40000, 3, 2048), (262144, 0, 2048), (5000, 2, 64),
                                               (5000, 0, 1)])
def test_candidate_pool_bit_exact(n, tie_levels, keep):
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context(cand_keep=keep)
    Q = 4
    sc = make_topk_scores(Q, n, seed=300 + n + tie_levels + keep, tie_levels=tie_levels)
    nv = torch.tensor([n, n - 5, 17, 0], dtype=torch.int32)
    cand = torch.full((Q, keep), -7, dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.candidate_pool_workspace_size(Q, n), DEV)
    ctx.candidate_pool(sc.to(DEV), nv.to(DEV), n, cand, ws)
    assert ctx.check()[0] == 0
    got = cand.cpu().numpy()
    s = sc.double().numpy()
    for qi in range(Q):
        ref = O.candidate_blocks(s[qi, :int(nv[qi])], 8, keep)
        assert np.array_equal(got[qi, :ref.shape[0]], ref), f"query {qi}"
        assert np.all(got[qi, ref.shape[0]:] == -1)


def _pool_case(n_vis, keep, seed):
    """A valid pool per query from generator scores (oracle's candidate_blocks)."""
    rng = np.random.default_rng(seed)
    cands = []
    for n in n_vis:
        c = O.candidate_blocks(rng.standard_normal(n), 8, keep)
        cands.append(np.concatenate([c, np.full(keep - c.shape[0], -1)]))
    return np.stack(cands).astype(np.int32)


@pytest.mark.parametrize("fmt", [0, 1, 3], ids=["bf16", "fp8", "mxfp4"])
def test_index_score_pool(fmt):
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    keep = 128
    ctx = context(cand_keep=keep, idx_key_format=fmt)
    wl = Workload("pool", 3, (40000, 3001, 9000), 4, seed=310 + fmt, idx_fp8=fmt != 0, key_fp4=fmt == 3)
    inp = make_inputs(wl, DEV, with_compress=False)
    Q = wl.n_query
    nv = inp["n_vis"]
    cand = _pool_case(nv.tolist(), keep, 311 + fmt)
    if fmt == 0:
        keys, ksc = inp["idx_keys"], None
        keys_np = bf16_np(keys)
    else:
        kf = inp["idx_keys_f32"]
        dim_b = 128 if fmt == 1 else 64
        keys = torch.empty((kf.shape[0], dim_b), dtype=torch.uint8, device=DEV)
        ksc = torch.empty((kf.shape[0], 4), dtype=torch.uint8, device=DEV)
        ctx.store_rows(kf, None, fmt, keys, ksc)
        keys_np = oracle_stored(f32_np(kf), fmt)
    ldc = keep * 8
    scores = torch.full((Q, ldc), float("nan"), device=DEV)
    n_pool = torch.full((Q,), -1, dtype=torch.int32, device=DEV)
    ctx.index_score_pool(wl.n_seq, inp["q_idx"], inp["w_heads"], keys, ksc, inp["pool_off"], inp["seq_of_q"], nv,
                         int(nv.max()), torch.tensor(cand, device=DEV), scores, n_pool)
    assert ctx.check()[0] == 0
    s = f32_np(scores)
    poff = inp["pool_off"].cpu().numpy()
    for qi in range(Q):
        b, n = int(inp["seq_of_q"][qi]), int(nv[qi])
        P = O.pool_entries(cand[qi][cand[qi] >= 0], n)
        assert int(n_pool[qi]) == P.shape[0]
        qv, w = bf16_np(inp["q_idx"][qi]), f32_np(inp["w_heads"][qi])
        kk = keys_np[poff[b] + P]
        ref = O.index_scores(qv, w, kk)
        assert np.all(np.abs(s[qi, :P.shape[0]] - ref) <= score_tolerance(ref, qv, w, kk)), f"query {qi}"
        assert np.all(np.isnan(s[qi, P.shape[0]:]))


@pytest.mark.parametrize("n,keep,k,tie_levels", [(30000, 2048, 512, 0), (30000, 2048, 512, 4), (5000, 64, 100, 0),
                                                 (700, 2048, 512, 0)])
def test_topk_pool_bit_exact(n, keep, k, tie_levels):
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context(cand_keep=keep)
    Q = 3
    full = make_topk_scores(Q, n, seed=320 + n + keep + tie_levels, tie_levels=tie_levels).double().numpy()
    nv = [n, n - 3, 300]
    ldc = keep * 8
    cand = np.full((Q, keep), -1, dtype=np.int32)
    comp = np.zeros((Q, ldc), dtype=np.float32)
    n_pool = np.zeros(Q, dtype=np.int32)
    for qi in range(Q):
        c = O.candidate_blocks(full[qi, :nv[qi]], 8, keep)
        cand[qi, :c.shape[0]] = c
        P = O.pool_entries(c, nv[qi])
        comp[qi, :P.shape[0]] = full[qi, P]
        n_pool[qi] = P.shape[0]
    out = torch.empty((Q, k), dtype=torch.int32, device=DEV)
    ws = binding.workspace(ctx.topk_workspace_size(Q, ldc), DEV)
    ctx.topk_pool(torch.tensor(comp, device=DEV), torch.tensor(n_pool, device=DEV), torch.tensor(cand, device=DEV),
                  k, out, ws)
    assert ctx.check()[0] == 0
    got = out.cpu().numpy()
    for qi in range(Q):
        ref = O.pool_topk(full[qi, :nv[qi]], cand[qi][cand[qi] >= 0], k)
        assert np.array_equal(got[qi], ref), f"query {qi}"


def _blocks_valid(got, ref, block_scores, tol):
    """The GPU's pool differs from the oracle's only among blocks whose oracle
    score is within `tol` of the weakest kept block's (near ties)."""
    a, b = set(int(x) for x in got if x >= 0), set(int(x) for x in ref)
    assert len(a) == len(b)
    if a == b:
        return True
    thr = min(block_scores[list(b - {max(b)})]) if len(b) > 1 else -np.inf
    for blk in a ^ b:
        assert abs(block_scores[blk] - thr) <= 2 * tol[blk] + 1e-30, f"block {blk} is not a near tie"
    return False


def test_step_candidate_source_then_pool_reader():
    """Layer 1: a Full decode step that is the candidate source (its pool of
    256 blocks of 8 written beside its attention). Layer 2: a Reindex step
    with its own q, q^I, weights, window and sink that scores and selects
    only inside that pool."""
    from compressed_sparse_attention_gb300 import binding
    from test_gpu_fullsize import Case, _full_state
    require_gpu()
    keep = 256
    wl = Workload("hier", 2, (70000, 52000), 4, seed=330, n_layers=2, value_std=1.0 / 22.6, outlier_frac=0.01)
    ctx = context(cand_keep=keep)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    c1 = Case(ctx, wl)
    c2 = Case(ctx, wl, layer=1, base=c1)
    g = torch.Generator(device=DEV).manual_seed(331)
    q_idx2 = torch.randn((wl.n_query, 8, 128), generator=g, device=DEV).to(torch.bfloat16)
    w2 = torch.rand((wl.n_query, 8), generator=g, device=DEV)
    i1, i2 = c1.inp, c2.inp
    Q = wl.n_query
    max_vis = int(i1["n_vis"].max())
    cand = torch.full((Q, keep), -7, dtype=torch.int32, device=DEV)

    def run(case, mode, role, q_idx, w, idx, out):
        i = case.inp
        ws = binding.workspace(ctx.step_workspace_size(Q, max_vis), DEV)
        full = mode == binding.MODE_FULL
        ctx.step(mode, wl.n_seq, max_vis, q=i["q"], q_pos=i["q_pos"], seq_of_q=i["seq_of_q"], n_vis=i["n_vis"],
                 sink=i["sink"], win_kv=i["win_kv"], win_off=i["win_off"], pool_kv=i1["pool_kv"],
                 pool_off=i1["pool_off"], topk_idx=idx, out=out, workspace=ws, q_idx=q_idx, w_heads=w,
                 idx_keys=i1["idx_keys"], raw=i["raw"] if full else None, gate=i["gate"] if full else None,
                 tok_off=i["tok_off"] if full else None, first_pos=i["first_pos"] if full else None,
                 norm_w=i["norm_w"] if full else None, w_idx=i["w_idx"] if full else None,
                 k_norm_w=i["k_norm_w"] if full else None, cand_role=role, cand=cand)
        assert ctx.check() == (0, 0)

    idx1 = torch.empty((Q, 512), dtype=torch.int32, device=DEV)
    out1 = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    run(c1, binding.MODE_FULL, binding.CAND_SOURCE, i1["q_idx"], i1["w_heads"], idx1, out1)
    idx2 = torch.empty_like(idx1)
    out2 = torch.empty_like(out1)
    run(c2, binding.MODE_REINDEX, binding.CAND_READ, q_idx2, w2, idx2, out2)
    state = _full_state(ctx, c1, geom, f)
    cand_np, sel2 = cand.cpu().numpy(), idx2.cpu().numpy()
    checked = 0
    for qi in range(Q):
        b, t, nv = int(i1["seq_of_q"][qi]), int(i1["q_pos"][qi]), int(i1["n_vis"][qi])
        keys, pool, _, _ = state(b)
        # layer 1's pool against the oracle's own
        qv1, wv1 = bf16_np(i1["q_idx"][qi]), f32_np(i1["w_heads"][qi])
        s1 = O.index_scores(qv1, wv1, keys[:nv])
        tol1 = score_tolerance(s1, qv1, wv1, keys[:nv])
        cand_o = O.candidate_blocks(s1, 8, keep)
        nb = -(-nv // 8)
        bmax = np.array([s1[8 * k:8 * k + 8].max() for k in range(nb)])
        btol = np.array([tol1[8 * k:8 * k + 8].max() for k in range(nb)])
        same_pool = _blocks_valid(cand_np[qi], cand_o, bmax, btol)
        assert np.all(np.diff(cand_np[qi][cand_np[qi] >= 0]) > 0)
        if not same_pool:
            continue
        # layer 2: its own scores inside the pool, selection and attention
        qv2, wv2 = bf16_np(q_idx2[qi]), f32_np(w2[qi])
        s2 = O.index_scores(qv2, wv2, keys[:nv])
        tol2 = score_tolerance(s2, qv2, wv2, keys[:nv])
        sel_o = O.pool_topk(s2, cand_o, 512)
        P = set(O.pool_entries(cand_o, nv).tolist())
        assert set(int(x) for x in sel2[qi] if x >= 0) <= P
        masked = np.where(np.isin(np.arange(nv), list(P)), s2, -np.inf)
        same = check_topk_valid(sel2[qi], sel_o, masked, tol2)
        if same:
            chosen = sel_o[sel_o >= 0]
            woff = i2["win_off"].cpu().numpy()
            cap = int(woff[b + 1] - woff[b])
            win_rows = bf16_np(i2["win_kv"][woff[b]:woff[b + 1]])
            rows = O.gather_rows(t, geom, lambda p_: win_rows[p_ % cap], pool[chosen], np.arange(chosen.shape[0]))
            q = bf16_np(i2["q"][qi])
            ref, _ = O.attend(q, t, rows, f32_np(i2["sink"]), geom.softmax_scale, f)
            bnd = attention_bound(q, t, rows, f32_np(i2["sink"]), geom.softmax_scale, f)
            assert_attention_close(bf16_np(out2[qi]), ref, bnd, f"reindex q{qi}")
            checked += 1
    assert checked >= 1, "no query had the oracle's pool and selection"
