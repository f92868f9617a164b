"""The pool-sharded step (compressed_sparse_attention_gb300.sharded) on one
GPU, G = 4 shards run in one process: each shard scans and selects over its
quarter of every sequence's pool, the (score, entry) pairs and the (m, l, O)
partials are exchanged by stacking, and every shard combines.

Checked:
  - each shard's local scores equal the unsharded scan's scores of the same
    entries bit for bit, so the merged selection is compared with csa2_topk
    over identical scores: it must be equal, index for index;
  - every shard ends with the same selection and the same output bits;
  - the combined output against the float64 oracle over the window and the
    selected rows (the attention tolerance), and lse within its bound (the
    bf16 weights the denominator sums, and the fp32 scores);
  - a shard that holds none of a short sequence's entries, and shards
    without the window, contribute empty partials;
  - the partial attention over the same selection with its columns shuffled
    (no shard's entries form one run of columns) meets the same bounds.
"""
import numpy as np
import pytest
import torch

from gpu_common import (assert_attention_close, attention_bound, bf16_np, context, f32_np, geometry, inv_freq,
                        lse_bound, require_gpu, stored_values)
from oracle import csa2_oracle as O
from test_gpu_fullsize import Case
from workloads import Workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
G = 4


@pytest.mark.parametrize("fp8", [False, True])
def test_sharded_step_equals_unsharded(fp8):
    require_gpu()
    from compressed_sparse_attention_gb300 import binding, sharded
    wl = Workload(f"sharded_{int(fp8)}", 3, (36000, 20000, 4100), 4, seed=1500 + int(fp8), kv_fp8=fp8, idx_fp8=fp8,
                  outlier_frac=0.01)
    ctx = context(kv_format=wl.kv_format, idx_key_format=wl.idx_key_format)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    case = Case(ctx, wl)
    i = case.inp
    Q, K = wl.n_query, wl.topk
    max_vis = int(i["n_vis"].max())
    full = torch.empty((Q, max_vis), dtype=torch.float32, device=DEV)
    ctx.index_score(wl.n_seq, i["q_idx"], i["w_heads"], i["idx_keys"], i.get("idx_key_scale"), i["pool_off"],
                    i["seq_of_q"], i["n_vis"], max_vis, full)
    sel_full = torch.empty((Q, K), dtype=torch.int32, device=DEV)
    ops = sharded.ContextOps(ctx)
    ctx.topk(full, i["n_vis"], max_vis, K, sel_full, ops.topk_workspace(Q, max_vis))
    shards = [sharded.shard_inputs(i, wl.n_seq, G, g) for g in range(G)]
    # each shard's local scores are the unsharded scores of its entries
    nv = i["n_vis"].tolist()
    for s in shards:
        w = max(1, s.hi - s.lo)
        nvl = torch.empty(Q, dtype=torch.int32, device=DEV)
        ctx.shard_visible(s.n_vis, s.lo, s.hi, nvl)
        loc = torch.empty((Q, w), dtype=torch.float32, device=DEV)
        ctx.index_score(s.n_seq, s.q_idx, s.w_heads, s.idx_keys, s.idx_key_scale, s.pool_off, s.seq_of_q, nvl, w, loc)
        for q in range(Q):
            n = int(nvl[q])
            assert n == max(0, min(nv[q] - s.lo, s.hi - s.lo))
            assert torch.equal(loc[q, :n].view(torch.int32), full[q, s.lo:s.lo + n].view(torch.int32))
    results = sharded.run_local([sharded.shard_step(ops, s, K) for s in shards])
    assert ctx.check() == (0, 0)
    out, lse, sel = results[0]
    for o2, l2, s2 in results[1:]:
        assert torch.equal(s2, sel) and torch.equal(o2.view(torch.int16), out.view(torch.int16))
        assert torch.equal(l2, lse)
    assert torch.equal(sel, sel_full), "the merged selection differs from csa2_topk's on the same scores"
    # the same selection with its columns shuffled: the partial attention then
    # cannot take a shard's entries as one run of columns and goes over every
    # column; the combined output must meet the same bounds
    perm = torch.stack([torch.randperm(K, generator=torch.Generator().manual_seed(77 + q)) for q in range(Q)])
    sel_p = torch.gather(sel, 1, perm.to(DEV)).contiguous()
    parts = []
    for s_ in shards:
        po = torch.empty((Q, 64, 512), dtype=torch.float32, device=DEV)
        pm = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
        pl = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
        ctx.attend_partial(s_.n_seq, s_.q, s_.q_pos, s_.seq_of_q, s_.with_window, s_.win_kv, s_.win_scale, s_.win_off,
                           s_.win_lo, s_.pool_kv, s_.pool_scale, s_.pool_off, sel_p, s_.lo, s_.hi, po, pm, pl)
        parts.append((po, pm, pl))
    out_p = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    lse_p = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
    ctx.attend_combine(*(torch.stack([pt[c] for pt in parts]) for c in range(3)), i["q_pos"], i["sink"], out_p, lse_p)
    assert ctx.check() == (0, 0)
    # the combined output against the oracle
    fmt = wl.kv_format
    sink = f32_np(i["sink"])
    poff, woff = i["pool_off"].tolist(), i["win_off"].tolist()
    for q in range(Q):
        b, t = int(i["seq_of_q"][q]), int(i["q_pos"][q])
        win = (stored_values(i["win_kv"][woff[b]:woff[b + 1]], i["win_scale"][woff[b]:woff[b + 1]], 1) if fp8
               else bf16_np(i["win_kv"][woff[b]:woff[b + 1]]))
        chosen = sel[q].cpu().numpy()
        chosen = chosen[chosen >= 0]
        prow = poff[b] + torch.as_tensor(chosen, device=DEV)
        pool = (stored_values(i["pool_kv"][prow], i["pool_scale"][prow], fmt) if fp8 else bf16_np(i["pool_kv"][prow]))
        cap = woff[b + 1] - woff[b]
        rows = O.gather_rows(t, geom, lambda p: win[p % cap], pool, np.arange(chosen.shape[0]))
        qv = bf16_np(i["q"][q])
        ref, ref_lse = O.attend(qv, t, rows, sink, geom.softmax_scale, f)
        for o_, l_, tag in ((out, lse, "sharded"), (out_p, lse_p, "sharded, shuffled selection")):
            assert_attention_close(bf16_np(o_[q]), ref, attention_bound(qv, t, rows, sink, geom.softmax_scale, f),
                                   f"{tag} q{q}")
            d_lse, lb = np.abs(f32_np(l_[q]) - ref_lse), lse_bound(qv, t, rows, geom.softmax_scale, f)
            assert np.all(d_lse <= lb), (f"{tag} q{q}: lse off by {float(d_lse.max()):.3e} at head "
                                         f"{int(np.argmax(d_lse - lb))}, bound {float(lb[np.argmax(d_lse - lb)]):.3e}; "
                                         f"gpu {float(f32_np(l_[q])[np.argmax(d_lse - lb)]):.6f} "
                                         f"oracle {float(ref_lse[np.argmax(d_lse - lb)]):.6f} rows {rows.shape[0]}")
