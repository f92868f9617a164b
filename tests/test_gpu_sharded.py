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
    without the window, contribute empty partials.
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


def _slice_rows(t, rows):
    return None if t is None else t[rows].contiguous()


def _shards(wl, inp):
    from compressed_sparse_attention_gb300.sharded import ShardInputs, shard_range
    poff = inp["pool_off"].tolist()
    longest = max(poff[b + 1] - poff[b] for b in range(wl.n_seq))
    out = []
    for g in range(G):
        lo, hi = shard_range(longest, G, g)
        rows, off = [], [0]
        for b in range(wl.n_seq):
            a, e = poff[b] + lo, min(poff[b + 1], poff[b] + hi)
            rows.extend(range(a, max(a, e)))
            off.append(len(rows))
        r = torch.tensor(rows if rows else [0], dtype=torch.long, device=DEV)
        first = g == 0
        out.append(ShardInputs(
            lo=lo, hi=hi, with_window=first, n_seq=wl.n_seq, q=inp["q"], q_pos=inp["q_pos"],
            seq_of_q=inp["seq_of_q"], n_vis=inp["n_vis"], q_idx=inp["q_idx"], w_heads=inp["w_heads"],
            sink=inp["sink"], pool_off=torch.tensor(off, dtype=torch.int64, device=DEV),
            pool_kv=_slice_rows(inp["pool_kv"], r), pool_scale=_slice_rows(inp.get("pool_scale"), r),
            idx_keys=_slice_rows(inp["idx_keys"], r), idx_key_scale=_slice_rows(inp.get("idx_key_scale"), r),
            win_kv=inp["win_kv"] if first else None, win_scale=inp.get("win_scale") if first else None,
            win_off=inp["win_off"] if first else None))
    return out


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
    shards = _shards(wl, i)
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
        assert_attention_close(bf16_np(out[q]), ref, attention_bound(qv, t, rows, sink, geom.softmax_scale, f),
                               f"sharded q{q}")
        d_lse, lb = np.abs(f32_np(lse[q]) - ref_lse), lse_bound(qv, t, rows, geom.softmax_scale, f)
        assert np.all(d_lse <= lb), (f"q{q}: lse off by {float(d_lse.max()):.3e} at head {int(np.argmax(d_lse - lb))}, "
                                     f"bound {float(lb[np.argmax(d_lse - lb)]):.3e}; "
                                     f"gpu {float(f32_np(lse[q])[np.argmax(d_lse - lb)]):.6f} "
                                     f"oracle {float(ref_lse[np.argmax(d_lse - lb)]):.6f} rows {rows.shape[0]}")
