"""The calls of compressed_sparse_attention_gb300.sharded.shard_step, done by
the float64 oracle on CPU tensors, for testing the sharded step's
orchestration and exchanges on CPU ranks (no GPU). Test infrastructure only.

Each method fills its output tensors as the C entry point of the same name
would: scores as fp32, selections as int32, partials (O, m, l) as fp32 with
m in natural-log units, the combined output as bf16.
"""
import numpy as np
import torch

from oracle import csa2_oracle as O
from oracle import formats as F


def _bf(t):
    return F.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy().view(np.uint16))


class OracleOps:
    def __init__(self, geom: O.Geometry, inv_freq: np.ndarray):
        self.geom, self.f = geom, inv_freq

    def shard_visible(self, n_vis, lo, hi, out):
        out.copy_(torch.clamp(n_vis.long() - lo, 0, hi - lo).to(torch.int32))

    def index_score(self, n_seq, q_idx, w_heads, idx_keys, idx_key_scale, pool_off, seq_of_q, n_vis, max_vis, scores):
        keys = _bf(idx_keys)
        for q in range(q_idx.shape[0]):
            b, nv = int(seq_of_q[q]), int(n_vis[q])
            r0 = int(pool_off[b])
            s = O.index_scores(_bf(q_idx[q]), w_heads[q].double().numpy(), keys[r0:r0 + nv])
            scores[q, :nv] = torch.from_numpy(s).to(torch.float32)

    def topk_workspace(self, n_query, max_vis):
        return None

    def topk(self, scores, n_vis, max_vis, k, out_idx, ws):
        for q in range(scores.shape[0]):
            nv = int(n_vis[q])
            out_idx[q] = torch.from_numpy(O.topk_select(scores[q, :nv].double().numpy(), k))

    def topk_pairs(self, scores, sel, base, pair_score, pair_idx):
        for q in range(sel.shape[0]):
            for i, j in enumerate(sel[q].tolist()):
                pair_score[q, i] = scores[q, j] if j >= 0 else float("-inf")
                pair_idx[q, i] = base + j if j >= 0 else -1

    def topk_merge(self, all_score, all_idx, k, out_idx):
        for q in range(all_idx.shape[1]):
            idx = all_idx[:, q, :].reshape(-1)
            sc = all_score[:, q, :].reshape(-1)
            keep = idx >= 0
            idx, sc = idx[keep], sc[keep]
            order = torch.argsort(idx)  # the union in entry order, so the oracle's tie rule is by entry
            idx, sc = idx[order], sc[order]
            pos = O.topk_select(sc.double().numpy(), k)
            out_idx[q] = torch.from_numpy(np.where(pos >= 0, idx.numpy()[np.maximum(pos, 0)], -1).astype(np.int32))

    def attend_partial(self, n_seq, q, q_pos, seq_of_q, with_window, win_kv, win_scale, win_off, win_lo, pool_kv,
                       pool_scale, pool_off, sel, lo, hi, part_o, part_m, part_l):
        g = self.geom
        pool = _bf(pool_kv)
        win = _bf(win_kv) if with_window else None
        for qi in range(q.shape[0]):
            b, t = int(seq_of_q[qi]), int(q_pos[qi])
            rows = []
            if with_window:
                w0, w1 = int(win_off[b]), int(win_off[b + 1])
                for p in O.window_positions(t, g.window):
                    rows.append(win[w0 + p % (w1 - w0)])
            for j in sel[qi].tolist():
                if lo <= j < hi:
                    rows.append(pool[int(pool_off[b]) + j - lo])
            if not rows:
                part_o[qi] = 0.0
                part_m[qi] = float("-inf")
                part_l[qi] = 0.0
                continue
            rows = np.stack(rows)
            qr = O.rope_rotate(_bf(q[qi]), t, self.f)
            s = g.softmax_scale * (qr @ rows.T)  # [H, R]
            m = s.max(axis=1)
            e = np.exp(s - m[:, None])
            part_o[qi] = torch.from_numpy(e @ rows).to(torch.float32)
            part_m[qi] = torch.from_numpy(m).to(torch.float32)
            part_l[qi] = torch.from_numpy(e.sum(axis=1)).to(torch.float32)

    def attend_combine(self, all_o, all_m, all_l, q_pos, sink, out, lse):
        sk = sink.double().numpy()
        for qi in range(all_o.shape[1]):
            m = all_m[:, qi].double().numpy()   # [G, H]
            lv = all_l[:, qi].double().numpy()
            o = all_o[:, qi].double().numpy()   # [G, H, D]
            M = np.maximum(m.max(axis=0), sk)
            w = np.where(np.isfinite(m), np.exp(m - M[None, :]), 0.0)
            den = (w * lv).sum(axis=0) + np.exp(sk - M)
            res = (w[:, :, None] * o).sum(axis=0) / den[:, None]
            res = O.rope_rotate(res, int(q_pos[qi]), self.f, inverse=True)
            out[qi] = torch.from_numpy(F.round_bf16(res)).to(torch.float32).to(torch.bfloat16)
            lse[qi] = torch.from_numpy(M + np.log(den)).to(torch.float32)
