"""The pool-sharded step's orchestration and its two exchanges on two CPU
ranks (gloo), no GPU: each rank runs compressed_sparse_attention_gb300.
sharded.shard_step on its half of each sequence's pool through
run_distributed (all-gathers of the (score, entry) pairs and of the
(m, l, O) partials), with the oracle standing in for the kernels
(tests/sharded_oracle_ops.py). Both ranks must end with the unsharded
selection and, within rounding, the unsharded attention output.
"""
import os
import socket
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K = 64


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    from workloads import Workload, make_inputs
    wl = Workload("shard_cpu", 2, (1400, 900), 4, seed=77, topk=K, value_std=1.0 / 22.6)
    return wl, make_inputs(wl, "cpu", with_compress=False)


def _shard_rows_by_index(inp, n_seq, lo, hi):
    """The shard's rows and offsets from an explicit row list (the slow,
    obvious form that sharded.shard_inputs is checked against)."""
    poff = inp["pool_off"].tolist()
    rows, off = [], [0]
    for b in range(n_seq):
        a, e = poff[b] + lo, min(poff[b + 1], poff[b] + hi)
        rows.extend(range(a, max(a, e)))
        off.append(len(rows))
    return torch.tensor(rows, dtype=torch.long), off


def test_shard_inputs_slices_every_sequence():
    """sharded.shard_inputs on CPU tensors: for G = 2, 3, 4 and 7 shards each
    shard's pool rows, index keys and offsets equal the explicit row list's,
    only the window shard carries the window, and a shard past every
    sequence's end keeps one row so that its arrays stay addressable."""
    from compressed_sparse_attention_gb300 import sharded
    wl, inp = _case()
    for world in (2, 3, 4, 7, 36):
        n_rows = 0
        for rank in range(world):
            s = sharded.shard_inputs(inp, wl.n_seq, world, rank)
            sel, off = _shard_rows_by_index(inp, wl.n_seq, s.lo, s.hi)
            assert s.pool_off.tolist() == off
            if sel.numel():
                assert torch.equal(s.pool_kv, inp["pool_kv"][sel]) and torch.equal(s.idx_keys, inp["idx_keys"][sel])
            else:
                assert s.pool_kv.shape[0] == 1 and off[-1] == 0
            assert s.with_window == (rank == 0) and (s.win_kv is not None) == (rank == 0)
            n_rows += sel.numel()
        assert n_rows == int(inp["pool_off"][-1])


def _ops():
    from oracle import csa2_oracle as O
    g = O.Geometry(topk=K)
    f = O.yarn_inv_freq(64, g.rope_theta, g.yarn_factor, g.yarn_orig_len, g.yarn_beta_fast, g.yarn_beta_slow)
    from sharded_oracle_ops import OracleOps
    return OracleOps(g, f), g, f


def _rank(rank, world, port, queue):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from compressed_sparse_attention_gb300 import sharded
    dist.init_process_group("gloo")
    wl, inp = _case()
    ops, _, _ = _ops()
    out, lse, sel = sharded.run_distributed(sharded.shard_step(ops, sharded.shard_inputs(inp, wl.n_seq, world, rank), K))
    queue.put((rank, out.view(torch.int16).numpy(), lse.numpy(), sel.numpy()))
    dist.destroy_process_group()


def test_two_gloo_ranks_give_the_unsharded_selection_and_output():
    mp = torch.multiprocessing.get_context("spawn")
    q = mp.Queue()
    port = _free_port()
    procs = [mp.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks hold the same result
    assert np.array_equal(res[0][1], res[1][1]) and np.array_equal(res[0][3], res[1][3])
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from oracle import csa2_oracle as O
    from oracle import formats as F
    wl, inp = _case()
    _, g, f = _ops()
    keys = F.bf16_bits_to_f64(inp["idx_keys"].view(torch.int16).numpy().view(np.uint16))
    pool = F.bf16_bits_to_f64(inp["pool_kv"].view(torch.int16).numpy().view(np.uint16))
    win = F.bf16_bits_to_f64(inp["win_kv"].view(torch.int16).numpy().view(np.uint16))
    poff, woff = inp["pool_off"].tolist(), inp["win_off"].tolist()
    out = F.bf16_bits_to_f64(res[0][1].view(np.uint16))
    for qi in range(wl.n_query):
        b, t, nv = int(inp["seq_of_q"][qi]), int(inp["q_pos"][qi]), int(inp["n_vis"][qi])
        qv = F.bf16_bits_to_f64(inp["q"][qi].view(torch.int16).numpy().view(np.uint16))
        qidx = F.bf16_bits_to_f64(inp["q_idx"][qi].view(torch.int16).numpy().view(np.uint16))
        # scores rounded to fp32, as the ranks exchange them
        sc = O.index_scores(qidx, inp["w_heads"][qi].double().numpy(), keys[poff[b]:poff[b] + nv])
        sel = O.topk_select(sc.astype(np.float32).astype(np.float64), K)
        assert np.array_equal(res[0][3][qi], sel), f"query {qi}: sharded selection differs"
        cap = woff[b + 1] - woff[b]
        rows = O.gather_rows(t, g, lambda p: win[woff[b] + p % cap], pool[poff[b]:poff[b + 1]], sel)
        ref, ref_lse = O.attend(qv, t, rows, inp["sink"].double().numpy(), g.softmax_scale, f)
        assert np.abs(out[qi] - ref).max() <= 2.0 ** -8 * np.abs(ref).max() + 1e-6
        assert np.allclose(res[0][2][qi], ref_lse, rtol=1e-6, atol=1e-5)
