"""The decode forms of the CSA2 step at small sizes, against the oracle.

With few queries the step runs the window tile beside top-k and spreads the
selected tiles over several CTAs per query, whose partials a merge kernel
combines; how many CTAs, and how many tiles each takes, depends on the number
of queries and on k. With more queries the window and the selected tiles
share one launch. These cases pick batch sizes and k so that each form is
taken (one selected tile for k = 128, five for k = 640, one to four CTAs per
query, the shared launch for 90 queries). Every query of a small batch, and a
sample of a large one, is checked: scores, selection, and the step's
attention output whenever the selection equals the oracle's.
"""
import pytest
import torch

from gpu_common import context, geometry, inv_freq, require_gpu
from test_gpu_fullsize import Case, _check_query, _full_state, _step
from workloads import Workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("n_seq,topk", [(1, 512), (3, 128), (5, 640), (40, 512), (70, 512), (90, 512)])
def test_step_decode_forms(n_seq, topk):
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    g = torch.Generator().manual_seed(900 + n_seq)
    lens = tuple(int(x) for x in torch.randint(2600, 9000, (n_seq,), generator=g))
    wl = Workload(f"forms_{n_seq}_{topk}", n_seq, lens, 4, seed=900 + n_seq + topk, topk=topk,
                  value_std=1.0 / 22.6, outlier_frac=0.01)
    ctx = context(topk=topk)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    case = Case(ctx, wl)
    idx = torch.empty((wl.n_query, topk), dtype=torch.int32, device=DEV)
    out, scores = _step(ctx, case, binding.MODE_FULL, idx)
    sel = idx.cpu().numpy()
    state = _full_state(ctx, case, geom, f)
    sample = range(wl.n_query) if wl.n_query <= 8 else sorted({0, 1, wl.n_query // 2, wl.n_query - 1})
    same = [_check_query(ctx, case, qi, geom, f, out, scores, sel, state, wl.name)[1] for qi in sample]
    assert sum(same) >= len(same) - 1, "the step's selection differs from the oracle's on more than one query"


@pytest.mark.parametrize("m", [1, 2])
def test_step_two_queries_per_sequence(m):
    """Two decode queries per sequence at t = N-2 and N-1 with compress ratio
    m: the step closes up to two groups per sequence, and the query at N-2
    sees only the entries that close by its own position. These entries are
    scored apart from the scan over the older ones while compress runs."""
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    n_seq = 6
    g = torch.Generator().manual_seed(950 + m)
    lens = tuple(int(x) * m for x in torch.randint(1500, 4000, (n_seq,), generator=g))
    wl = Workload(f"two_q_m{m}", n_seq, lens, m, seed=950 + m, n_query_per_seq=2, value_std=1.0 / 22.6,
                  outlier_frac=0.01)
    ctx = context(compress_ratio=m)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    case = Case(ctx, wl)
    idx = torch.empty((wl.n_query, wl.topk), dtype=torch.int32, device=DEV)
    out, scores = _step(ctx, case, binding.MODE_FULL, idx)
    sel = idx.cpu().numpy()
    state = _full_state(ctx, case, geom, f)
    same = [_check_query(ctx, case, qi, geom, f, out, scores, sel, state, wl.name)[1] for qi in range(wl.n_query)]
    assert sum(same) >= len(same) - 1


@pytest.mark.parametrize("mode", ["full", "reindex", "reuse"])
def test_step_host_equals_step(mode):
    """csa2_step_host gives the bits csa2_step gives. Pinned host buffers:
    q staged by a kernel on the copy stream beside the scan, the raw tokens and
    gates read in place by compress, the output written straight into host
    memory by the step's last launch. Pageable host buffers: copy-engine copies
    through the staging buffers. Also captured into a graph and replayed."""
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    code = {"full": binding.MODE_FULL, "reindex": binding.MODE_REINDEX, "reuse": binding.MODE_REUSE}[mode]
    wl = Workload("host_io", 5, (4100, 9000, 3003, 2600, 7777), 4, seed=960, value_std=1.0 / 22.6)
    ctx = context()
    case = Case(ctx, wl)
    i = case.inp
    Q = wl.n_query
    max_vis = int(i["n_vis"].max())
    idx = torch.empty((Q, 512), dtype=torch.int32, device=DEV)
    out_dev = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = binding.workspace(ctx.step_workspace_size(Q, max_vis), DEV)
    common = dict(q_pos=i["q_pos"], seq_of_q=i["seq_of_q"], n_vis=i["n_vis"], sink=i["sink"], win_kv=i["win_kv"],
                  win_off=i["win_off"], pool_kv=i["pool_kv"], pool_off=i["pool_off"], topk_idx=idx, workspace=ws,
                  q_idx=i["q_idx"], w_heads=i["w_heads"], idx_keys=i["idx_keys"], tok_off=i["tok_off"],
                  first_pos=i["first_pos"], norm_w=i["norm_w"], w_idx=i["w_idx"], k_norm_w=i["k_norm_w"])
    # a Full step first: it fills the pool and the selection Reuse reads
    ctx.step(binding.MODE_FULL, wl.n_seq, max_vis, q=i["q"], raw=i["raw"], gate=i["gate"], out=out_dev, **common)
    if code != binding.MODE_FULL:
        ctx.step(code, wl.n_seq, max_vis, q=i["q"], raw=i["raw"], gate=i["gate"], out=out_dev, **common)
    torch.cuda.synchronize()
    ref = out_dev.cpu()
    sel = idx.clone()
    sq, sraw, sgate = torch.zeros_like(i["q"]), torch.zeros_like(i["raw"]), torch.zeros_like(i["gate"])
    sout = torch.zeros_like(out_dev)
    prep = ctx.prepare_step(code, wl.n_seq, max_vis, q=sq, raw=sraw, gate=sgate, out=sout, **common)
    hq, hraw, hgate = (t.cpu().pin_memory() for t in (i["q"], i["raw"], i["gate"]))
    hout = torch.empty(out_dev.shape, dtype=out_dev.dtype).pin_memory()
    prep.run_host(q=hq, raw=hraw, gate=hgate, out=hout)
    torch.cuda.synchronize()
    assert ctx.check() == (0, 0)
    assert torch.equal(hout, ref)
    assert torch.equal(idx, sel)
    assert torch.equal(sq, i["q"]), "q is staged into the device buffer"
    assert float(sraw.float().abs().sum()) == 0.0 and float(sgate.abs().sum()) == 0.0, \
        "pinned raw tokens and gates are read in place, not staged"
    assert float(sout.float().abs().sum()) == 0.0, "a pinned output is written directly, not staged"
    # pageable host buffers: copy-engine copies through the staging buffers
    pq, praw, pgate = (t.cpu().clone() for t in (i["q"], i["raw"], i["gate"]))
    sq.zero_()
    hpage = torch.zeros(out_dev.shape, dtype=out_dev.dtype)
    prep.run_host(q=pq, raw=praw, gate=pgate, out=hpage)
    torch.cuda.synchronize()
    assert ctx.check() == (0, 0)
    assert torch.equal(hpage, ref) and torch.equal(sout.cpu(), ref) and torch.equal(idx, sel)
    assert torch.equal(sq, i["q"]) and torch.equal(sraw, i["raw"]) and torch.equal(sgate, i["gate"])
    # the same step captured with its copies and replayed
    hout2 = torch.zeros_like(hout).pin_memory()
    graph = prep.host_graph(q=hq, raw=hraw, gate=hgate, out=hout2)
    for _ in range(2):
        graph.launch()
    torch.cuda.synchronize()
    assert ctx.check() == (0, 0)
    assert torch.equal(hout2, ref)
