"""How a context behaves around its calls, on the GPU.

* A bounded device wait that runs out: the wait probe waits, with the
  attention kernels' own bounded mbarrier wait, on a barrier that nothing
  arrives at. The wait must give up after its limit, csa2_check must report
  CSA2_ERR_TIMEOUT with the timeout bit, and the context must stay usable
  (the next step on it runs clean and gives the same output as before).
* Two contexts used at once on two streams: each context owns its scan
  counters, side stream and events, so two steps enqueued on two streams
  with no ordering between them give the bits each gives alone.
"""
import pytest
import torch

from gpu_common import context, require_gpu
from test_gpu_fullsize import Case, _step
from workloads import Workload

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _small_case(ctx, seed):
    wl = Workload(f"ctx_use_{seed}", 4, (3100, 5000, 2600, 7000), 4, seed=seed, value_std=1.0 / 22.6,
                  outlier_frac=0.01)
    return Case(ctx, wl)


def test_wait_timeout_is_reported_and_the_context_stays_usable():
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    ctx = context()
    case = _small_case(ctx, 1201)
    idx = torch.empty((case.wl.n_query, case.wl.topk), dtype=torch.int32, device=DEV)
    out0, _ = _step(ctx, case, binding.MODE_FULL, idx)
    out0 = out0.clone()
    with pytest.raises(binding.Csa2Error):
        ctx.debug_wait_timeout(0)  # outside 1 .. 1e9: rejected on the host, nothing enqueued
    ctx.debug_wait_timeout(1_000_000)  # 1 ms
    flags, st = ctx.check()
    assert st == 5, f"expected CSA2_ERR_TIMEOUT, got status {st}"
    assert flags & binding.FLAG_WAIT_TIMEOUT
    # the word was cleared by csa2_check and the context still works
    assert ctx.check() == (0, 0)
    case2 = _small_case(ctx, 1201)  # the same inputs again (Full mode rewrites the entries it compresses)
    out1, _ = _step(ctx, case2, binding.MODE_FULL, idx)
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))


def test_two_contexts_on_two_streams_at_once():
    require_gpu()
    from compressed_sparse_attention_gb300 import binding
    ctx_a = binding.Context()
    ctx_b = binding.Context()
    ca, cb = _small_case(ctx_a, 1301), _small_case(ctx_b, 1302)
    idx_a = torch.empty((ca.wl.n_query, ca.wl.topk), dtype=torch.int32, device=DEV)
    idx_b = torch.empty_like(idx_a)
    # alone, one after the other
    ref_a, _ = _step(ctx_a, ca, binding.MODE_REINDEX, idx_a)
    ref_b, _ = _step(ctx_b, cb, binding.MODE_REINDEX, idx_b)
    ref_a, ref_b = ref_a.clone(), ref_b.clone()
    sel_a, sel_b = idx_a.clone(), idx_b.clone()
    # at once: each context on its own stream, several times in a row
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    for _ in range(4):
        oa = torch.empty_like(ref_a)
        ob = torch.empty_like(ref_b)
        wa = binding.workspace(ctx_a.step_workspace_size(ca.wl.n_query, int(ca.inp["n_vis"].max())), DEV)
        wb = binding.workspace(ctx_b.step_workspace_size(cb.wl.n_query, int(cb.inp["n_vis"].max())), DEV)
        ia, ib = torch.empty_like(idx_a), torch.empty_like(idx_b)
        torch.cuda.synchronize()
        for ctx, case, st, o, w, i in ((ctx_a, ca, sa, oa, wa, ia), (ctx_b, cb, sb, ob, wb, ib)):
            inp = case.inp
            with torch.cuda.stream(st):
                ctx.step(binding.MODE_REINDEX, case.wl.n_seq, int(inp["n_vis"].max()), q=inp["q"],
                         q_pos=inp["q_pos"], seq_of_q=inp["seq_of_q"], n_vis=inp["n_vis"], sink=inp["sink"],
                         win_kv=inp["win_kv"], win_off=inp["win_off"], pool_kv=inp["pool_kv"],
                         pool_off=inp["pool_off"], topk_idx=i, out=o, workspace=w, q_idx=inp["q_idx"],
                         w_heads=inp["w_heads"], idx_keys=inp["idx_keys"])
        torch.cuda.synchronize()
        outs.append((oa, ob, ia, ib))
    for ctx, st in ((ctx_a, sa), (ctx_b, sb)):
        with torch.cuda.stream(st):
            assert ctx.check() == (0, 0)
    for oa, ob, ia, ib in outs:
        assert torch.equal(ia, sel_a) and torch.equal(ib, sel_b)
        assert torch.equal(oa.view(torch.int16), ref_a.view(torch.int16))
        assert torch.equal(ob.view(torch.int16), ref_b.view(torch.int16))
