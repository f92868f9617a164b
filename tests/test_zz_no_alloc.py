"""csa2_attend_noalloc: the attention entry point for callers that cannot
allocate device memory (a host that owns all device memory through its own
pool, or a loop that must not trigger the allocator's implicit
synchronisation). It keeps its split-K scratch in a library-owned device array
instead of a caller workspace. It runs the same plan and the same kernels as
csa2_attend, only with the scratch at another address, so its output and lse
must equal csa2_attend's bit for bit on the same inputs, call after call (the
array keeps the previous call's contents).

This file is collected last so that a run stopping at the first failure has
already run every other test; it builds its own context and inputs, so it
passes alone in a fresh process as well as after the rest of the suite.
"""
import ctypes as C

import pytest
import torch

from gpu_common import require_gpu
from workloads import Workload, make_inputs, make_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _noalloc(ctx, n_seq, inp, sel, out, lse):
    lib = ctx.lib
    st = lib.csa2_attend_noalloc(ctx.h, C.c_void_p(torch.cuda.current_stream().cuda_stream), n_seq,
                                 inp["q"].shape[0], _ptr(inp["q"]), _ptr(inp["q_pos"]), _ptr(inp["seq_of_q"]),
                                 _ptr(inp["win_kv"]), None, _ptr(inp["win_off"]), None, _ptr(inp["pool_kv"]), None,
                                 _ptr(inp["pool_off"]), _ptr(sel), _ptr(inp["sink"]), _ptr(out), _ptr(lse))
    return st


def _same(a: torch.Tensor, b: torch.Tensor):
    return torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                       b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


def test_attend_noalloc_matches_attend_twice_in_a_row():
    require_gpu()
    from compressed_sparse_attention_gb300 import binding, build
    build.build()
    ctx = binding.Context()
    for call, seed in enumerate((101, 202)):
        # a few decode queries with several 128-row tiles each, so the split-K
        # scratch is used; the second call's inputs differ from the first's
        wl = Workload(f"noalloc_{call}", 6, (3000, 4100, 700, 9000, 2051, 5000), 4, seed=seed,
                      value_std=1.0 / 22.6)
        inp = make_inputs(wl, DEV, with_compress=False)
        sel = make_selection(wl, inp["n_vis"], seed, DEV)
        Q = wl.n_query
        assert ctx.attend_workspace_size(Q) > 0, "the case must exercise the scratch"
        ref = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
        ref_lse = torch.empty((Q, 64), dtype=torch.float32, device=DEV)
        ws = binding.workspace(ctx.attend_workspace_size(Q), DEV)
        ctx.attend(wl.n_seq, inp["q"], inp["q_pos"], inp["seq_of_q"], inp["win_kv"], None, inp["win_off"], None,
                   inp["pool_kv"], None, inp["pool_off"], sel, inp["sink"], ref, ref_lse, ws)
        out = torch.full((Q, 64, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((Q, 64), float("nan"), dtype=torch.float32, device=DEV)
        assert _noalloc(ctx, wl.n_seq, inp, sel, out, lse) == 0, ctx.lib.csa2_last_error(ctx.h).decode()
        flags, st = ctx.check()
        assert flags == 0 and st == 0
        assert _same(out, ref), f"call {call}: output differs from csa2_attend"
        assert _same(lse, ref_lse), f"call {call}: lse differs from csa2_attend"


def test_attend_noalloc_scratch_bound():
    """The fixed scratch either covers every query count's split-K partials
    (then the entry point runs at the count that needs the most, and matches
    csa2_attend there), or a count beyond it is rejected before anything is
    enqueued. Which case holds depends on the SM count: with bf16 partials a
    152-SM GPU needs at most ~20 MB."""
    require_gpu()
    from compressed_sparse_attention_gb300 import binding, build
    build.build()
    ctx = binding.Context()
    limit = 32 << 20
    need = {n: ctx.attend_workspace_size(n) for n in range(1, 4096)}
    n_big = next((n for n, b in need.items() if b > limit), None)
    if n_big is None:
        n_max = max(need, key=need.get)
        wl = Workload("noalloc_max", 1, (4096,), 4, seed=4, n_query_per_seq=n_max)
        inp = make_inputs(wl, DEV, with_compress=False)
        sel = make_selection(wl, inp["n_vis"], 4, DEV)
        ref = torch.empty((n_max, 64, 512), dtype=torch.bfloat16, device=DEV)
        ws = binding.workspace(need[n_max], DEV)
        ctx.attend(1, inp["q"], inp["q_pos"], inp["seq_of_q"], inp["win_kv"], None, inp["win_off"], None,
                   inp["pool_kv"], None, inp["pool_off"], sel, inp["sink"], ref, None, ws)
        out = torch.full((n_max, 64, 512), float("nan"), dtype=torch.bfloat16, device=DEV)
        assert _noalloc(ctx, 1, inp, sel, out, None) == 0, ctx.lib.csa2_last_error(ctx.h).decode()
        flags, st = ctx.check()
        assert flags == 0 and st == 0
        assert _same(out, ref)
        return
    wl = Workload("noalloc_big", 1, (4096,), 4, seed=3, n_query_per_seq=n_big)
    inp = make_inputs(wl, DEV, with_compress=False)
    sel = make_selection(wl, inp["n_vis"], 3, DEV)
    out = torch.zeros((n_big, 64, 512), dtype=torch.bfloat16, device=DEV)
    st = _noalloc(ctx, 1, inp, sel, out, None)
    assert st == 6, f"expected CSA2_ERR_WORKSPACE, got {st}"
    msg = ctx.lib.csa2_last_error(ctx.h).decode()
    assert "scratch" in msg and str(limit) in msg
    assert float(out.float().abs().sum()) == 0.0  # nothing was enqueued
