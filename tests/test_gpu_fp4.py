"""The fp4 storage formats on the GPU against the oracle's.

* csa2_store_rows with CSA2_KV_FP4_E4M3_B16 / CSA2_KV_MXFP4_B32: codes and
  scales bit-exact when both sides quantise identical fp32 values (blocks of
  zeros, of subnormal-scale values, of exact grid midpoints, random rows);
* the index scan over MXFP4 keys and attention over fp4 pool rows (with an
  fp8 window), each against the oracle run on the oracle's own dequantised
  rows of the same fp32 values.
"""
import numpy as np
import pytest
import torch

from gpu_common import (assert_attention_close, assert_rows_close_stored, attention_bound, bf16_np, context, f32_np,
                        geometry, inv_freq, oracle_fp8_rows, require_gpu, score_tolerance)
from oracle import csa2_oracle as O
from oracle import formats as F
from workloads import Workload, make_inputs, make_selection

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rows(n, dim, seed):
    """fp32 rows with the hard cases planted: a zero block, a block far below
    the scale floor, a block of exact e2m1 midpoints, wide magnitudes."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((n, dim), generator=g) * torch.exp(torch.empty((n, 1)).uniform_(-5, 4, generator=g))
    x[0, :32] = 0.0
    x[1, :32] = torch.randn(32, generator=g) * 1e-9
    # amax 6 in the first 16-channel block -> scale 1 (fp4) / 2^0 (mxfp4): exact ties
    x[2, :16] = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -5.0, 0.0, 4.0, -6.0, 3.0, 1.0])
    x[2, 16:32] = torch.tensor([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] * 2)
    x[3, :] = -0.0
    return x.float()


@pytest.mark.parametrize("dim", [512, 128])
@pytest.mark.parametrize("fmt", ["fp4", "mxfp4"])
def test_store_rows_fp4_bit_exact(dim, fmt):
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context()
    x = _rows(257, dim, seed=dim + (1 if fmt == "fp4" else 2))
    block = 16 if fmt == "fp4" else 32
    out = torch.full((x.shape[0], dim // 2), 0xAA, dtype=torch.uint8, device=DEV)
    sc = torch.full((x.shape[0], dim // block), 0xAA, dtype=torch.uint8, device=DEV)
    code = binding.KV_FP4 if fmt == "fp4" else binding.KV_MXFP4
    ctx.store_rows(x.to(DEV), None, code, out, sc)
    torch.cuda.synchronize()
    xn = x.double().numpy()
    if fmt == "fp4":
        codes, sref = F.fp4_block_quantize(xn)
    else:
        codes, sref = F.mxfp4_block_quantize(xn)
    assert np.array_equal(sc.cpu().numpy(), sref), "scales differ"
    assert np.array_equal(out.cpu().numpy(), F.pack_e2m1(codes)), "codes differ"


@pytest.mark.parametrize("fmt", ["fp4", "mxfp4"])
def test_store_rows_fp4_rotated(fmt):
    """With RoPE the GPU rotates in fp32 and the oracle in float64, so a value
    at a grid midpoint may go either way: stored rows within the e2m1 bound of
    the exact rotated values, scales within one code of the oracle's."""
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context()
    f = inv_freq(geometry(ctx.cfg))
    x = _rows(64, 512, seed=9)
    pos = torch.arange(64, dtype=torch.int64) * 977 + 5
    code = binding.KV_FP4 if fmt == "fp4" else binding.KV_MXFP4
    out = torch.empty((64, 256), dtype=torch.uint8, device=DEV)
    sc = torch.empty((64, 512 // (16 if fmt == "fp4" else 32)), dtype=torch.uint8, device=DEV)
    ctx.store_rows(x.to(DEV), pos.to(DEV), code, out, sc)
    torch.cuda.synchronize()
    exact = O.rope_rotate(x.double().numpy(), pos.numpy(), f)
    assert_rows_close_stored(out, sc, exact, code, f"rope store {fmt}")


@pytest.mark.parametrize("idx_heads", [8, 16, 32])
def test_index_score_mxfp4_keys(idx_heads):
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context(idx_heads=idx_heads, idx_key_format=binding.KV_MXFP4)
    wl = Workload("idx_fp4", 3, (4000, 148, 10404), 4, seed=51 + idx_heads, idx_heads=idx_heads, idx_fp8=True,
                  n_query_per_seq=2)
    inp = make_inputs(wl, DEV, with_compress=False)
    Q = wl.n_query
    nv = inp["n_vis"].clone()
    nv[1] = 7
    nv[2] = 0
    max_vis = int(nv.max())
    kf = inp["idx_keys_f32"]
    keys = torch.empty((kf.shape[0], 64), dtype=torch.uint8, device=DEV)
    ksc = torch.empty((kf.shape[0], 4), dtype=torch.uint8, device=DEV)
    ctx.store_rows(kf, None, binding.KV_MXFP4, keys, ksc)
    keys_np = F.mxfp4_block_dequantize(*F.mxfp4_block_quantize(f32_np(kf)))
    scores = torch.full((Q, max_vis + 3), float("nan"), device=DEV)
    ctx.index_score(wl.n_seq, inp["q_idx"], inp["w_heads"], keys, ksc, inp["pool_off"], inp["seq_of_q"], nv,
                    max_vis, scores)
    assert ctx.check()[0] == 0
    s = f32_np(scores)
    poff = inp["pool_off"].cpu().numpy()
    for qi in range(Q):
        b, n = int(inp["seq_of_q"][qi]), int(nv[qi])
        qv, w = bf16_np(inp["q_idx"][qi]), f32_np(inp["w_heads"][qi])
        kk = keys_np[poff[b]:poff[b] + n]
        ref = O.index_scores(qv, w, kk)
        assert np.all(np.abs(s[qi, :n] - ref) <= score_tolerance(ref, qv, w, kk)), f"query {qi}"
        assert np.all(np.isnan(s[qi, n:]))


@pytest.mark.parametrize("n_seq,ctx_len", [(3, (3000, 9000, 700)), (40, None)])
def test_attend_fp4_pool_fp8_window(n_seq, ctx_len):
    """Plain attend (one launch + merge, or the shared launch) over fp4 pool
    rows and an fp8 window, against the oracle on its own dequantised rows."""
    from compressed_sparse_attention_gb300 import binding
    require_gpu()
    ctx = context(kv_format=binding.KV_FP4)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    lens = ctx_len or tuple(2000 + 97 * i for i in range(n_seq))
    wl = Workload("att_fp4", n_seq, lens, 4, seed=61 + n_seq, kv_fp8=True, outlier_frac=0.01)
    inp = make_inputs(wl, DEV, with_compress=False)
    Q = wl.n_query
    win = inp["win_kv_f32"]
    win_codes = torch.empty(win.shape, dtype=torch.uint8, device=DEV)
    win_sc = torch.empty((win.shape[0], 16), dtype=torch.uint8, device=DEV)
    ctx.store_rows(win, None, binding.KV_FP8, win_codes, win_sc)
    pool = inp["pool_kv_f32"]
    pool_codes = torch.empty((pool.shape[0], 256), dtype=torch.uint8, device=DEV)
    pool_sc = torch.empty((pool.shape[0], 32), dtype=torch.uint8, device=DEV)
    ctx.store_rows(pool, None, binding.KV_FP4, pool_codes, pool_sc)
    sel = make_selection(wl, inp["n_vis"], 7 + n_seq, DEV)
    out = torch.empty((Q, 64, 512), dtype=torch.bfloat16, device=DEV)
    ws = binding.workspace(ctx.attend_workspace_size(Q), DEV)
    ctx.attend(wl.n_seq, inp["q"], inp["q_pos"], inp["seq_of_q"], win_codes, win_sc, inp["win_off"], None,
               pool_codes, pool_sc, inp["pool_off"], sel, inp["sink"], out, None, ws)
    assert ctx.check()[0] == 0
    win_np = oracle_fp8_rows(f32_np(win))[2]
    woff = inp["win_off"].cpu().numpy()
    poff = inp["pool_off"].cpu().numpy()
    sel_np = sel.cpu().numpy()
    pool_np = f32_np(pool)
    for qi in (range(Q) if Q <= 4 else (0, 7, Q - 1)):
        b = int(inp["seq_of_q"][qi])
        t = int(inp["q_pos"][qi])
        cap = int(woff[b + 1] - woff[b])
        chosen = sel_np[qi][sel_np[qi] >= 0]
        prow = F.fp4_block_dequantize(*F.fp4_block_quantize(pool_np[poff[b] + chosen]))
        rows = O.gather_rows(t, geom, lambda p_: win_np[woff[b] + p_ % cap], prow, np.arange(chosen.shape[0]))
        q = bf16_np(inp["q"][qi])
        sink = f32_np(inp["sink"])
        ref, _ = O.attend(q, t, rows, sink, geom.softmax_scale, f)
        bnd = attention_bound(q, t, rows, sink, geom.softmax_scale, f)
        assert_attention_close(bf16_np(out[qi]), ref, bnd, f"q{qi}")


@pytest.mark.parametrize("n_seq", [3, 40])
def test_step_full_fp4(n_seq):
    """A Full decode step with fp4 pool rows, an fp8 window and mxfp4 keys:
    the entries compressed at this step, scores, selection and attention."""
    from compressed_sparse_attention_gb300 import binding
    from test_gpu_fullsize import Case, _check_query, _full_state, _step
    require_gpu()
    g = torch.Generator().manual_seed(700 + n_seq)
    lens = tuple(int(x) for x in torch.randint(2600, 9000, (n_seq,), generator=g))
    wl = Workload(f"step_fp4_{n_seq}", n_seq, lens, 4, seed=700 + n_seq, value_std=1.0 / 22.6, outlier_frac=0.01,
                  kv_fp8=True, idx_fp8=True, pool_fp4=True, key_fp4=True)
    ctx = context(kv_format=wl.kv_format, idx_key_format=wl.idx_key_format)
    geom = geometry(ctx.cfg)
    f = inv_freq(geom)
    case = Case(ctx, wl)
    idx = torch.empty((wl.n_query, wl.topk), dtype=torch.int32, device=DEV)
    out, scores = _step(ctx, case, binding.MODE_FULL, idx)
    sel = idx.cpu().numpy()
    state = _full_state(ctx, case, geom, f)
    sample = range(wl.n_query) if wl.n_query <= 8 else sorted({0, 1, wl.n_query // 2, wl.n_query - 1})
    same = [_check_query(ctx, case, qi, geom, f, out, scores, sel, state, wl.name)[1] for qi in sample]
    assert sum(same) >= len(same) - 1
