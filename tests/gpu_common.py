"""Helpers shared by the GPU parity tests: context setup, conversions of the
device tensors to float64 for the oracle, and the tolerances.

Tolerances:
  attention : per element |gpu - oracle| <= 2e-2 + u (D + B + |oracle|) + S,
              and ||gpu - oracle|| / ||oracle|| <= 1e-2 per query, where
              u = 2^-8 is bf16's unit roundoff, B = sum_r p_r |v_r| (the size
              of the weighted sum before cancellation), D = sum_r p_r |v_r - o|
              (its spread about the output) and S the fp32 score term; each
              term is derived in attention_bound below
  lse       : |gpu - oracle| <= u + max_r delta_r per head (lse_bound)
  scores    : |gpu - oracle| <= 1e-3 |oracle| + 1e-5 * sum_h |w_h| ||q_h|| ||k||
              (relative 1e-3, plus the fp32 accumulation bound of a 128-term dot)
  top-k     : bit-exact on identical fp32 scores
  stored rows (bf16): |gpu - oracle| <= 1 bf16 ulp of the oracle value + 1e-5 * row rms
  stored rows (fp4/mxfp4, from values the GPU computes in fp32): per block of
              scale s, |stored - exact| <= s + max(0, amax - 6 s) (half the
              widest e2m1 gap, or the saturation), the scale byte within one
              code of the oracle's

Every attention comparison also records its raw max-abs error and rel-L2
against the stated flat bars (2e-2, 1e-2) in PARITY_LOG; the test session
prints them per test at the end (tests/conftest.py).
"""
from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O
from oracle import formats as F

ATT_MAX_ABS = 2e-2          # the stated flat bar for unit-scale outputs
ATT_REL_L2 = 1e-2           # the stated relative-L2 bar, per query
BF16_U = 2.0 ** -8          # bf16 unit roundoff: 8 significant bits, round to nearest
ATT_MMA_STEPS = 40          # fp32 roundings of one score: 36 MMA K-steps of 16 (32 + 4 rope hi/lo) + margin
ATT_WEIGHT_FIX = 2.0 ** -21  # per weight: the log2(e) scaling, the max subtraction and exp2f (2 ulp)

# (test id, what, max-abs, rel-L2, worst |err| / limit, elements above the flat 2e-2, elements)
PARITY_LOG = []
SCORE_REL = 1e-3
SCORE_ABS_FRAC = 1e-5


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


_CTX_CACHE = {}


def context(**overrides):
    from compressed_sparse_attention_gb300 import binding, build
    build.build()
    key = tuple(sorted(overrides.items()))
    if key not in _CTX_CACHE:
        _CTX_CACHE[key] = binding.Context(**overrides)
    return _CTX_CACHE[key]


def geometry(cfg) -> O.Geometry:
    return O.Geometry(n_heads=cfg.n_heads, head_dim=cfg.head_dim, rope_dim=cfg.rope_dim, window=cfg.window,
                      compress_ratio=cfg.compress_ratio, idx_heads=cfg.idx_heads, idx_dim=cfg.idx_dim,
                      topk=cfg.topk, softmax_scale=float(cfg.softmax_scale), norm_eps=float(cfg.norm_eps),
                      rope_theta=cfg.rope_theta, yarn_factor=cfg.yarn_factor, yarn_orig_len=cfg.yarn_orig_len,
                      yarn_beta_fast=cfg.yarn_beta_fast, yarn_beta_slow=cfg.yarn_beta_slow)


def inv_freq(geom: O.Geometry) -> np.ndarray:
    if geom.rope_dim == 0:
        return np.zeros(0)
    return O.yarn_inv_freq(geom.rope_dim, geom.rope_theta, geom.yarn_factor, geom.yarn_orig_len,
                           geom.yarn_beta_fast, geom.yarn_beta_slow)


def bf16_np(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a bf16 tensor."""
    u = t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
    return F.bf16_bits_to_f64(u)


def f32_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().double().numpy()


def oracle_fp8_rows(x_f32: np.ndarray):
    """The oracle's own fp8 block-32 quantisation of fp32 rows: (codes, exps, values)."""
    codes, exps = F.fp8_block_quantize(x_f32)
    return codes, exps, F.fp8_block_dequantize(codes, exps)


# storage format codes of the library (kv_format / idx_key_format)
FMT_BF16, FMT_FP8, FMT_FP4, FMT_MXFP4 = 0, 1, 2, 3
SCALE_BLOCK = {FMT_FP8: 32, FMT_FP4: 16, FMT_MXFP4: 32}


def code_bytes(dim: int, fmt: int) -> int:
    """Bytes of one stored row's codes (scales excluded)."""
    return {FMT_BF16: 2 * dim, FMT_FP8: dim, FMT_FP4: dim // 2, FMT_MXFP4: dim // 2}[fmt]


def stored_values(codes, scale, fmt: int) -> np.ndarray:
    """Exact values of rows stored in format `fmt`, decoded by the oracle."""
    if fmt == FMT_BF16:
        return bf16_np(codes)
    c = codes.cpu().numpy() if isinstance(codes, torch.Tensor) else codes
    sc = scale.cpu().numpy() if isinstance(scale, torch.Tensor) else scale
    if fmt == FMT_FP8:
        return F.fp8_block_dequantize(c, sc)
    if fmt == FMT_FP4:
        return F.fp4_block_dequantize(F.unpack_e2m1(c), sc)
    if fmt == FMT_MXFP4:
        return F.mxfp4_block_dequantize(F.unpack_e2m1(c), sc)
    raise ValueError(fmt)


def oracle_stored(x: np.ndarray, fmt: int) -> np.ndarray:
    """The oracle's own stored form of float64 rows: quantise, then decode."""
    if fmt == FMT_BF16:
        return F.round_bf16(x)
    if fmt == FMT_FP8:
        return F.fp8_block_dequantize(*F.fp8_block_quantize(x))
    if fmt == FMT_FP4:
        return F.fp4_block_dequantize(*F.fp4_block_quantize(x))
    if fmt == FMT_MXFP4:
        return F.mxfp4_block_dequantize(*F.mxfp4_block_quantize(x))
    raise ValueError(fmt)


def scale_values(scale, fmt: int) -> np.ndarray:
    sc = scale.cpu().numpy() if isinstance(scale, torch.Tensor) else np.asarray(scale)
    return F.e4m3_bits_to_f64(sc) if fmt == FMT_FP4 else F.ue8m0_to_f64(sc)


def storage_bound(exact: np.ndarray, scale, fmt: int) -> np.ndarray:
    """Per element bound on |stored - exact| for rows the GPU quantised from
    values it computed in fp32 (so either neighbour of a grid midpoint may be
    taken): one bf16 ulp; one e4m3 step (2^-3 relative, 2^-9 of the scale
    below the normal range); for e2m1 half the widest gap (2 s) plus what
    saturation at 6 s clips."""
    if fmt == FMT_BF16:
        rms = np.sqrt(np.mean(exact * exact, axis=-1, keepdims=True))
        return F.bf16_ulp(exact) + 1e-5 * rms
    blk = SCALE_BLOCK[fmt]
    s = scale_values(scale, fmt)
    if fmt == FMT_FP8:
        return 2.0 ** -3 * np.abs(exact) + 2.0 ** -9 * np.repeat(s, blk, axis=-1) + 1e-30
    amax = np.abs(exact).reshape(*exact.shape[:-1], -1, blk).max(axis=-1)
    per_block = s + np.maximum(0.0, amax * (1 + 1e-6) - 6.0 * s)
    return np.repeat(per_block, blk, axis=-1) + 1e-6 * np.abs(exact) + 1e-30


def assert_rows_close_stored(codes, scale, exact: np.ndarray, fmt: int, what: str = ""):
    """Rows the GPU stored against the float64 values they encode; for the
    scaled formats also the scale bytes against the oracle's (within one code)."""
    got = stored_values(codes, scale, fmt)
    bad = np.abs(got - exact) > storage_bound(exact, scale, fmt)
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, worst {float(np.abs(got - exact).max()):.3e}"
    if fmt in (FMT_FP4, FMT_MXFP4):
        ref_sc = (F.fp4_block_quantize(exact) if fmt == FMT_FP4 else F.mxfp4_block_quantize(exact))[1]
        d = np.abs(scale.cpu().numpy().astype(np.int32) - ref_sc.astype(np.int32))
        assert d.max(initial=0) <= 1, f"{what}: scale bytes differ by {int(d.max())} codes"


class AttBound:
    """The magnitudes the attention error bound is built from, per head and
    channel of one query: B = sum_r p_r |v_r|, D = sum_r p_r |v_r - o| and
    the fp32 score term S."""

    def __init__(self, sum_pv: np.ndarray, spread: np.ndarray, score: np.ndarray):
        self.sum_pv, self.spread, self.score = sum_pv, spread, score


def attention_bound(q, t, rows, sink, scale, f) -> AttBound:
    """Per-element error terms of one query's attention output.

    The GPU computes o = sum_r P_r v_r / (sum_r P_r + e^sink) with bf16 rows,
    fp32 scores, P rounded to bf16 and an fp32 sum. Against the float64
    oracle (w_r = p_r / den its exact weights, o its output, u = 2^-8 the
    bf16 unit roundoff):
      * P in bf16: each weight moves by at most u of itself, and the
        denominator sums the same rounded weights, so to first order o moves
        by sum_r w_r eps_r (v_r - o), at most u D with D = sum_r w_r |v_r - o|;
      * split-K partials stored in bf16: each partial moves by at most u of
        its own weighted sum, which the merge weights bring to u B in all,
        B = sum_r w_r |v_r|;
      * the output rounded to bf16: half an ulp, at most u |o|;
      * fp32 scores: s_r = tau q~ . v_r accumulated by the tensor core in
        fp32 over 36 K-steps, each rounding at most 2^-24 of a running sum no
        larger than tau sum_i |q~_i| |v_ri|; with the exp2 and scaling steps
        each weight's relative error is delta_r <= 40 * 2^-24 * tau *
        sum_i |q~_i||v_ri| + 2^-21, and o moves by at most
        S = sum_r w_r delta_r |v_r - o|.
    The two channels of a rope pair share the sum of their bounds, since the
    output's de-rotation mixes them.
    """
    p, _ = O.attention_weights(q, t, rows, sink, scale, f)
    rows = np.asarray(rows, dtype=np.float64).reshape(-1, np.asarray(q).shape[1])
    ar = np.abs(rows)
    bnd = p @ ar
    o = p @ rows  # [H, D], the output before the de-rotation (p already includes the sink's share)
    dev = np.abs(rows[None, :, :] - o[:, None, :])  # [H, R, D]: |v_r - o|
    spread = np.einsum("hr,hrd->hd", p, dev)
    qr = O.rope_rotate(np.asarray(q, dtype=np.float64), t, f)
    delta = ATT_MMA_STEPS * 2.0 ** -24 * abs(scale) * (np.abs(qr) @ ar.T) + ATT_WEIGHT_FIX  # [H, R]
    sc = np.einsum("hr,hrd->hd", p * delta, dev)
    del dev
    r = 2 * f.shape[0]
    if r:
        d = bnd.shape[-1]
        for x in (bnd, spread, sc):
            pair = x[:, d - r::2] + x[:, d - r + 1::2]
            x[:, d - r::2] = pair
            x[:, d - r + 1::2] = pair
    return AttBound(bnd, spread, sc)


def lse_bound(q, t, rows, scale, f) -> np.ndarray:
    """Per head bound on |lse_gpu - lse_oracle|: the denominator sums the
    bf16-rounded weights (relative u = 2^-8, so log(den) moves by at most u)
    and each weight carries the fp32 score error delta_r of attention_bound,
    so log(den) moves by at most max_r delta_r more."""
    rows = np.asarray(rows, dtype=np.float64).reshape(-1, np.asarray(q).shape[1])
    if rows.shape[0] == 0:
        return np.full(np.asarray(q).shape[0], 1e-6)
    qr = O.rope_rotate(np.asarray(q, dtype=np.float64), t, f)
    delta = ATT_MMA_STEPS * 2.0 ** -24 * abs(scale) * (np.abs(qr) @ np.abs(rows).T) + ATT_WEIGHT_FIX
    return BF16_U + delta.max(axis=1) + 1e-6


def _current_test() -> str:
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def assert_attention_close(got: np.ndarray, ref: np.ndarray, bound: AttBound, what: str = ""):
    """Per element |gpu - oracle| <= 2e-2 + u (D + B + |oracle|) + S, and
    rel-L2 <= 1e-2 (terms as in attention_bound). The raw max-abs error and
    rel-L2 against the flat 2e-2 / 1e-2 bars go to PARITY_LOG and into the
    assertion message."""
    err = np.abs(got - ref)
    lim = ATT_MAX_ABS + BF16_U * (bound.spread + bound.sum_pv + np.abs(ref)) + bound.score
    worst = int(np.argmax(err / lim)) if err.size else 0
    den = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / den if den > 0 else float(np.linalg.norm(got - ref))
    max_abs = float(err.max()) if err.size else 0.0
    used = float((err / lim).flat[worst]) if err.size else 0.0
    n_over = int((err > ATT_MAX_ABS).sum())
    PARITY_LOG.append((_current_test(), what, max_abs, rel, used, n_over, int(err.size)))
    ok = bool(np.all(err <= lim)) and rel <= ATT_REL_L2
    assert ok, (f"{what}: worst |err| {float(err.flat[worst]):.3e} at |ref| {float(np.abs(ref).flat[worst]):.3e} "
                f"(B {float(bound.sum_pv.flat[worst]):.3e}, D {float(bound.spread.flat[worst]):.3e}, "
                f"S {float(bound.score.flat[worst]):.3e}, limit "
                f"{float(lim.flat[worst]):.3e}); max-abs {max_abs:.3e} vs 2e-2 ({n_over} elements above), "
                f"rel-L2 {rel:.3e} vs 1e-2")


def score_tolerance(ref: np.ndarray, q_idx: np.ndarray, w: np.ndarray, keys: np.ndarray) -> np.ndarray:
    bound = (np.abs(w) * np.linalg.norm(q_idx, axis=1)).sum() * np.linalg.norm(keys, axis=1)
    return SCORE_REL * np.abs(ref) + SCORE_ABS_FRAC * bound


def assert_rows_close_bf16(got: np.ndarray, ref: np.ndarray, what: str = ""):
    rms = np.sqrt(np.mean(ref * ref, axis=-1, keepdims=True))
    tol = F.bf16_ulp(ref) + 1e-5 * rms
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off, worst {float(np.abs(got - ref).max()):.3e}"


def assert_rows_close_fp8(got: np.ndarray, ref: np.ndarray, scale: np.ndarray, what: str = ""):
    """One e4m3 grid step: relative 2^-3 of the value plus the subnormal step 2^-9 * scale."""
    tol = 2.0 ** -3 * np.abs(ref) + 2.0 ** -9 * np.repeat(scale, 32, axis=-1) + 1e-30
    bad = np.abs(got - ref) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} elements off"


def check_topk_valid(sel_gpu: np.ndarray, sel_ref: np.ndarray, scores_ref: np.ndarray, tol: np.ndarray):
    """The GPU's selection differs from the oracle's only among scores within `tol` of the threshold."""
    a = set(int(x) for x in sel_gpu if x >= 0)
    b = set(int(x) for x in sel_ref if x >= 0)
    assert len(a) == len(b)
    if a == b:
        return True
    thr = min(scores_ref[list(b)]) if b else -np.inf
    for j in a ^ b:
        assert abs(scores_ref[j] - thr) <= 2 * tol[j] + 1e-30, f"entry {j} is not a near tie"
    return False


def rope_sanity(ctx):
    """The library's RoPE frequencies against the oracle's own (both computed in double)."""
    g = geometry(ctx.cfg)
    ref = inv_freq(g)
    got = np.array(ctx.rope_frequencies())
    assert np.allclose(got, ref, rtol=1e-14, atol=0)
