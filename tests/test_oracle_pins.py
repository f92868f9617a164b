"""Pins of the CPU oracle to facts fixed outside it (no GPU needed).

Each test checks the oracle against something it cannot simply agree with by
construction: a worked example printed on the pages (tests/golden), a closed
form, an invariant, brute force through a library routine, or an independent
library implementation of a number format.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import csa2_oracle as O
from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


NO_ROPE = np.zeros(0)


# ---------------------------------------------------------------- worked examples

def test_softmax_worked_example():
    g = golden("softmax_worked_example.json")
    k2 = math.log(3.0)
    # key and value share a row: channel 0 carries the key, channel 1 the value
    rows = np.array([[0.0, g["values"][0]], [k2, g["values"][1]]])
    q = np.array([[g["q"], 0.0]])
    out, lse = O.attend(q, 0, rows, np.array([-np.inf]), 1.0, NO_ROPE)
    assert out[0, 1] == pytest.approx(g["output"], abs=1e-12)
    assert out[0, 0] == pytest.approx(g["weights"][1] * k2, abs=1e-12)
    assert lse[0] == pytest.approx(math.log(1.0 + 3.0), abs=1e-12)


def test_pooling_worked_example():
    g = golden("pooling_worked_example.json")
    c = np.array(g["c"])
    # weights (0.75, 0.25) come from logits that differ by ln 3, the same on both channels
    gate = np.array([[math.log(3.0)] * 2, [0.0] * 2]) + 0.37
    kv, c_hat, _ = O.compress(c, gate, g["m"], 0, np.ones(2), 0.0, NO_ROPE)
    pooled = np.array(g["pooled"])
    assert np.allclose(c_hat[0] * math.sqrt(np.mean(pooled ** 2)), pooled, atol=1e-12)
    assert np.allclose(kv, c_hat)  # no rope dims here


def test_indexer_worked_example():
    g = golden("indexer_worked_example.json")
    s = O.index_scores(np.array([g["q_idx"]]), np.array([g["omega"]]), np.array(g["keys"]))
    assert np.array_equal(s, np.array(g["scores"]))
    assert O.topk_select(s, 1).tolist() == g["top1"]
    # entries 1 and 2 tie at 0: the lower index wins the second slot
    assert O.topk_select(s, 2).tolist() == [0, 1]
    assert O.topk_select(s, 5).tolist() == [0, 1, 2, -1, -1]


def test_window_worked_example():
    g = golden("window_worked_example.json")
    wp = O.window_positions(g["i"], g["w"], g["s"])
    assert (wp[0], wp[-1], len(wp)) == (g["first_key"], g["last_key"], g["n_keys"])
    assert len(O.window_positions(g["i"], g["w"], 0)) == g["n_keys_uncut"]
    assert len(O.window_positions(50, 128)) == 51
    assert len(O.window_positions(127, 128)) == 128
    assert len(O.window_positions(5000, 128)) == 128


def test_kv_bytes_worked_example():
    g = golden("kv_bytes_worked_example.json")
    assert O.global_kv_bytes_per_token(g["example_layers"]) == g["example_bytes_per_token"]
    bm = O.entry_bytes(512, "fp4_e4m3_b16")
    bi = O.entry_bytes(128, "mxfp4_b32")
    assert (bm, bi) == (g["main_entry_bytes"], g["index_entry_bytes"])
    b = O.global_kv_bytes_per_token([(bm, bi, m) for m in g["model_layers_m"]])
    assert b == g["model_bytes_per_token"]
    assert round(b * 1e6 / 1e9, 2) == g["context_1m_gb"]
    # this build's storage formats
    assert O.entry_bytes(512, "bf16") == 1024
    assert O.entry_bytes(512, "fp8_b32") == 528
    assert O.entry_bytes(128, "bf16") == 256
    assert O.entry_bytes(128, "fp8_b32") == 132


# ---------------------------------------------------------------- softmax closed forms

def test_sink_neg_inf_equal_scores_is_mean():
    rng = np.random.default_rng(0)
    rows = rng.standard_normal((7, 16))
    q = np.zeros((3, 16))
    out, _ = O.attend(q, 0, rows, np.full(3, -np.inf), 1.0, NO_ROPE)
    assert np.allclose(out, rows.mean(axis=0)[None, :], atol=1e-12)


def test_sink_zero_equal_scores_weights_one_over_n_plus_one():
    rng = np.random.default_rng(1)
    rows = rng.standard_normal((9, 16))
    q = np.zeros((2, 16))
    out, lse = O.attend(q, 0, rows, np.zeros(2), 1.0, NO_ROPE)
    assert np.allclose(out, rows.sum(axis=0)[None, :] / 10.0, atol=1e-12)
    assert np.allclose(lse, math.log(10.0))


def test_permuting_rows_leaves_output():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((40, 32))
    q = rng.standard_normal((4, 32))
    sink = rng.standard_normal(4)
    f = O.yarn_inv_freq(8, 10000.0, 1.0, 1.0, 32, 1)
    a, la = O.attend(q, 77, rows, sink, 0.3, f)
    b, lb = O.attend(q, 77, rows[rng.permutation(40)], sink, 0.3, f)
    assert np.allclose(a, b, atol=1e-12) and np.allclose(la, lb, atol=1e-12)


def test_identical_rows_give_derotated_row():
    # every row equal to v: out = RoPE_{-t}(v) * (1 - sink weight)
    rng = np.random.default_rng(3)
    v = rng.standard_normal(32)
    rows = np.tile(v, (5, 1))
    q = rng.standard_normal((2, 32))
    f = O.yarn_inv_freq(8, 10000.0, 1.0, 1.0, 32, 1)
    t = 1234
    out, lse = O.attend(q, t, rows, np.array([0.5, -3.0]), 0.2, f)
    # the rotation, written as complex multiplication by exp(-i t f)
    z = (v[24::2] + 1j * v[25::2]) * np.exp(-1j * t * f)
    v_der = v.copy()
    v_der[24::2], v_der[25::2] = z.real, z.imag
    qr = O.rope_rotate(q, t, f)
    s = 0.2 * (qr @ v)
    p_rows = 5 * np.exp(s) / (5 * np.exp(s) + np.exp([0.5, -3.0]))
    assert np.allclose(out, p_rows[:, None] * v_der[None, :], atol=1e-12)


def test_empty_rows_and_neg_inf_sink_give_zero():
    out, lse = O.attend(np.ones((2, 8)), 3, np.zeros((0, 8)), np.full(2, -np.inf), 1.0, NO_ROPE)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


# ---------------------------------------------------------------- RoPE / YaRN

def test_rope_inverse_is_identity_and_relative():
    rng = np.random.default_rng(4)
    f = O.yarn_inv_freq(64, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    x = rng.standard_normal((3, 512))
    y = O.rope_rotate(O.rope_rotate(x, 98765, f), 98765, f, inverse=True)
    assert np.allclose(x, y, atol=1e-12)
    assert np.array_equal(O.rope_rotate(x, 0, f), x)
    # only the last 64 dims move
    assert np.array_equal(O.rope_rotate(x, 12345, f)[:, :448], x[:, :448])
    q, k = rng.standard_normal(512), rng.standard_normal(512)
    d1 = O.rope_rotate(q, 5, f) @ O.rope_rotate(k, 3, f)
    d2 = O.rope_rotate(q, 100005, f) @ O.rope_rotate(k, 100003, f)
    assert d1 == pytest.approx(d2, rel=1e-9)


def test_rope_matches_complex_multiplication():
    rng = np.random.default_rng(5)
    f = O.yarn_inv_freq(64, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    x = rng.standard_normal(512)
    t = 4321
    z = (x[448::2] + 1j * x[449::2]) * np.exp(1j * t * f)
    y = O.rope_rotate(x, t, f)
    assert np.allclose(y[448::2], z.real) and np.allclose(y[449::2], z.imag)


def test_yarn_plain_rope_when_factor_one():
    f = O.yarn_inv_freq(64, 10000.0, 1.0, 65536.0, 32.0, 1.0)
    assert np.allclose(f, [10000.0 ** (-2 * i / 64) for i in range(32)], rtol=1e-15)


def test_yarn_ramp_boundaries_from_turn_counts():
    d, theta, L, s = 64, 160000.0, 65536.0, 16.0
    f = O.yarn_inv_freq(d, theta, s, L, 32.0, 1.0)
    base = np.array([theta ** (-2 * i / d) for i in range(d // 2)])

    def turns(i):  # times pair i turns over the original context
        return L / (2 * math.pi * theta ** (2 * i / d))

    lo = max(i for i in range(d // 2) if turns(i) > 32)   # last pair turning > 32 times
    hi = min(i for i in range(d // 2) if turns(i) < 1)    # first pair turning < 1 time
    assert (lo, hi) == (15, 25)
    # fast pairs keep their frequency, slow pairs are divided by the factor
    assert np.allclose(f[: lo + 1], base[: lo + 1], rtol=1e-15)
    assert np.allclose(f[hi:], base[hi:] / s, rtol=1e-15)
    # halfway along the ramp the blend is an even mix
    assert f[20] == pytest.approx(base[20] * (0.5 / s + 0.5), rel=1e-14)
    ratio = f / base
    assert np.all(np.diff(ratio) <= 1e-15)


# ---------------------------------------------------------------- compressor

def _rand_comp(m, T=8, D=32, seed=6):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((T, D)), rng.standard_normal((T, D)), 0.5 + rng.random(D)


def test_compress_ratio_one_is_rmsnorm_then_rope():
    raw, _, w = _rand_comp(1)
    f = O.yarn_inv_freq(8, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    kv, c_hat, _ = O.compress(raw, None, 1, 40, w, 1e-20, f)
    rms = np.sqrt(np.mean(raw ** 2, axis=1, keepdims=True))
    assert np.allclose(c_hat, raw / rms * w, atol=1e-12)
    assert np.allclose(kv, O.rope_rotate(c_hat, 40 + np.arange(8), f), atol=1e-12)


def test_compress_gate_shift_invariance_and_mean_pool():
    raw, gate, w = _rand_comp(4, T=12)
    _, a, _ = O.compress(raw, gate, 4, 0, w, 1e-20, NO_ROPE)
    shift = np.repeat(np.random.default_rng(7).standard_normal((3, 1, 32)), 4, axis=1).reshape(12, 32)
    _, b, _ = O.compress(raw, gate + shift, 4, 0, w, 1e-20, NO_ROPE)
    assert np.allclose(a, b, atol=1e-12)
    _, c, _ = O.compress(raw, np.zeros_like(gate), 4, 0, np.ones(32), 0.0, NO_ROPE)
    mean = raw.reshape(3, 4, 32).mean(axis=1)
    assert np.allclose(c, mean / np.sqrt(np.mean(mean ** 2, axis=1, keepdims=True)), atol=1e-12)


def test_compress_rope_at_first_token_and_unrotated_index_key():
    raw, gate, w = _rand_comp(2, T=6, D=32)
    f = O.yarn_inv_freq(8, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    rng = np.random.default_rng(8)
    wi, kn = rng.standard_normal((16, 32)), 0.5 + rng.random(16)
    kv0, ch0, k0 = O.compress(raw, gate, 2, 0, w, 1e-20, f, wi, kn)
    kv1, ch1, k1 = O.compress(raw, gate, 2, 1000, w, 1e-20, f, wi, kn)
    assert np.allclose(ch0, ch1) and np.allclose(k0, k1)  # no position in c_hat or k_I
    assert np.allclose(kv1, O.rope_rotate(ch1, np.array([1000, 1002, 1004]), f))
    assert np.allclose(kv0[0], ch0[0])  # group 0 sits at position 0
    # k_I is RMS-normalised: unit RMS before its weight
    assert np.allclose(np.sqrt(np.mean((k0 / kn) ** 2, axis=1)), 1.0)


@pytest.mark.parametrize("m", [1, 2, 4])
def test_compressor_state_chunking_independent(m):
    """Fed token by token, in random chunks, or at once, the stateful
    compressor emits the same entries (exactly) as one compress of every
    complete group, and keeps the open tail pending."""
    rng = np.random.default_rng(60 + m)
    T, D = 61, 32
    raw, gate = rng.standard_normal((T, D)), rng.standard_normal((T, D))
    w = 0.5 + rng.random(D)
    f = O.yarn_inv_freq(8, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    wi, kn = rng.standard_normal((16, D)), 0.5 + rng.random(16)
    n_full = (T // m) * m
    kv_ref, ch_ref, k_ref = O.compress(raw[:n_full], gate[:n_full], m, 0, w, 1e-20, f, wi, kn)

    def run(chunks):
        st = O.CompressorState(m, w, 1e-20, f, wi, kn)
        got, p = [], 0
        for c in chunks:
            got += st.feed(raw[p:p + c], gate[p:p + c], p)
            p += c
        return st, got

    cuts = rng.integers(0, 7, size=40)
    cuts = cuts[np.cumsum(cuts) <= T]
    for chunks in ([T], [1] * T, list(cuts) + [T - int(cuts.sum())]):
        st, got = run(chunks)
        assert [g[0] for g in got] == list(range(T // m))
        assert np.array_equal(np.stack([g[1] for g in got]), kv_ref)
        assert np.array_equal(np.stack([g[2] for g in got]), ch_ref)
        # the key's matrix product goes through BLAS, whose summation order
        # depends on how many rows it multiplies at once: float64 rounding only
        assert np.allclose(np.stack([g[3] for g in got]), k_ref, rtol=1e-13, atol=1e-13)
        assert st.pending() == T - n_full


def test_compressor_state_emits_only_when_a_group_closes():
    rng = np.random.default_rng(66)
    raw, gate = rng.standard_normal((9, 16)), rng.standard_normal((9, 16))
    st = O.CompressorState(4, np.ones(16), 1e-20, NO_ROPE)
    emitted = [len(st.feed(raw[i:i + 1], gate[i:i + 1], i)) for i in range(9)]
    assert emitted == [0, 0, 0, 1, 0, 0, 0, 1, 0]  # a step at a non-flush position writes nothing
    with pytest.raises(ValueError):
        st.feed(raw[:1], gate[:1], 3)  # out of order


# ---------------------------------------------------------------- indexer and top-k

def test_candidate_pool_is_everything_when_few_blocks():
    """With no more blocks than n_keep the pool is every visible entry and the
    pool top-k is the plain top-k (R, C3 reduces to C2 step 3)."""
    rng = np.random.default_rng(80)
    s = rng.standard_normal(1000)
    cand = O.candidate_blocks(s, 8, 2048)
    assert np.array_equal(cand, np.arange(125))
    assert np.array_equal(O.pool_entries(cand, 1000), np.arange(1000))
    assert np.array_equal(O.pool_topk(s, cand, 100), O.topk_select(s, 100))


def test_candidate_blocks_brute_force_and_ties():
    rng = np.random.default_rng(81)
    for n in (37, 64, 203):
        s = np.round(rng.standard_normal(n), 1)  # many equal block maxima
        for keep in (1, 3, 6):
            nb = -(-n // 8)
            best = [max(s[8 * b:8 * b + 8]) for b in range(nb)]
            rank = sorted(range(nb), key=lambda b: (b != nb - 1, -best[b], b))  # newest block first, then by score
            assert list(O.candidate_blocks(s, 8, keep)) == sorted(rank[:keep])


def test_candidate_pool_pins_the_block_still_filling():
    """An older full block that outscores the newest, half-filled block does
    not push it out of the pool (P, "The container")."""
    s = np.concatenate([np.full(8, 5.0), np.full(8, 4.0), np.full(3, -1.0)])
    assert list(O.candidate_blocks(s, 8, 1)) == [2]
    assert list(O.candidate_blocks(s, 8, 2)) == [0, 2]
    assert list(O.pool_entries(O.candidate_blocks(s, 8, 2), 19)) == list(range(8)) + [16, 17, 18]


def test_pool_topk_selects_inside_the_pool():
    rng = np.random.default_rng(82)
    s = rng.standard_normal(4096)
    cand = O.candidate_blocks(s, 8, 64)
    P = O.pool_entries(cand, 4096)
    assert P.shape[0] <= 64 * 8 and np.all(np.diff(P) > 0)
    sel = O.pool_topk(s, cand, 40)
    assert set(sel) <= set(P)
    # the k largest pool scores, ties to the lower entry
    order = sorted(P, key=lambda j: (-s[j], j))[:40]
    assert list(sel) == sorted(order)


def test_hierarchical_pool_size_arithmetic():
    """R, C3: 2,048 blocks of 8 bound the pool at 16,384 entries; at N = 10^6
    decoder scoring per query falls from 5 x 10^6 to 10^6 + 4 x 16,384, about
    1.07 x 10^6 (4.7x), and each Reindex layer scores 61x fewer entries."""
    s = np.random.default_rng(83).standard_normal(200000)
    assert O.pool_entries(O.candidate_blocks(s, 8, 2048), s.shape[0]).shape[0] == 2048 * 8 == 16384
    per_query = 10 ** 6 + 4 * 16384
    assert round(per_query / 1e6, 2) == 1.07 and round(5e6 / per_query, 1) == 4.7
    assert int(10 ** 6 / 16384) == 61


def test_index_scores_closed_forms():
    rng = np.random.default_rng(9)
    qi, keys = rng.standard_normal((8, 16)), rng.standard_normal((50, 16))
    w = rng.random(8)
    s = O.index_scores(qi, w, keys)
    # one head with weight 1 is the ReLU of the dot product
    one = O.index_scores(qi[:1], np.ones(1), keys)
    assert np.allclose(one, np.maximum(keys @ qi[0], 0))
    assert np.allclose(O.index_scores(qi, 3.0 * w, keys), 3.0 * s)
    assert np.allclose(O.index_scores(-qi, w, -keys), s)


@pytest.mark.parametrize("tie_levels", [0, 3, 17])
def test_topk_matches_python_sorted(tie_levels):
    from workloads import make_topk_scores
    sc = make_topk_scores(4, 300, seed=tie_levels, tie_levels=tie_levels).numpy()
    for k in (1, 7, 64, 299, 300, 512):
        for row in sc:
            ref = sorted(range(len(row)), key=lambda j: (-float(row[j]) if row[j] != 0 else 0.0, j))[:k]
            exp = sorted(ref) + [-1] * (k - len(ref))
            assert O.topk_select(row, k).tolist() == exp


def test_topk_negative_zero_ties_positive_zero():
    s = np.array([-0.0, 0.0, -1.0, 0.0], dtype=np.float32)
    assert O.topk_select(s, 1).tolist() == [0]
    assert O.topk_select(s, 2).tolist() == [0, 1]


# ---------------------------------------------------------------- brute force through a library routine

def _brute_force(q, t, rows, sink, scale, f):
    """Dense attention via torch's scaled_dot_product_attention in float64.

    The sink enters as one extra key whose logit is sink_h and whose value is 0:
    queries get one extra channel equal to 1, and the sink key holds sink_h there.
    RoPE is complex multiplication of adjacent pairs.
    """
    H, D = q.shape
    r = 2 * f.shape[0]

    def rot(x, ang):
        x = x.copy()
        z = (x[..., D - r::2] + 1j * x[..., D - r + 1::2]) * np.exp(1j * ang)
        x[..., D - r::2], x[..., D - r + 1::2] = z.real, z.imag
        return x

    qr = rot(q, t * f) * scale
    R = rows.shape[0]
    qa = np.concatenate([qr, np.ones((H, 1))], axis=1)[None, :, None, :]
    ka = np.zeros((1, H, R + 1, D + 1))
    ka[0, :, :R, :D] = rows
    ka[0, :, R, D] = sink
    va = np.zeros((1, H, R + 1, D))
    va[0, :, :R, :] = rows
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(qa), torch.from_numpy(ka), torch.from_numpy(va), scale=1.0).numpy()[0, :, 0, :]
    return rot(o, -t * f)


@pytest.mark.parametrize("t", [0, 3, 6, 17, 40])
@pytest.mark.parametrize("m", [1, 2, 4])
def test_untruncated_csa2_equals_dense_attention(t, m):
    geom = O.Geometry(n_heads=4, head_dim=32, rope_dim=8, window=8, compress_ratio=m,
                      idx_heads=2, idx_dim=16, topk=64)
    rng = np.random.default_rng(100 + t * 7 + m)
    f = O.yarn_inv_freq(8, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    win = rng.standard_normal((64, 32))         # raw rows by position
    comp = rng.standard_normal((64, 32))        # compressed rows by entry index
    keys = rng.standard_normal((64, 16))
    q = rng.standard_normal((4, 32))
    sink = rng.standard_normal(4)
    out, lse, sel, sc = O.step_query(O.MODE_FULL, geom, f, q=q, t=t, win_rows_by_pos=lambda p: win[p],
                                     comp_rows=comp, sink=sink, q_idx=rng.standard_normal((2, 16)),
                                     w_heads=rng.random(2), idx_keys=keys)
    n_vis = sum(1 for j in range(64) if (j + 1) * m - 1 <= t)
    assert sel.tolist() == list(range(n_vis)) + [-1] * (64 - n_vis)
    rows = np.concatenate([win[max(0, t - 7): t + 1], comp[:n_vis]], axis=0)
    ref = _brute_force(q, t, rows, sink, geom.softmax_scale, f)
    assert np.allclose(out, ref, atol=1e-12)


def test_reuse_equals_reindex_with_its_selection():
    geom = O.Geometry(n_heads=4, head_dim=32, rope_dim=8, window=8, compress_ratio=1,
                      idx_heads=2, idx_dim=16, topk=5)
    rng = np.random.default_rng(11)
    f = O.yarn_inv_freq(8, 160000.0, 16.0, 65536.0, 32.0, 1.0)
    win, comp, keys = rng.standard_normal((64, 32)), rng.standard_normal((64, 32)), rng.standard_normal((64, 16))
    kw = dict(q=rng.standard_normal((4, 32)), t=30, win_rows_by_pos=lambda p: win[p], comp_rows=comp,
              sink=rng.standard_normal(4))
    a, la, sel, _ = O.step_query(O.MODE_REINDEX, geom, f, q_idx=rng.standard_normal((2, 16)),
                                 w_heads=rng.random(2), idx_keys=keys, **kw)
    b, lb, sel2, _ = O.step_query(O.MODE_REUSE, geom, f, sel=sel, **kw)
    assert np.array_equal(sel, sel2) and np.array_equal(a, b)


# ---------------------------------------------------------------- number formats against torch's own conversions

def test_bf16_rounding_matches_torch():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(20000, generator=g) * 8)
    ref = x.to(torch.bfloat16).view(torch.uint16).numpy()
    got = F.f64_to_bf16_bits(x.double().numpy())
    assert np.array_equal(ref, got)
    one = 1.0
    assert F.f64_to_bf16_bits(np.array([one + 2 ** -8]))[0] == 0x3F80       # tie -> even
    assert F.f64_to_bf16_bits(np.array([one + 3 * 2 ** -8]))[0] == 0x3F82   # tie -> even (up)
    assert F.f64_to_bf16_bits(np.array([-2.0]))[0] == 0xC000
    assert F.bf16_bits_to_f64(np.array([0x3F80], dtype=np.uint16))[0] == 1.0


def test_e4m3_rounding_matches_torch_within_range():
    g = torch.Generator().manual_seed(1)
    x = torch.randn(20000, generator=g, dtype=torch.float32) * torch.exp(torch.randn(20000, generator=g) * 3)
    x = x.clamp(-448, 448)
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.f64_to_e4m3_bits(x.double().numpy())
    assert np.array_equal(ref, got)
    vals = F.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    tv = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(vals), np.isnan(tv))
    assert np.array_equal(vals[~np.isnan(vals)], tv[~np.isnan(tv)])


def test_e4m3_special_points():
    assert F.f64_to_e4m3_bits(np.array([448.0]))[0] == 0x7E
    assert F.f64_to_e4m3_bits(np.array([470.0]))[0] == 0x7E     # saturates
    assert F.f64_to_e4m3_bits(np.array([-1e9]))[0] == 0xFE
    assert F.f64_to_e4m3_bits(np.array([2.0 ** -9]))[0] == 0x01  # smallest subnormal
    assert F.f64_to_e4m3_bits(np.array([2.0 ** -10]))[0] == 0x00  # tie -> even (zero)
    assert F.f64_to_e4m3_bits(np.array([3 * 2.0 ** -10]))[0] == 0x02  # tie -> even (two quanta)


def test_fp8_block_scale_choice():
    E = F.fp8_block_scale_exponent
    assert E(448.0) == 127
    assert E(np.nextafter(448.0, 1e9)) == 128
    assert E(224.0) == 126
    assert E(224.5) == 127
    assert E(1.0) == 127 - 8
    assert E(0.0) == 0
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 64)) * np.exp(rng.standard_normal((6, 1)) * 4)
    codes, exps = F.fp8_block_quantize(x)
    back = F.fp8_block_dequantize(codes, exps)
    # within half a quantum of the block's grid (3 fraction bits)
    blk = np.abs(x).reshape(6, 2, 32).max(axis=2)
    assert np.all(np.abs(back - x).reshape(6, 2, 32) <= blk[:, :, None] * 2.0 ** -4 + 1e-300)
    assert np.all(np.abs(back).reshape(6, 2, 32).max(axis=2) <= 448 * F.ue8m0_to_f64(exps))


def test_fp8_block_scale_vectorised_equals_scalar_definition():
    rng = np.random.default_rng(13)
    amax = np.abs(rng.standard_normal(5000)) * np.exp(rng.standard_normal(5000) * 6)
    amax[:6] = [0.0, 448.0, np.nextafter(448.0, 1e9), 224.0, 2.0 ** -140, 3.0e38]
    got = F.fp8_block_scale_exponents(amax)
    ref = np.array([F.fp8_block_scale_exponent(float(a)) for a in amax], dtype=np.uint8)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- fp4 formats

def test_fp4_worked_example():
    """The page's 4-of-16 example: amax 2.4 gives s = 0.4 before the scale
    itself is rounded to E4M3 (0.40625); both give codes (6, 3, -1.5, 0)."""
    g = golden("fp4_worked_example.json")
    x = np.zeros((1, 16))
    x[0, :4] = g["x"]
    # the page's arithmetic with its unrounded scale
    s0 = g["scale_from_amax"]
    assert np.allclose(np.array(g["x"]) / s0, g["x_over_s"], rtol=0, atol=1e-12)
    assert F.e2m1_codes_to_f64(F.f64_to_e2m1_codes(np.array(g["x_over_s"]))).tolist() == g["codes"]
    assert np.allclose(s0 * np.array(g["codes"]), g["decoded"], atol=1e-12)
    # the stored form: scale e4m3(amax / 6), codes from x / stored scale
    codes, sbits = F.fp4_block_quantize(x)
    s = float(F.e4m3_bits_to_f64(sbits)[0, 0])
    assert s == 0.40625                                  # nearest E4M3 to 0.4 (1.625 * 2^-2)
    assert F.e2m1_codes_to_f64(codes)[0, :4].tolist() == g["codes"]
    dec = F.fp4_block_dequantize(codes, sbits)[0, :4]
    assert np.array_equal(dec, s * np.array(g["codes"]))
    assert np.allclose(dec, g["decoded"], rtol=2.0 ** -4, atol=0)  # one E4M3 scale step from the page's


def test_fp4_zero_block_takes_the_floor_scale():
    g = golden("fp4_worked_example.json")
    codes, sbits = F.fp4_block_quantize(np.zeros((2, 32)))
    assert g["amax_floor"] == F.FP4_AMAX_FLOOR == 6 * 2.0 ** -9
    assert np.all(F.e4m3_bits_to_f64(sbits) == 2.0 ** -9)   # e4m3(floor / 6): the smallest subnormal
    assert np.all(F.e2m1_codes_to_f64(codes) == 0.0)
    assert np.all(F.fp4_block_dequantize(codes, sbits) == 0.0)


def test_fp4_scale_is_amax_over_six_not_amax():
    x = np.zeros((1, 16))
    x[0, 0], x[0, 1] = 3.0, -1.0
    codes, sbits = F.fp4_block_quantize(x)
    assert float(F.e4m3_bits_to_f64(sbits)[0, 0]) == 0.5     # 3 / 6, exact in E4M3 (e4m3(3) would be 6x)
    assert F.e2m1_codes_to_f64(codes)[0, :2].tolist() == [6.0, -2.0]


def test_e2m1_rounding_ties_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.26, 2.6, 5.1, 7.0, 1e9, -0.25, -0.76, -3.5])
    got = F.e2m1_codes_to_f64(F.f64_to_e2m1_codes(x))
    # ties go to the code with a zero mantissa bit: 0, 1, 1, 2, 2, 4, 4
    assert got.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 0.5, 3.0, 6.0, 6.0, 6.0, -0.0, -1.0, -4.0]
    assert int(F.f64_to_e2m1_codes(np.array([-0.25]))[0]) == 8   # the sign survives rounding to zero
    # every code decodes onto the page's grid and encodes back to itself
    allc = np.arange(16, dtype=np.uint8)
    assert set(np.abs(F.e2m1_codes_to_f64(allc)).tolist()) == {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    assert np.array_equal(F.f64_to_e2m1_codes(F.e2m1_codes_to_f64(allc)), allc)


def test_mxfp4_scale_is_rounded_power_of_two():
    def ebyte(amax):
        x = np.zeros((1, 32))
        x[0, 0] = amax
        return int(F.mxfp4_block_quantize(x)[1][0, 0])
    assert ebyte(6.0) == 127            # 2^round(log2(1)) = 1
    assert ebyte(8.4) == 127            # log2(1.4) = 0.485 -> 0
    assert ebyte(8.5) == 128            # log2(1.417) = 0.502 -> 1
    assert ebyte(3.0) == 126
    assert ebyte(0.0) == 1              # floor 6 * 2^-126 -> 2^-126
    x = np.zeros((1, 32))
    x[0, :2] = [8.4, -0.3]
    codes, e = F.mxfp4_block_quantize(x)
    # scale 1: 8.4 saturates to the largest code, -0.3 rounds to -0.5
    assert F.mxfp4_block_dequantize(codes, e)[0, :2].tolist() == [6.0, -0.5]


def test_fp4_pack_nibble_order_and_roundtrip():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 16, size=(5, 64)).astype(np.uint8)
    packed = F.pack_e2m1(codes)
    assert packed.shape == (5, 32)
    assert int(packed[0, 0]) == int(codes[0, 0]) | (int(codes[0, 1]) << 4)
    assert np.array_equal(F.unpack_e2m1(packed), codes)


def test_fp4_roundtrip_error_bound():
    """Decoded values sit on the scaled grid, within half a grid gap of x
    (the largest gap, 4..6, bounds it by one scale unit) unless saturated."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 512)) * np.exp(rng.uniform(-6, 6, size=(64, 1)))
    codes, sbits = F.fp4_block_quantize(x)
    dec = F.fp4_block_dequantize(codes, sbits)
    s = np.repeat(F.e4m3_bits_to_f64(sbits), 16, axis=1)
    on_grid = np.isin(np.abs(dec / s), F.E2M1_VALUES)
    assert on_grid.all()
    unsat = np.abs(x / s) <= 6.0
    assert np.all(np.abs(x - dec)[unsat] <= s[unsat] * 1.0 + 1e-300)
    # the scale is within one E4M3 rounding of amax / 6
    amax = np.abs(x.reshape(64, 32, 16)).max(axis=2)
    sv = F.e4m3_bits_to_f64(sbits)
    assert np.all(np.abs(sv - amax / 6) <= np.maximum(amax / 6, 2.0 ** -6) * 2.0 ** -4 + 2.0 ** -10)
