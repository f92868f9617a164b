"""Byte accounting of bench.py's HBM fractions, written out by hand for the
workloads it is quoted on (no GPU): the figures a roofline fraction divides by
must be the bytes the step has to move, no more and no fewer."""
import bench
from workloads import PRESETS

ROW_BF16 = 512 * 2          # one 512-wide bf16 KV row
KEY_BF16 = 128 * 2          # one 128-wide bf16 index key
Q_IN_OUT = 64 * 512 * 2 * 2  # q in and the output out, 64 heads x 512 bf16 each


def test_reuse_layer_bytes_mixed_batch():
    """A Reuse layer reads the borrowed selection, the 128 window rows and 512
    selected rows of each query, q, and writes the output: every sequence of
    the mixed batch is at least 1K long, so each query has all of them."""
    wl = PRESETS["mixed_reuse_b64"]
    per_query = 128 * ROW_BF16 + 512 * ROW_BF16 + 512 * 4 + Q_IN_OUT
    assert bench.reuse_bytes(wl) == wl.n_query * per_query == 50_462_720


def test_reindex_layer_bytes_mixed_batch():
    """A Reindex layer adds every visible index key (ratio 1: n_vis = t + 1 at
    position t = length - 1) and q^I, omega; nothing is compressed."""
    wl = PRESETS["mixed_reuse_b64"]
    keys = sum(n * KEY_BF16 for n in wl.ctx_len)
    per_query = 8 * 128 * 2 + 8 * 4 + 128 * ROW_BF16 + 512 * ROW_BF16 + Q_IN_OUT
    assert bench.algorithmic_bytes(wl, has_compress=False) == keys + wl.n_query * per_query


def test_decode_64k_step_bytes():
    """The headline step: 16,384 keys, 640 rows, q in and out, q^I and omega
    per query, plus each sequence's closing group (4 tokens of raw bf16 and fp32
    gates in, one pool row and one key out)."""
    wl = PRESETS["decode_64k_b32"]
    per_query = 16384 * KEY_BF16 + 640 * ROW_BF16 + Q_IN_OUT + 8 * 128 * 2 + 8 * 4
    per_group = 4 * 512 * (2 + 4) + ROW_BF16 + KEY_BF16
    assert bench.algorithmic_bytes(wl) == 32 * (per_query + per_group) == 159_884_288
