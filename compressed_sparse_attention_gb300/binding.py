"""Thin Python binding of the CSA2 C ABI (include/csa2.h).

Argument marshalling only: every function here checks that its tensors live
on the context's CUDA device with the expected dtype and contiguity, takes
their data pointers and the current CUDA stream, and calls the C entry point
of the same name. All arithmetic happens in the library's CUDA kernels. There
is no fallback: if the shared library is missing or a call fails, an error is
raised.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

_LIB = None

CSA2_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported geometry", 3: "CUDA error",
          4: "bad input recorded on the device", 5: "device wait timed out", 6: "workspace too small"}
KV_BF16, KV_FP8, KV_FP4, KV_MXFP4 = 0, 1, 2, 3
CAND_NONE, CAND_SOURCE, CAND_READ = 0, 1, 2  # csa2_kv_format
MODE_FULL, MODE_REINDEX, MODE_REUSE = 0, 1, 2

FLAG_BAD_TOPK_INDEX = 0x01
FLAG_BAD_WINDOW = 0x02
FLAG_BAD_SEGMENT = 0x04
FLAG_NVIS_TOO_LARGE = 0x08
FLAG_WAIT_TIMEOUT = 0x10
FLAG_BAD_QUERY = 0x20


class Csa2Error(RuntimeError):
    def __init__(self, status, msg=""):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class HostIO(C.Structure):
    _fields_ = [("q", C.c_void_p), ("raw", C.c_void_p), ("gate", C.c_void_p), ("out", C.c_void_p)]


class Config(C.Structure):
    _fields_ = [("n_heads", C.c_int32), ("head_dim", C.c_int32), ("rope_dim", C.c_int32),
                ("window", C.c_int32), ("compress_ratio", C.c_int32), ("idx_heads", C.c_int32),
                ("idx_dim", C.c_int32), ("topk", C.c_int32), ("kv_format", C.c_int32),
                ("idx_key_format", C.c_int32), ("softmax_scale", C.c_float), ("norm_eps", C.c_float),
                ("rope_theta", C.c_double), ("yarn_factor", C.c_double), ("yarn_orig_len", C.c_double),
                ("yarn_beta_fast", C.c_double), ("yarn_beta_slow", C.c_double),
                ("cand_block", C.c_int32), ("cand_keep", C.c_int32)]


class StepArgs(C.Structure):
    _fields_ = [("mode", C.c_int32), ("n_seq", C.c_int32), ("n_query", C.c_int32), ("max_vis", C.c_int64),
                ("q", C.c_void_p), ("q_pos", C.c_void_p), ("seq_of_q", C.c_void_p), ("n_vis", C.c_void_p),
                ("q_idx", C.c_void_p), ("w_heads", C.c_void_p), ("sink", C.c_void_p),
                ("win_kv", C.c_void_p), ("win_scale", C.c_void_p), ("win_off", C.c_void_p),
                ("win_lo", C.c_void_p),
                ("pool_kv", C.c_void_p), ("pool_scale", C.c_void_p), ("idx_keys", C.c_void_p),
                ("idx_key_scale", C.c_void_p), ("pool_off", C.c_void_p),
                ("n_tokens", C.c_int64), ("raw", C.c_void_p), ("gate", C.c_void_p), ("tok_off", C.c_void_p),
                ("first_pos", C.c_void_p), ("norm_w", C.c_void_p), ("w_idx", C.c_void_p),
                ("k_norm_w", C.c_void_p),
                ("topk_idx", C.c_void_p), ("out", C.c_void_p), ("lse", C.c_void_p),
                ("workspace", C.c_void_p), ("workspace_bytes", C.c_size_t),
                ("append", C.c_int32), ("state_raw", C.c_void_p), ("state_gate", C.c_void_p),
                ("cand_role", C.c_int32), ("cand", C.c_void_p)]


# name -> (restype, argtypes); every symbol include/csa2.h declares
SIGNATURES = {
    "csa2_default_config": (None, [C.POINTER(Config)]),
    "csa2_create": (C.c_int, [C.POINTER(Config), C.POINTER(C.c_void_p)]),
    "csa2_destroy": (None, [C.c_void_p]),
    "csa2_last_error": (C.c_char_p, [C.c_void_p]),
    "csa2_status_string": (C.c_char_p, [C.c_int]),
    "csa2_rope_frequencies": (C.c_int, [C.c_void_p, C.POINTER(C.c_double), C.c_int32]),
    "csa2_check": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(C.c_uint32)]),
    "csa2_debug_wait_timeout": (C.c_int, [C.c_void_p, C.c_void_p, C.c_uint64]),
    "csa2_store_rows": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_int32, C.c_void_p,
                                  C.c_int32, C.c_void_p, C.c_void_p]),
    "csa2_compress": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int64,
                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_compress_append": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32, C.c_int64,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                       C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_index_score": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                   C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                   C.c_void_p, C.c_int64]),
    "csa2_topk_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int32, C.c_int64]),
    "csa2_candidate_pool_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int32, C.c_int64]),
    "csa2_candidate_pool": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p,
                                      C.c_int64, C.c_void_p, C.c_void_p, C.c_size_t]),
    "csa2_index_score_pool": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64,
                                        C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_topk_pool": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p,
                                 C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t]),
    "csa2_topk": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_int64,
                            C.c_int32, C.c_void_p, C.c_void_p, C.c_size_t]),
    "csa2_attend_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int32]),
    "csa2_attend": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                              C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                              C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                              C.c_void_p, C.c_size_t]),
    "csa2_step_host": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_step_graph_create": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_step_graph_launch": (C.c_int, [C.c_void_p, C.c_void_p]),
    "csa2_step_graph_destroy": (None, [C.c_void_p]),
    "csa2_step_workspace_size": (C.c_size_t, [C.c_void_p, C.c_int32, C.c_int64]),
    "csa2_step": (C.c_int, [C.c_void_p, C.c_void_p, C.POINTER(StepArgs)]),
    "csa2_last_launch_count": (C.c_int32, [C.c_void_p]),
    "csa2_shard_visible": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_int64,
                                     C.c_void_p]),
    "csa2_topk_pairs": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_void_p, C.c_int64, C.c_void_p, C.c_int32,
                                  C.c_int64, C.c_void_p, C.c_void_p]),
    "csa2_topk_merge": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                  C.c_int32, C.c_void_p]),
    "csa2_attend_partial": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64,
                                      C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_attend_combine": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
    "csa2_attend_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p,
                                      C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]),
}


def library_path() -> str:
    return _build.LIB_PATH


def load_library(path: str | None = None):
    """Load libcsa2.so (built by build.build()); raises if it is absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CSA2 CUDA library not built: {path} is missing "
                           "(run compressed_sparse_attention_gb300.build.build())")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def default_config(**overrides) -> Config:
    lib = load_library()
    cfg = Config()
    lib.csa2_default_config(C.byref(cfg))
    for k, v in overrides.items():
        if k in ("kv_format", "idx_key_format") and isinstance(v, str):
            v = {"bf16": KV_BF16, "fp8": KV_FP8, "fp4": KV_FP4, "mxfp4": KV_MXFP4}[v]
        setattr(cfg, k, v)
    return cfg


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


class Context:
    """Owns one csa2_ctx bound to the current CUDA device."""

    def __init__(self, cfg: Config | None = None, **overrides):
        self.lib = load_library()
        self.cfg = cfg if cfg is not None else default_config(**overrides)
        self.device = torch.device("cuda", torch.cuda.current_device())
        h = C.c_void_p()
        st = self.lib.csa2_create(C.byref(self.cfg), C.byref(h))
        if st != CSA2_OK:
            raise Csa2Error(st, "csa2_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None):
            self.lib.csa2_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- marshalling helpers
    def _p(self, t, dtype=None, name="tensor"):
        if t is None:
            return None
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.device != self.device:
            raise ValueError(f"{name} must be on {self.device}, is on {t.device}")
        if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
            raise TypeError(f"{name} must be {dtype}, is {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()

    def _ok(self, st, what):
        if st != CSA2_OK:
            raise Csa2Error(st, f"{what}: {self.lib.csa2_last_error(self.h).decode()}")

    @property
    def last_launch_count(self) -> int:
        return int(self.lib.csa2_last_launch_count(self.h))

    def rope_frequencies(self):
        n = max(1, self.cfg.rope_dim // 2)
        buf = (C.c_double * n)()
        self._ok(self.lib.csa2_rope_frequencies(self.h, buf, n), "csa2_rope_frequencies")
        return [buf[i] for i in range(self.cfg.rope_dim // 2)]

    def check(self):
        """Synchronise the current stream; return the device error word (raises on error)."""
        fl = C.c_uint32(0)
        st = self.lib.csa2_check(self.h, C.c_void_p(_stream()), C.byref(fl))
        if st not in (CSA2_OK, 4, 5):
            self._ok(st, "csa2_check")
        return int(fl.value), st

    def debug_wait_timeout(self, limit_ns: int):
        """Enqueue the wait probe (csa2_debug_wait_timeout) on the current stream."""
        self._ok(self.lib.csa2_debug_wait_timeout(self.h, C.c_void_p(_stream()), int(limit_ns)),
                 "csa2_debug_wait_timeout")

    # -- entry points
    def store_rows(self, rows, pos, fmt, out, out_scale=None):
        n, dim = rows.shape
        self._ok(self.lib.csa2_store_rows(self.h, C.c_void_p(_stream()), self._p(rows, torch.float32, "rows"),
                                          n, dim, self._p(pos, torch.int64, "pos"), fmt,
                                          self._p(out, None, "out"), self._p(out_scale, torch.uint8, "out_scale")),
                 "csa2_store_rows")

    def compress(self, raw, gate, n_seq, tok_off, first_pos, pool_off, norm_w, w_idx, k_norm_w,
                 pool_kv, pool_kv_scale, idx_keys, idx_key_scale):
        n_tokens = raw.shape[0]
        self._ok(self.lib.csa2_compress(
            self.h, C.c_void_p(_stream()), self._p(raw, torch.bfloat16, "raw"), self._p(gate, torch.float32, "gate"),
            n_seq, n_tokens, self._p(tok_off, torch.int64, "tok_off"), self._p(first_pos, torch.int64, "first_pos"),
            self._p(pool_off, torch.int64, "pool_off"), self._p(norm_w, torch.float32, "norm_w"),
            self._p(w_idx, torch.bfloat16, "w_idx"), self._p(k_norm_w, torch.float32, "k_norm_w"),
            self._p(pool_kv, None, "pool_kv"), self._p(pool_kv_scale, torch.uint8, "pool_kv_scale"),
            self._p(idx_keys, None, "idx_keys"), self._p(idx_key_scale, torch.uint8, "idx_key_scale")),
            "csa2_compress")

    def compress_append(self, raw, gate, n_seq, tok_off, first_pos, pool_off, norm_w, w_idx, k_norm_w,
                        pool_kv, pool_kv_scale, idx_keys, idx_key_scale, state_raw, state_gate):
        n_tokens = 0 if raw is None else raw.shape[0]
        self._ok(self.lib.csa2_compress_append(
            self.h, C.c_void_p(_stream()), self._p(raw, torch.bfloat16, "raw"), self._p(gate, torch.float32, "gate"),
            n_seq, n_tokens, self._p(tok_off, torch.int64, "tok_off"), self._p(first_pos, torch.int64, "first_pos"),
            self._p(pool_off, torch.int64, "pool_off"), self._p(norm_w, torch.float32, "norm_w"),
            self._p(w_idx, torch.bfloat16, "w_idx"), self._p(k_norm_w, torch.float32, "k_norm_w"),
            self._p(pool_kv, None, "pool_kv"), self._p(pool_kv_scale, torch.uint8, "pool_kv_scale"),
            self._p(idx_keys, None, "idx_keys"), self._p(idx_key_scale, torch.uint8, "idx_key_scale"),
            self._p(state_raw, torch.bfloat16, "state_raw"), self._p(state_gate, torch.float32, "state_gate")),
            "csa2_compress_append")

    def index_score(self, n_seq, q_idx, w_heads, idx_keys, idx_key_scale, pool_off, seq_of_q, n_vis, max_vis,
                    scores):
        self._ok(self.lib.csa2_index_score(
            self.h, C.c_void_p(_stream()), n_seq, q_idx.shape[0], self._p(q_idx, torch.bfloat16, "q_idx"),
            self._p(w_heads, torch.float32, "w_heads"), self._p(idx_keys, None, "idx_keys"),
            self._p(idx_key_scale, torch.uint8, "idx_key_scale"), self._p(pool_off, torch.int64, "pool_off"),
            self._p(seq_of_q, torch.int32, "seq_of_q"), self._p(n_vis, torch.int32, "n_vis"), max_vis,
            self._p(scores, torch.float32, "scores"), scores.shape[1]), "csa2_index_score")

    # -- the hierarchical indexer's pool
    def candidate_pool_workspace_size(self, n_query, max_vis) -> int:
        return int(self.lib.csa2_candidate_pool_workspace_size(self.h, n_query, max_vis))

    def candidate_pool(self, scores, n_vis, max_vis, cand, workspace):
        self._ok(self.lib.csa2_candidate_pool(
            self.h, C.c_void_p(_stream()), n_vis.shape[0], self._p(scores, torch.float32, "scores"), scores.shape[1],
            self._p(n_vis, torch.int32, "n_vis"), max_vis, self._p(cand, torch.int32, "cand"),
            self._p(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size()), "csa2_candidate_pool")

    def index_score_pool(self, n_seq, q_idx, w_heads, idx_keys, idx_key_scale, pool_off, seq_of_q, n_vis, max_vis,
                         cand, scores_pool, n_pool):
        self._ok(self.lib.csa2_index_score_pool(
            self.h, C.c_void_p(_stream()), n_seq, q_idx.shape[0], self._p(q_idx, torch.bfloat16, "q_idx"),
            self._p(w_heads, torch.float32, "w_heads"), self._p(idx_keys, None, "idx_keys"),
            self._p(idx_key_scale, torch.uint8, "idx_key_scale"), self._p(pool_off, torch.int64, "pool_off"),
            self._p(seq_of_q, torch.int32, "seq_of_q"), self._p(n_vis, torch.int32, "n_vis"), max_vis,
            self._p(cand, torch.int32, "cand"), self._p(scores_pool, torch.float32, "scores_pool"),
            self._p(n_pool, torch.int32, "n_pool")), "csa2_index_score_pool")

    def topk_pool(self, scores_pool, n_pool, cand, k, out_idx, workspace):
        self._ok(self.lib.csa2_topk_pool(
            self.h, C.c_void_p(_stream()), n_pool.shape[0], self._p(scores_pool, torch.float32, "scores_pool"),
            self._p(n_pool, torch.int32, "n_pool"), self._p(cand, torch.int32, "cand"), k,
            self._p(out_idx, torch.int32, "out_idx"), self._p(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size()), "csa2_topk_pool")

    def topk_workspace_size(self, n_query, max_vis) -> int:
        return int(self.lib.csa2_topk_workspace_size(self.h, n_query, max_vis))

    def topk(self, scores, n_vis, max_vis, k, out_idx, workspace):
        self._ok(self.lib.csa2_topk(
            self.h, C.c_void_p(_stream()), scores.shape[0], self._p(scores, torch.float32, "scores"),
            scores.shape[1], self._p(n_vis, torch.int32, "n_vis"), max_vis, k,
            self._p(out_idx, torch.int32, "out_idx"), self._p(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size()), "csa2_topk")

    def attend_workspace_size(self, n_query) -> int:
        return int(self.lib.csa2_attend_workspace_size(self.h, n_query))

    def attend(self, n_seq, q, q_pos, seq_of_q, win_kv, win_scale, win_off, win_lo, pool_kv, pool_scale, pool_off,
               topk_idx, sink, out, lse, workspace):
        self._ok(self.lib.csa2_attend(
            self.h, C.c_void_p(_stream()), n_seq, q.shape[0], self._p(q, torch.bfloat16, "q"),
            self._p(q_pos, torch.int64, "q_pos"), self._p(seq_of_q, torch.int32, "seq_of_q"),
            self._p(win_kv, None, "win_kv"), self._p(win_scale, torch.uint8, "win_scale"),
            self._p(win_off, torch.int64, "win_off"), self._p(win_lo, torch.int64, "win_lo"),
            self._p(pool_kv, None, "pool_kv"), self._p(pool_scale, torch.uint8, "pool_scale"),
            self._p(pool_off, torch.int64, "pool_off"), self._p(topk_idx, torch.int32, "topk_idx"),
            self._p(sink, torch.float32, "sink"), self._p(out, torch.bfloat16, "out"),
            self._p(lse, torch.float32, "lse"), self._p(workspace, None, "workspace"),
            0 if workspace is None else workspace.numel() * workspace.element_size()), "csa2_attend")

    # -- pool sharding (csa2_shard_visible .. csa2_attend_combine)
    def shard_visible(self, n_vis, lo, hi, out):
        self._ok(self.lib.csa2_shard_visible(self.h, C.c_void_p(_stream()), n_vis.shape[0],
                                             self._p(n_vis, torch.int32, "n_vis"), int(lo), int(hi),
                                             self._p(out, torch.int32, "n_vis_shard")), "csa2_shard_visible")

    def topk_pairs(self, scores, sel, index_base, pair_score, pair_idx):
        self._ok(self.lib.csa2_topk_pairs(self.h, C.c_void_p(_stream()), sel.shape[0],
                                          self._p(scores, torch.float32, "scores"), scores.shape[1],
                                          self._p(sel, torch.int32, "sel"), sel.shape[1], int(index_base),
                                          self._p(pair_score, torch.float32, "pair_score"),
                                          self._p(pair_idx, torch.int32, "pair_idx")), "csa2_topk_pairs")

    def topk_merge(self, pair_score, pair_idx, k, out_idx):
        """pair_score / pair_idx [n_lists, n_query, list_len] -> out_idx [n_query, k]."""
        n_lists, n_query, list_len = pair_idx.shape
        self._ok(self.lib.csa2_topk_merge(self.h, C.c_void_p(_stream()), n_query, n_lists, list_len,
                                          self._p(pair_score, torch.float32, "pair_score"),
                                          self._p(pair_idx, torch.int32, "pair_idx"), k,
                                          self._p(out_idx, torch.int32, "out_idx")), "csa2_topk_merge")

    def attend_partial(self, n_seq, q, q_pos, seq_of_q, with_window, win_kv, win_scale, win_off, win_lo, pool_kv,
                       pool_scale, pool_off, topk_idx, shard_lo, shard_hi, part_o, part_m, part_l):
        self._ok(self.lib.csa2_attend_partial(
            self.h, C.c_void_p(_stream()), n_seq, q.shape[0], self._p(q, torch.bfloat16, "q"),
            self._p(q_pos, torch.int64, "q_pos"), self._p(seq_of_q, torch.int32, "seq_of_q"), 1 if with_window else 0,
            self._p(win_kv, None, "win_kv"), self._p(win_scale, torch.uint8, "win_scale"),
            self._p(win_off, torch.int64, "win_off"), self._p(win_lo, torch.int64, "win_lo"),
            self._p(pool_kv, None, "pool_kv"), self._p(pool_scale, torch.uint8, "pool_scale"),
            self._p(pool_off, torch.int64, "pool_off"), self._p(topk_idx, torch.int32, "topk_idx"),
            int(shard_lo), int(shard_hi), self._p(part_o, torch.float32, "part_o"),
            self._p(part_m, torch.float32, "part_m"), self._p(part_l, torch.float32, "part_l")),
            "csa2_attend_partial")

    def attend_combine(self, part_o, part_m, part_l, q_pos, sink, out, lse=None):
        """part_o [n_parts, n_query, 64, 512], part_m / part_l [n_parts, n_query, 64]."""
        n_parts, n_query = part_m.shape[0], part_m.shape[1]
        self._ok(self.lib.csa2_attend_combine(
            self.h, C.c_void_p(_stream()), n_query, n_parts, self._p(part_o, torch.float32, "part_o"),
            self._p(part_m, torch.float32, "part_m"), self._p(part_l, torch.float32, "part_l"),
            self._p(q_pos, torch.int64, "q_pos"), self._p(sink, torch.float32, "sink"),
            self._p(out, torch.bfloat16, "out"), self._p(lse, torch.float32, "lse")), "csa2_attend_combine")

    def step_workspace_size(self, n_query, max_vis) -> int:
        return int(self.lib.csa2_step_workspace_size(self.h, n_query, max_vis))

    def step(self, mode, n_seq, max_vis, **kw):
        self._ok(self.lib.csa2_step(self.h, C.c_void_p(_stream()), C.byref(self.step_args(mode, n_seq, max_vis, **kw))),
                 "csa2_step")

    def prepare_step(self, mode, n_seq, max_vis, **kw) -> "PreparedStep":
        """The step's argument block built once, for a serving loop that reuses
        its buffers from step to step: each run is then a single C call."""
        return PreparedStep(self, self.step_args(mode, n_seq, max_vis, **kw), kw)

    def step_args(self, mode, n_seq, max_vis, *, q, q_pos, seq_of_q, n_vis, sink, win_kv, win_off, pool_kv,
                  pool_off, topk_idx, out, workspace, q_idx=None, w_heads=None, win_scale=None, win_lo=None,
                  pool_scale=None, idx_keys=None, idx_key_scale=None, raw=None, gate=None, tok_off=None,
                  first_pos=None, norm_w=None, w_idx=None, k_norm_w=None, lse=None, append=False, state_raw=None,
                  state_gate=None, cand_role=0, cand=None) -> StepArgs:
        a = StepArgs()
        a.mode, a.n_seq, a.n_query, a.max_vis = mode, n_seq, q.shape[0], max_vis
        a.q = self._p(q, torch.bfloat16, "q")
        a.q_pos = self._p(q_pos, torch.int64, "q_pos")
        a.seq_of_q = self._p(seq_of_q, torch.int32, "seq_of_q")
        a.n_vis = self._p(n_vis, torch.int32, "n_vis")
        a.q_idx = self._p(q_idx, torch.bfloat16, "q_idx")
        a.w_heads = self._p(w_heads, torch.float32, "w_heads")
        a.sink = self._p(sink, torch.float32, "sink")
        a.win_kv = self._p(win_kv, None, "win_kv")
        a.win_scale = self._p(win_scale, torch.uint8, "win_scale")
        a.win_off = self._p(win_off, torch.int64, "win_off")
        a.win_lo = self._p(win_lo, torch.int64, "win_lo")
        a.pool_kv = self._p(pool_kv, None, "pool_kv")
        a.pool_scale = self._p(pool_scale, torch.uint8, "pool_scale")
        a.idx_keys = self._p(idx_keys, None, "idx_keys")
        a.idx_key_scale = self._p(idx_key_scale, torch.uint8, "idx_key_scale")
        a.pool_off = self._p(pool_off, torch.int64, "pool_off")
        a.n_tokens = 0 if raw is None else raw.shape[0]
        a.raw = self._p(raw, torch.bfloat16, "raw")
        a.gate = self._p(gate, torch.float32, "gate")
        a.tok_off = self._p(tok_off, torch.int64, "tok_off")
        a.first_pos = self._p(first_pos, torch.int64, "first_pos")
        a.norm_w = self._p(norm_w, torch.float32, "norm_w")
        a.w_idx = self._p(w_idx, torch.bfloat16, "w_idx")
        a.k_norm_w = self._p(k_norm_w, torch.float32, "k_norm_w")
        a.topk_idx = self._p(topk_idx, torch.int32, "topk_idx")
        a.out = self._p(out, torch.bfloat16, "out")
        a.lse = self._p(lse, torch.float32, "lse")
        a.workspace = self._p(workspace, None, "workspace")
        a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
        a.append = 1 if append else 0
        a.state_raw = self._p(state_raw, torch.bfloat16, "state_raw")
        a.state_gate = self._p(state_gate, torch.float32, "state_gate")
        a.cand_role = cand_role
        a.cand = self._p(cand, torch.int32, "cand")
        return a


class PreparedStep:
    """A csa2_step argument block kept alive with the tensors it points at."""

    def __init__(self, ctx: Context, args: StepArgs, tensors: dict):
        self.ctx, self.args, self._keep = ctx, args, tensors
        self.io = HostIO()

    def run(self):
        self.ctx._ok(self.ctx.lib.csa2_step(self.ctx.h, C.c_void_p(_stream()), C.byref(self.args)), "csa2_step")

    def run_host(self, q=None, raw=None, gate=None, out=None):
        """csa2_step_host: the step with its inputs in host tensors (pinned):
        q is copied in beside the scan, the raw tokens and gates before
        compress. A pinned `out` is written by the step directly; any other
        host `out` gets one copy of the prepared device output."""
        io = self.io
        io.q = None if q is None else q.data_ptr()
        io.raw = None if raw is None else raw.data_ptr()
        io.gate = None if gate is None else gate.data_ptr()
        io.out = None if out is None else out.data_ptr()
        self.ctx._ok(self.ctx.lib.csa2_step_host(self.ctx.h, C.c_void_p(_stream()), C.byref(self.args),
                                                 C.byref(io)), "csa2_step_host")

    def host_graph(self, q=None, raw=None, gate=None, out=None) -> "StepGraph":
        """csa2_step_graph_create: this step with these host buffers captured
        once; each StepGraph.launch() repeats the copies and the step."""
        io = HostIO()
        io.q = None if q is None else q.data_ptr()
        io.raw = None if raw is None else raw.data_ptr()
        io.gate = None if gate is None else gate.data_ptr()
        io.out = None if out is None else out.data_ptr()
        h = C.c_void_p()
        self.ctx._ok(self.ctx.lib.csa2_step_graph_create(self.ctx.h, C.byref(self.args), C.byref(io), C.byref(h)),
                     "csa2_step_graph_create")
        return StepGraph(self, h, (q, raw, gate, out))


class StepGraph:
    """A captured host step; holds the prepared step and host tensors it uses."""

    def __init__(self, prep: PreparedStep, handle, host_tensors):
        self.prep, self.h, self._keep = prep, handle, host_tensors

    def launch(self):
        self.prep.ctx._ok(self.prep.ctx.lib.csa2_step_graph_launch(self.h, C.c_void_p(_stream())),
                          "csa2_step_graph_launch")

    def __del__(self):
        if getattr(self, "h", None):
            self.prep.ctx.lib.csa2_step_graph_destroy(self.h)
            self.h = None


def workspace(nbytes: int, device=None) -> torch.Tensor:
    """A 256-byte-aligned byte buffer of at least nbytes (caching-allocator memory)."""
    t = torch.empty(max(int(nbytes), 1) + 256, dtype=torch.uint8, device=device or "cuda")
    off = (-t.data_ptr()) % 256
    return t[off:off + max(int(nbytes), 1)]
