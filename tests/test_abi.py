"""The C-ABI library builds, loads and exports every symbol include/csa2.h declares.

No compute call is made here (no GPU is needed).
"""
import ctypes as C
import os
import re

import pytest

from compressed_sparse_attention_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "csa2.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib_path():
    return build.build()


def test_header_declares_the_four_steps_and_the_mode_dispatch():
    names = declared_functions()
    for n in ("csa2_compress", "csa2_index_score", "csa2_topk", "csa2_attend", "csa2_step",
              "csa2_create", "csa2_destroy", "csa2_check"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = C.CDLL(lib_path)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert missing == []


def test_binding_covers_every_declared_symbol(lib_path):
    from compressed_sparse_attention_gb300 import binding
    assert sorted(binding.SIGNATURES) == declared_functions()
    binding.load_library(lib_path)


def test_default_config_and_status_strings(lib_path):
    from compressed_sparse_attention_gb300 import binding
    cfg = binding.default_config()
    assert (cfg.n_heads, cfg.head_dim, cfg.rope_dim, cfg.window, cfg.compress_ratio) == (64, 512, 64, 128, 4)
    assert (cfg.idx_heads, cfg.idx_dim, cfg.topk) == (8, 128, 512)
    assert cfg.softmax_scale == pytest.approx(512 ** -0.5)
    assert cfg.rope_theta == 160000.0 and cfg.yarn_factor == 16.0 and cfg.yarn_orig_len == 65536.0
    lib = binding.load_library()
    assert lib.csa2_status_string(0) == b"ok"
    assert lib.csa2_status_string(6) == b"workspace too small"


def test_create_rejects_unsupported_geometry_without_touching_cuda(lib_path):
    from compressed_sparse_attention_gb300 import binding
    lib = binding.load_library()
    h = C.c_void_p()
    for field, bad in (("n_heads", 32), ("head_dim", 256), ("idx_heads", 12), ("topk", 4096),
                       ("window", 256), ("rope_dim", 32)):
        cfg = binding.default_config()
        setattr(cfg, field, bad)
        assert lib.csa2_create(C.byref(cfg), C.byref(h)) == 2
    assert lib.csa2_create(None, C.byref(h)) == 1


def test_null_context_is_rejected(lib_path):
    from compressed_sparse_attention_gb300 import binding
    lib = binding.load_library()
    assert lib.csa2_topk_workspace_size(None, 4, 100) == 0
    assert lib.csa2_check(None, None, None) == 1
    assert lib.csa2_last_error(None) == b"no context"
