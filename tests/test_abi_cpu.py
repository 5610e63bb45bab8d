"""Host-side checks of the C ABI library (no GPU needed): it loads, exports every
symbol include/entmaxkv.h declares, and rejects bad arguments before launching."""
from __future__ import annotations

import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "entmaxkv.h")


@pytest.fixture(scope="module")
def L():
    from sparse_long_context_08_b300 import build, entmaxkv
    build.build()
    return entmaxkv


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|int32_t|size_t|const char\*)\s+(entmaxkv_\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_four_stages():
    syms = declared_symbols()
    for s in ("entmaxkv_build_page_meta", "entmaxkv_score_pages", "entmaxkv_select",
              "entmaxkv_decode"):
        assert s in syms


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    for s in declared_symbols():
        assert hasattr(lib, s), s
    assert set(declared_symbols()) <= set(L.SYMBOLS) | {"entmaxkv_version"}


def test_status_strings_and_version(L):
    assert L.entmaxkv_status_string(0) == "ok"
    assert "workspace" in L.entmaxkv_status_string(3)
    assert L.entmaxkv_status_string(99) == "unknown status"
    assert "timeout" in L.entmaxkv_status_string(L.EKV_DEVICE_TIMEOUT)
    assert L.entmaxkv_version() >= 10000


def test_workspace_size_is_host_only_and_monotone(L):
    a = L.entmaxkv_workspace_size(8, 32, 8, 128, 32, 4096, 128)
    b = L.entmaxkv_workspace_size(8, 32, 8, 128, 32, 4096, 256)
    assert 0 < a < b
    assert L.entmaxkv_workspace_size(8, 30, 8, 128, 32, 4096, 128) == 0   # Hq % Hkv
    assert L.entmaxkv_workspace_size(0, 32, 8, 128, 32, 4096, 128) == 0


def test_full_workspace_size_matches_a_whole_cache_selection(L):
    # the full-cache decode selects every page: its workspace is the decode
    # workspace at cap = max_pages, with per-head candidate buffers once the
    # cache holds more tokens than the shared-memory threshold kernel keeps
    f = L.entmaxkv_full_workspace_size(8, 32, 8, 128, 32, 4096)
    assert f == L.entmaxkv_workspace_size(8, 32, 8, 128, 32, 4096, 4096)
    assert f >= 8 * 32 * 4096 * 32 * 8          # candidates + positions, 8 B per token
    assert L.entmaxkv_full_workspace_size(8, 30, 8, 128, 32, 4096) == 0
    small = L.entmaxkv_workspace_size(1, 8, 8, 64, 16, 64, 64)      # 1024 tokens: no buffers
    assert small < 8 * 64 * 16 * 8 + L.entmaxkv_workspace_size(1, 8, 8, 64, 16, 64, 63)


def _kv(**over):
    from sparse_long_context_08_b300.entmaxkv import _PagedKV
    f = dict(k_pool=16, v_pool=16, dtype=1, num_blocks=4, num_kv_heads=1, page_size=16,
             head_dim=128, page_table=16, max_pages=4, seq_lens=16, batch=1)
    f.update(over)
    return _PagedKV(**f)


def test_invalid_arguments_are_rejected_before_any_launch(L):
    lib = L.lib()
    kv = _kv()
    ref = C.byref(kv)
    nz = C.c_void_p(16)
    # null cache
    assert lib.entmaxkv_decode(nz, 1, 1.0, None, nz, nz, 4, 1.5, nz, None, None, C.c_void_p(256),
                               1 << 20, None) == L.EKV_INVALID_ARG
    # alpha <= 1
    assert lib.entmaxkv_decode(nz, 1, 1.0, ref, nz, nz, 4, 1.0, nz, None, None, C.c_void_p(256),
                               1 << 20, None) == L.EKV_INVALID_ARG
    # scale <= 0
    assert lib.entmaxkv_decode(nz, 1, 0.0, ref, nz, nz, 4, 1.5, nz, None, None, C.c_void_p(256),
                               1 << 20, None) == L.EKV_INVALID_ARG
    # workspace too small / misaligned
    assert lib.entmaxkv_decode(nz, 1, 1.0, ref, nz, nz, 4, 1.5, nz, None, None, C.c_void_p(256),
                               16, None) == L.EKV_WORKSPACE_TOO_SMALL
    assert lib.entmaxkv_decode(nz, 1, 1.0, ref, nz, nz, 4, 1.5, nz, None, None, C.c_void_p(272),
                               1 << 20, None) == L.EKV_INVALID_ARG
    # unsupported head_dim / page size / group
    assert lib.entmaxkv_decode(nz, 1, 1.0, C.byref(_kv(head_dim=96)), nz, nz, 4, 1.5, nz, None,
                               None, C.c_void_p(256), 1 << 20, None) == L.EKV_UNSUPPORTED
    assert lib.entmaxkv_decode(nz, 1, 1.0, C.byref(_kv(page_size=8)), nz, nz, 4, 1.5, nz, None,
                               None, C.c_void_p(256), 1 << 20, None) == L.EKV_UNSUPPORTED
    assert lib.entmaxkv_decode(nz, 3, 1.0, ref, nz, nz, 4, 1.5, nz, None, None, C.c_void_p(256),
                               1 << 20, None) == L.EKV_UNSUPPORTED
    # misaligned pool
    assert lib.entmaxkv_decode(nz, 1, 1.0, C.byref(_kv(k_pool=18)), nz, nz, 4, 1.5, nz, None,
                               None, C.c_void_p(256), 1 << 20, None) == L.EKV_INVALID_ARG
    # select: bad policy, budget below a page, gauss with alpha outside {1.5, 2}
    assert lib.entmaxkv_select(nz, ref, 1, 7, 64, 1.5, 0.1, nz, nz, None, None, 0,
                               None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_select(nz, ref, 1, 0, 8, 1.5, 0.1, nz, nz, None, None, 0,
                               None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_select(nz, ref, 1, 1, 64, 1.7, 0.1, nz, nz, None, None, 0,
                               None) == L.EKV_UNSUPPORTED
    # score: missing metadata for the policy
    from sparse_long_context_08_b300.entmaxkv import _PageMeta
    empty = _PageMeta(None, None, None, None)
    assert lib.entmaxkv_score_pages(nz, 1, 1.0, ref, C.byref(empty), 0, nz,
                                    None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_score_pages(nz, 1, 1.0, ref, C.byref(empty), 1, nz,
                                    None) == L.EKV_INVALID_ARG
    # build: nothing requested
    assert lib.entmaxkv_build_page_meta(ref, 0, 4, C.byref(empty), 0, 0,
                                        None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_read_device_status(None, None) == L.EKV_INVALID_ARG
    # wait self-check: the limit must be 1 .. 100000 us
    assert lib.entmaxkv_check_wait_timeout(0, None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_check_wait_timeout(100001, None) == L.EKV_INVALID_ARG
    # full-cache decode: same checks as decode, no selection
    assert lib.entmaxkv_decode_full(nz, 1, 1.0, None, 1.5, nz, None, None, C.c_void_p(256),
                                    1 << 30, None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_decode_full(nz, 1, 1.0, ref, 1.0, nz, None, None, C.c_void_p(256),
                                    1 << 30, None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_decode_full(nz, 1, 1.0, ref, 1.5, nz, None, None, C.c_void_p(272),
                                    1 << 30, None) == L.EKV_INVALID_ARG
    assert lib.entmaxkv_decode_full(nz, 1, 1.0, ref, 1.5, nz, None, None, C.c_void_p(256),
                                    16, None) == L.EKV_WORKSPACE_TOO_SMALL
    assert lib.entmaxkv_decode_full(nz, 3, 1.0, ref, 1.5, nz, None, None, C.c_void_p(256),
                                    1 << 30, None) == L.EKV_UNSUPPORTED      # group of 3


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    from sparse_long_context_08_b300 import entmaxkv
    monkeypatch.setattr(entmaxkv, "_lib", None)
    monkeypatch.setattr(entmaxkv, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        entmaxkv.lib()
