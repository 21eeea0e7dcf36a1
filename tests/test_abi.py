"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/qskv.h declares, and rejects bad arguments
on the host before any launch."""
import ctypes
import os
import re

import pytest

import query_aware_sparse_kv_gb300 as qskv
from query_aware_sparse_kv_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return qskv.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "qskv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qskv_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = _declared()
    for n in ("qskv_kv_meta_build", "qskv_page_select", "qskv_sparse_paged_decode", "qskv_cascade_paged_decode"):
        assert n in names
    assert sorted(binding.EXPORTS) == names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert lib.qskv_status_string(code).decode() == name


def test_shape_checks_fail_before_any_launch(lib):
    ws = ctypes.create_string_buffer(4096 + 256)
    wsp = ctypes.c_void_p((ctypes.addressof(ws) + 255) // 256 * 256)
    bad = [
        (qskv.make_shape(2, 6, 4, 128, 16, 8, 16), 1),  # Hq not a multiple of Hkv
        (qskv.make_shape(2, 48, 4, 128, 16, 8, 16), 2),  # G = 12
        (qskv.make_shape(2, 8, 2, 96, 16, 8, 16), 2),  # head_dim 96
        (qskv.make_shape(2, 8, 2, 128, 8, 8, 16), 2),  # page_size 8
        (qskv.make_shape(0, 8, 2, 128, 16, 8, 16), 1),  # empty batch
    ]
    for shape, want in bad:
        st = lib.qskv_page_select(None, 1, None, 1, None, None, ctypes.byref(shape), 4, None, None, None, wsp, 4096,
                                  None)
        assert st == want, (shape, st, lib.qskv_last_error_message())
        assert lib.qskv_last_error_message().decode()
        st = lib.qskv_sparse_paged_decode(None, 1, None, None, 1, None, None, ctypes.byref(shape), None, None, 0, 0.0,
                                          None, None, wsp, 4096, None)
        assert st == want
        assert lib.qskv_workspace_size(ctypes.byref(shape)) == 0


def test_argument_checks(lib):
    shape = qskv.make_shape(2, 8, 2, 128, 16, 8, 16)
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    # NULL pointers
    st = lib.qskv_page_select(None, 1, p, 1, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None)
    assert st == 1
    # top_k < 1
    st = lib.qskv_page_select(p, 1, p, 1, p, p, ctypes.byref(shape), 0, p, p, None, p, 4096, None)
    assert st == 1
    # misaligned q
    st = lib.qskv_page_select(ctypes.c_void_p(base + 4), 1, p, 1, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096,
                              None)
    assert st == 1
    # bad dtype
    st = lib.qskv_sparse_paged_decode(p, 7, p, p, 1, p, p, ctypes.byref(shape), None, None, 0, 0.0, p, None, p, 4096,
                                      None)
    assert st == 2
    # selected without n_selected
    st = lib.qskv_sparse_paged_decode(p, 1, p, p, 1, p, p, ctypes.byref(shape), p, None, 4, 0.0, p, None, p, 4096,
                                      None)
    assert st == 1
    # negative scale
    st = lib.qskv_sparse_paged_decode(p, 1, p, p, 1, p, p, ctypes.byref(shape), None, None, 0, -1.0, p, None, p, 4096,
                                      None)
    assert st == 1
    # meta build: negative count, misaligned workspace, n_pages == 0 is a no-op
    assert lib.qskv_kv_meta_build(p, 1, ctypes.byref(shape), p, p, -1, p, p, 4096, None) == 1
    assert lib.qskv_kv_meta_build(p, 1, ctypes.byref(shape), p, p, 1, p, ctypes.c_void_p(base + 8), 4096, None) == 3
    assert lib.qskv_kv_meta_build(p, 1, ctypes.byref(shape), p, p, 0, p, p, 4096, None) == 0


def test_refresh_select_argument_checks(lib):
    """The fused refresh + selection rejects what it cannot do before any launch."""
    shape = qskv.make_shape(2, 8, 2, 128, 16, 8, 16)
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    f = lib.qskv_page_select_refresh
    assert f(p, 1, p, p, 0, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) == 2  # fp32 KV
    assert f(p, 1, None, p, 1, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) == 1  # no k_pool
    assert f(p, 1, p, p, 1, p, p, ctypes.byref(shape), 0, p, p, None, p, 4096, None) == 1  # top_k 0
    assert f(p, 1, ctypes.c_void_p(base + 8), p, 1, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) == 1
    assert "bf16" in (f(p, 1, p, p, 0, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) and
                      lib.qskv_last_error_message().decode())


def test_cascade_argument_checks(lib):
    shape = qskv.make_shape(2, 8, 2, 128, 16, 8, 16)
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)

    def call(q=p, kv_dtype=1, prefix=4, out=p, scale=0.0, shp=shape):
        return lib.qskv_cascade_paged_decode(q, 1, p, p, kv_dtype, p, p, ctypes.byref(shp), prefix, scale, out, None,
                                             p, 4096, None)

    assert call(kv_dtype=0) == 2          # fp32 KV cache
    assert call(q=None) == 1              # NULL query
    assert call(prefix=-1) == 1           # prefix outside [0, max_pages]
    assert call(prefix=9) == 1
    assert call(out=ctypes.c_void_p(base + 4)) == 1  # misaligned output
    assert call(scale=-2.0) == 1
    assert call(shp=qskv.make_shape(2, 8, 2, 96, 16, 8, 16)) == 2  # head_dim 96
    assert lib.qskv_last_error_message().decode()
    assert lib.qskv_cascade_workspace_size(ctypes.byref(shape), -1) == 0
    assert lib.qskv_cascade_workspace_size(ctypes.byref(shape), 9) == 0


def test_centroid_argument_checks(lib):
    shape = qskv.make_shape(2, 8, 2, 128, 16, 8, 16)
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)
    # centroid build: negative count, NULL output, misaligned centroids, empty list is a no-op
    assert lib.qskv_kv_centroid_build(p, 1, ctypes.byref(shape), p, p, -1, p, p, 4096, None) == 1
    assert lib.qskv_kv_centroid_build(p, 1, ctypes.byref(shape), p, p, 2, None, p, 4096, None) == 1
    assert lib.qskv_kv_centroid_build(p, 1, ctypes.byref(shape), p, p, 2, ctypes.c_void_p(base + 8), p, 4096,
                                      None) == 1
    assert lib.qskv_kv_centroid_build(p, 1, ctypes.byref(shape), p, p, 0, p, p, 4096, None) == 0
    # selection: top_k < 1, NULL centroids, bad q dtype
    assert lib.qskv_page_select_centroid(p, 1, p, p, p, ctypes.byref(shape), 0, p, p, None, p, 4096, None) == 1
    assert lib.qskv_page_select_centroid(p, 1, None, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) == 1
    assert lib.qskv_page_select_centroid(p, 9, p, p, p, ctypes.byref(shape), 4, p, p, None, p, 4096, None) == 2


def test_binding_fails_loudly_without_the_library(tmp_path):
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(binding.QskvLibraryMissing):
            binding.load(str(tmp_path / "missing.so"))
    finally:
        binding._lib = saved


def test_select_decode_argument_checks(lib):
    """The one-call step rejects what it cannot do before any launch."""
    shape = qskv.make_shape(2, 8, 2, 128, 16, 8, 16)
    buf = ctypes.create_string_buffer(1 << 16)
    base = (ctypes.addressof(buf) + 255) // 256 * 256
    p = ctypes.c_void_p(base)

    def call(q=p, kv_dtype=1, k_pool=p, top_k=4, scale=0.0, out=p, lse=None, shp=shape):
        return lib.qskv_select_decode(q, 1, k_pool, p, p, kv_dtype, p, p, ctypes.byref(shp), top_k, scale, p, p, None,
                                      out, lse, p, 4096, None)

    assert call(kv_dtype=0) == 2                     # fp32 KV: the separate calls serve it
    assert "bf16" in lib.qskv_last_error_message().decode()
    assert call(k_pool=None) == 1                    # NULL K pool
    assert call(top_k=0) == 1
    assert call(scale=-1.0) == 1
    assert call(out=ctypes.c_void_p(base + 4)) == 1  # misaligned output
    assert call(lse=ctypes.c_void_p(base + 2)) == 1  # misaligned lse
    assert call(q=ctypes.c_void_p(base + 8)) == 1    # misaligned query
    assert call(shp=qskv.make_shape(2, 8, 2, 96, 16, 8, 16)) == 2  # head_dim 96
