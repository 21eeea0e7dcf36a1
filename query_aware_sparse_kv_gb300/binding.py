"""ctypes binding of libqskv.so (include/qskv.h).

Argument marshalling only: every function here turns torch tensors into the
raw pointers, sizes and the current CUDA stream the C ABI takes, calls it,
and raises on a non-OK status.  All arithmetic runs in the library's CUDA
kernels; there is no CPU fallback.  If the library has not been built, the
first call raises ``QskvLibraryMissing``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqskv.so")

QSKV_F32, QSKV_BF16 = 0, 1
STATUS = {0: "QSKV_OK", 1: "QSKV_ERR_INVALID_ARG", 2: "QSKV_ERR_UNSUPPORTED", 3: "QSKV_ERR_WORKSPACE",
          4: "QSKV_ERR_CUDA", 5: "QSKV_ERR_DEVICE_INDEX", 6: "QSKV_ERR_DEVICE_TIMEOUT"}

# Every function the header declares, in declaration order.
EXPORTS = ("qskv_workspace_size", "qskv_kv_meta_build", "qskv_page_select", "qskv_page_select_refresh",
           "qskv_kv_centroid_build", "qskv_page_select_centroid", "qskv_page_select_approx",
           "qskv_sparse_paged_decode", "qskv_select_decode", "qskv_sparse_paged_decode_noalloc",
           "qskv_cascade_workspace_size", "qskv_cascade_paged_decode", "qskv_get_error", "qskv_status_string",
           "qskv_last_error_message")


class QskvLibraryMissing(RuntimeError):
    pass


class QskvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_pages", ctypes.c_int32),
                ("num_pool_pages", ctypes.c_int32)]

    def __repr__(self):
        return "Shape(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


_lib = None


def load(path: str = LIB_PATH):
    """Load libqskv.so once and declare its prototypes."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise QskvLibraryMissing(f"{path} is missing: build it with query_aware_sparse_kv_gb300.build.build()")
    lib = ctypes.CDLL(path)
    vp, i32p, f32p, sz, i32 = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
    sp = ctypes.POINTER(Shape)
    lib.qskv_workspace_size.restype = sz
    lib.qskv_workspace_size.argtypes = [sp]
    lib.qskv_kv_meta_build.restype = ctypes.c_int
    lib.qskv_kv_meta_build.argtypes = [vp, ctypes.c_int, sp, i32p, i32p, i32, vp, vp, sz, vp]
    lib.qskv_page_select.restype = ctypes.c_int
    lib.qskv_page_select.argtypes = [vp, ctypes.c_int, vp, ctypes.c_int, i32p, i32p, sp, i32, i32p, i32p, f32p, vp,
                                     sz, vp]
    lib.qskv_page_select_refresh.restype = ctypes.c_int
    lib.qskv_page_select_refresh.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, i32p, i32p, sp, i32, i32p, i32p,
                                             f32p, vp, sz, vp]
    lib.qskv_kv_centroid_build.restype = ctypes.c_int
    lib.qskv_kv_centroid_build.argtypes = [vp, ctypes.c_int, sp, i32p, i32p, i32, f32p, vp, sz, vp]
    lib.qskv_page_select_centroid.restype = ctypes.c_int
    lib.qskv_page_select_centroid.argtypes = [vp, ctypes.c_int, f32p, i32p, i32p, sp, i32, i32p, i32p, f32p, vp,
                                              sz, vp]
    lib.qskv_page_select_approx.restype = ctypes.c_int
    lib.qskv_page_select_approx.argtypes = [ctypes.c_int, vp, ctypes.c_int, vp, ctypes.c_int, i32p, i32p, sp, i32,
                                            ctypes.c_double, ctypes.c_uint64, i32p, i32p, f32p, vp, sz, vp]
    lib.qskv_sparse_paged_decode.restype = ctypes.c_int
    lib.qskv_sparse_paged_decode.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, i32p, i32p, sp, i32p, i32p, i32,
                                             ctypes.c_float, f32p, f32p, vp, sz, vp]
    lib.qskv_select_decode.restype = ctypes.c_int
    lib.qskv_select_decode.argtypes = [vp, ctypes.c_int, vp, vp, vp, ctypes.c_int, i32p, i32p, sp, i32, ctypes.c_float,
                                       i32p, i32p, f32p, f32p, f32p, vp, sz, vp]
    lib.qskv_sparse_paged_decode_noalloc.restype = ctypes.c_int
    lib.qskv_sparse_paged_decode_noalloc.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, i32p, i32p, sp, i32p,
                                                     i32p, i32, ctypes.c_float, f32p, f32p, vp]
    lib.qskv_cascade_workspace_size.restype = sz
    lib.qskv_cascade_workspace_size.argtypes = [sp, i32]
    lib.qskv_cascade_paged_decode.restype = ctypes.c_int
    lib.qskv_cascade_paged_decode.argtypes = [vp, ctypes.c_int, vp, vp, ctypes.c_int, i32p, i32p, sp, i32,
                                              ctypes.c_float, f32p, f32p, vp, sz, vp]
    lib.qskv_get_error.restype = ctypes.c_int
    lib.qskv_get_error.argtypes = [vp, vp]
    lib.qskv_status_string.restype = ctypes.c_char_p
    lib.qskv_status_string.argtypes = [ctypes.c_int]
    lib.qskv_last_error_message.restype = ctypes.c_char_p
    lib.qskv_last_error_message.argtypes = []
    _lib = lib
    return lib


def _check(status: int):
    if status != 0:
        raise QskvError(status, load().qskv_last_error_message().decode())


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return QSKV_F32
    if t.dtype == torch.bfloat16:
        return QSKV_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (fp32 or bf16)")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_shape(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages, num_pool_pages) -> Shape:
    return Shape(int(batch), int(num_q_heads), int(num_kv_heads), int(head_dim), int(page_size), int(max_pages),
                 int(num_pool_pages))


def workspace_size(shape: Shape) -> int:
    n = load().qskv_workspace_size(ctypes.byref(shape))
    if n == 0:
        raise QskvError(1, load().qskv_last_error_message().decode())
    return int(n)


def kv_meta_build(k_pool: torch.Tensor, page_ids: torch.Tensor, valid_tokens: torch.Tensor, meta: torch.Tensor,
                  shape: Shape, workspace: torch.Tensor, stream=None):
    _check(load().qskv_kv_meta_build(_ptr(k_pool), _dtype(k_pool), ctypes.byref(shape), _ptr(page_ids),
                                     _ptr(valid_tokens), int(page_ids.numel()), _ptr(meta), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))


def page_select(q: torch.Tensor, meta: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor, top_k: int,
                selected: torch.Tensor, n_selected: torch.Tensor, shape: Shape, workspace: torch.Tensor,
                scores: Optional[torch.Tensor] = None, stream=None):
    _check(load().qskv_page_select(_ptr(q), _dtype(q), _ptr(meta), _dtype(meta), _ptr(page_table), _ptr(seq_lens),
                                   ctypes.byref(shape), int(top_k), _ptr(selected), _ptr(n_selected), _ptr(scores),
                                   _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def page_select_refresh(q: torch.Tensor, k_pool: torch.Tensor, meta: torch.Tensor, page_table: torch.Tensor,
                        seq_lens: torch.Tensor, top_k: int, selected: torch.Tensor, n_selected: torch.Tensor,
                        shape: Shape, workspace: torch.Tensor, scores: Optional[torch.Tensor] = None, stream=None):
    """The last page of every sequence gets its metadata rebuilt from k_pool,
    then the selection runs (one launch less than kv_meta_build + page_select)."""
    _check(load().qskv_page_select_refresh(_ptr(q), _dtype(q), _ptr(k_pool), _ptr(meta), _dtype(k_pool),
                                           _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape), int(top_k),
                                           _ptr(selected), _ptr(n_selected), _ptr(scores), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream(stream)))


def select_decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, meta: torch.Tensor,
                  page_table: torch.Tensor, seq_lens: torch.Tensor, top_k: int, selected: torch.Tensor,
                  n_selected: torch.Tensor, out: torch.Tensor, shape: Shape, workspace: torch.Tensor,
                  lse: Optional[torch.Tensor] = None, scores: Optional[torch.Tensor] = None, sm_scale: float = 0.0,
                  stream=None):
    """One decode step: last-page metadata refresh, bound scores, exact top-K
    and the sparse decode (one to three launches by shape, see
    qskv_select_decode in include/qskv.h)."""
    _check(load().qskv_select_decode(_ptr(q), _dtype(q), _ptr(k_pool), _ptr(v_pool), _ptr(meta), _dtype(k_pool),
                                     _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape), int(top_k),
                                     float(sm_scale), _ptr(selected), _ptr(n_selected), _ptr(scores), _ptr(out),
                                     _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def kv_centroid_build(k_pool: torch.Tensor, page_ids: torch.Tensor, valid_tokens: torch.Tensor,
                      centroids: torch.Tensor, shape: Shape, workspace: torch.Tensor, stream=None):
    """Per-(page, KV head) mean of the valid keys into fp32 ``centroids``
    [Npool][Hkv][d] (the Block Top-K summary)."""
    if centroids.dtype != torch.float32:
        raise TypeError("centroids must be float32")
    _check(load().qskv_kv_centroid_build(_ptr(k_pool), _dtype(k_pool), ctypes.byref(shape), _ptr(page_ids),
                                         _ptr(valid_tokens), int(page_ids.numel()), _ptr(centroids),
                                         _ptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def page_select_centroid(q: torch.Tensor, centroids: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                         top_k: int, selected: torch.Tensor, n_selected: torch.Tensor, shape: Shape,
                         workspace: torch.Tensor, scores: Optional[torch.Tensor] = None, stream=None):
    """Block Top-K selection: score q . centroid per page, keep the top_k."""
    if centroids.dtype != torch.float32:
        raise TypeError("centroids must be float32")
    _check(load().qskv_page_select_centroid(_ptr(q), _dtype(q), _ptr(centroids), _ptr(page_table), _ptr(seq_lens),
                                            ctypes.byref(shape), int(top_k), _ptr(selected), _ptr(n_selected),
                                            _ptr(scores), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)))


SCORERS = {"bound": 0, "centroid": 1}


def page_select_approx(q: torch.Tensor, meta: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                       top_k: int, selected: torch.Tensor, n_selected: torch.Tensor, shape: Shape,
                       workspace: torch.Tensor, epsilon: float, seed: int, scorer: str = "bound",
                       scores: Optional[torch.Tensor] = None, stream=None):
    """Selection with the lossy top-K: radix passes until at most
    floor(epsilon * top_k) pages are undecided, the rest sampled from the
    threshold bucket (random start from SplitMix64(seed))."""
    _check(load().qskv_page_select_approx(SCORERS[scorer], _ptr(q), _dtype(q), _ptr(meta), _dtype(meta),
                                          _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape), int(top_k),
                                          float(epsilon), int(seed) & (2 ** 64 - 1), _ptr(selected),
                                          _ptr(n_selected), _ptr(scores), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def sparse_paged_decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor,
                        seq_lens: torch.Tensor, out: torch.Tensor, shape: Shape, workspace: torch.Tensor,
                        selected: Optional[torch.Tensor] = None, n_selected: Optional[torch.Tensor] = None,
                        top_k: int = 0, lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0, stream=None):
    _check(load().qskv_sparse_paged_decode(_ptr(q), _dtype(q), _ptr(k_pool), _ptr(v_pool), _dtype(k_pool),
                                           _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape), _ptr(selected),
                                           _ptr(n_selected), int(top_k), float(sm_scale), _ptr(out), _ptr(lse),
                                           _ptr(workspace), workspace.numel() * workspace.element_size(),
                                           _stream(stream)))


def sparse_paged_decode_noalloc(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                                page_table: torch.Tensor, seq_lens: torch.Tensor, out: torch.Tensor, shape: Shape,
                                selected: Optional[torch.Tensor] = None, n_selected: Optional[torch.Tensor] = None,
                                top_k: int = 0, lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0,
                                stream=None):
    """sparse_paged_decode for callers that cannot allocate device memory
    (their memory planner owns all of HBM, or their decode loop must not
    call the allocator).  The library's built-in 8 MiB scratch replaces the
    workspace; this wrapper allocates nothing either.  Calls that may overlap
    on the GPU share that scratch and race."""
    _check(load().qskv_sparse_paged_decode_noalloc(_ptr(q), _dtype(q), _ptr(k_pool), _ptr(v_pool), _dtype(k_pool),
                                                   _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape),
                                                   _ptr(selected), _ptr(n_selected), int(top_k), float(sm_scale),
                                                   _ptr(out), _ptr(lse), _stream(stream)))


def cascade_workspace_size(shape: Shape, prefix_pages: int) -> int:
    n = load().qskv_cascade_workspace_size(ctypes.byref(shape), int(prefix_pages))
    if n == 0:
        raise QskvError(1, load().qskv_last_error_message().decode())
    return int(n)


def cascade_paged_decode(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, page_table: torch.Tensor,
                         seq_lens: torch.Tensor, out: torch.Tensor, shape: Shape, workspace: torch.Tensor,
                         prefix_pages: int, lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0, stream=None):
    """Dense decode of a batch whose rows share their first `prefix_pages`
    pages (the workspace must hold cascade_workspace_size bytes)."""
    _check(load().qskv_cascade_paged_decode(_ptr(q), _dtype(q), _ptr(k_pool), _ptr(v_pool), _dtype(k_pool),
                                            _ptr(page_table), _ptr(seq_lens), ctypes.byref(shape), int(prefix_pages),
                                            float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)))


def get_error(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise, read and clear the device error flags; returns the status."""
    return int(load().qskv_get_error(_ptr(workspace), _stream(stream)))


def last_error_message() -> str:
    return load().qskv_last_error_message().decode()
