"""Query-aware sparse paged KV decode for GB300 (sm_103a).

The computation lives in libqskv.so (CUDA kernels behind the C ABI declared
in include/qskv.h); this package is its binding:

  kv_meta_build        per-page min/max key metadata
  page_select          bound score of every page and top-K per (sequence, KV head)
  page_select_refresh  the same, after rebuilding every sequence's last-page
                       metadata in the same launch
  kv_centroid_build,   Block Top-K: per-page mean key, and q . centroid scores
  page_select_centroid   with the same top-K
  page_select_approx   either score with a lossy top-K (early exit + sampling)
  sparse_paged_decode  split-K attention over the selected pages, LSE merge
  select_decode        one step in one call: last-page refresh, scoring,
                       top-K and the sparse decode (the decode ranks its
                       own rows when they go one row per k CTAs)
  cascade_paged_decode dense decode of a batch sharing a page prefix: the
                       prefix once per KV head on the tensor cores, the rest
                       paged, LSE merge

plus ``PagedDecoder`` (buffer plumbing for a whole step) and ``workloads``
(seeded synthetic inputs).  Nothing here computes on the CPU: without the
built library every call raises.
"""
from .binding import (QSKV_BF16, QSKV_F32, QskvError, QskvLibraryMissing, Shape, cascade_paged_decode,
                      cascade_workspace_size, get_error, kv_centroid_build, kv_meta_build, last_error_message, load,
                      make_shape, page_select, page_select_approx, page_select_refresh, page_select_centroid,
                      select_decode, sparse_paged_decode, sparse_paged_decode_noalloc, workspace_size)
from .engine import PagedDecoder, from_inputs

__all__ = ["QSKV_BF16", "QSKV_F32", "QskvError", "QskvLibraryMissing", "Shape", "cascade_paged_decode",
           "cascade_workspace_size", "get_error", "kv_centroid_build", "kv_meta_build", "page_select_approx", "page_select_centroid",
           "last_error_message", "load", "make_shape", "page_select", "page_select_refresh", "select_decode",
           "sparse_paged_decode",
           "sparse_paged_decode_noalloc", "workspace_size",
           "PagedDecoder", "from_inputs"]
