"""CPU oracle for query-aware sparse paged decode -- TEST INFRASTRUCTURE ONLY.

A Python front end (argument marshalling) over ``qskv_oracle.c``, a plain
double-precision C statement of the method.  Only ``tests/``, the package
smoke check and the benchmark's CPU-baseline leg may import this package; the
CUDA library and its Python binding never do.

Every function states the passage it follows:
  TinyServe query-aware page selection article -- s2.1 metadata (per-page
  element-wise min/max of the keys), s2.2 bound score, s2.3 top-K pages and
  attention over only those pages;
  CS336 Lecture 10 "Inference" -- s2.3 decode attention, s9.2 PagedAttention
  block tables and shared prefixes;
  Quail AI-SQL engine article -- partial attention merged by log-sum-exp;
  Vortex sparse-attention digest, method overview item 1 -- per-block mean
  keys ("centroids") from the cache phase, Block Top-K scoring q . centroid;
  item 3 -- a lossy radix Top-K with early exit and random sampling from the
  threshold bin (its random numbers from SplitMix64, Steele, Lea and Flood 2014).
"""

from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qskv_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libqskv_oracle.so")
_lib = None

F32, BF16 = 0, 1

_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (OpenMP over rows)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        cc = os.environ.get("CC", "gcc")
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.orc_meta.restype = ctypes.c_int
        lib.orc_meta.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, _i32p, _i32p, ctypes.c_int64, _f64p]
        lib.orc_bound.restype = ctypes.c_double
        lib.orc_bound.argtypes = [_f64p, _f64p, _f64p, ctypes.c_int]
        lib.orc_row_scores.restype = ctypes.c_int
        lib.orc_row_scores.argtypes = [_f64p, ctypes.c_int, _f64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _i32p, ctypes.c_int, _f64p]
        lib.orc_centroid.restype = ctypes.c_int
        lib.orc_centroid.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, _i32p, _i32p, ctypes.c_int64, _f64p]
        lib.orc_centroid_scores.restype = ctypes.c_int
        lib.orc_centroid_scores.argtypes = [_f64p, ctypes.c_int, _f64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, _i32p, ctypes.c_int, _f64p]
        lib.orc_splitmix64.restype = ctypes.c_uint64
        lib.orc_splitmix64.argtypes = [ctypes.c_uint64, ctypes.c_uint64]
        lib.orc_select_approx.restype = ctypes.c_int
        lib.orc_select_approx.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_uint64, ctypes.c_int64, _i32p]
        lib.orc_select.restype = ctypes.c_int
        lib.orc_select.argtypes = [_f64p, ctypes.c_int, ctypes.c_int, _i32p]
        lib.orc_attend_row.restype = ctypes.c_int
        lib.orc_attend_row.argtypes = [_f64p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       _i32p, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_int, ctypes.c_double,
                                       _f64p, _f64p]
        lib.orc_set_threads.restype = ctypes.c_int
        lib.orc_set_threads.argtypes = [ctypes.c_int]
        lib.orc_step.restype = ctypes.c_int
        lib.orc_step.argtypes = [_f64p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, _f64p, ctypes.c_int,
                                 _i32p, _i32p,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_double, _i32p,
                                 ctypes.c_int, _i32p, _i32p, _f64p, _f64p, _f64p]
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _pool(t: torch.Tensor):
    """Raw pointer + dtype code of a contiguous CPU KV pool (fp32 or bf16)."""
    assert t.device.type == "cpu" and t.is_contiguous()
    if t.dtype == torch.float32:
        return ctypes.c_void_p(t.data_ptr()), F32
    if t.dtype == torch.bfloat16:
        return ctypes.c_void_p(t.data_ptr()), BF16
    raise TypeError(f"unsupported KV dtype {t.dtype}")


def meta(k_pool: torch.Tensor, page_ids, valid_tokens, out: np.ndarray | None = None) -> np.ndarray:
    """TinyServe s2.1: per-(page, KV head) min and max of the valid keys.

    Returns float64 [Npool][Hkv][2][d] (min row, max row); pages not listed
    are NaN (or keep ``out``'s values)."""
    lib = _load()
    n_pool, hkv, P, d = k_pool.shape
    if out is None:
        out = np.full((n_pool, hkv, 2, d), np.nan)
    ids, vt = _i32(page_ids), _i32(valid_tokens)
    ptr, dt = _pool(k_pool)
    rc = lib.orc_meta(ptr, dt, n_pool, hkv, P, d, _p(ids, _i32p), _p(vt, _i32p), len(ids), _p(out, _f64p))
    if rc != 0:
        raise IndexError("oracle meta: page id or valid-token count out of range")
    return out


def bound(q, m, M) -> float:
    """TinyServe s2.2: sum_i q[i] * (q[i] > 0 ? M[i] : m[i]) for one page."""
    q, m, M = _f64(q), _f64(m), _f64(M)
    return _load().orc_bound(_p(q, _f64p), _p(m, _f64p), _p(M, _f64p), len(q))


def row_scores(q_group, meta_arr: np.ndarray, table_row, n_b: int, g: int) -> np.ndarray:
    """TinyServe s2.2-2.3: S(j) = max over the group's heads of the bound, j < n_b."""
    qg = _f64(q_group)
    G, d = qg.shape
    n_pool, hkv = meta_arr.shape[:2]
    tr = _i32(table_row)
    out = np.empty(max(n_b, 1))
    _load().orc_row_scores(_p(qg, _f64p), G, _p(meta_arr, _f64p), n_pool, hkv, g, d, _p(tr, _i32p), n_b,
                           _p(out, _f64p))
    return out[:n_b]


def centroids(k_pool: torch.Tensor, page_ids, valid_tokens, out: np.ndarray | None = None) -> np.ndarray:
    """Vortex item 1 (cache phase): per-(page, KV head) mean of the valid keys.

    Returns float64 [Npool][Hkv][d]; pages not listed are NaN (or keep
    ``out``'s values)."""
    lib = _load()
    n_pool, hkv, P, d = k_pool.shape
    if out is None:
        out = np.full((n_pool, hkv, d), np.nan)
    ids, vt = _i32(page_ids), _i32(valid_tokens)
    ptr, dt = _pool(k_pool)
    rc = lib.orc_centroid(ptr, dt, n_pool, hkv, P, d, _p(ids, _i32p), _p(vt, _i32p), len(ids), _p(out, _f64p))
    if rc != 0:
        raise IndexError("oracle centroids: page id or valid-token count out of range")
    return out


def centroid_row_scores(q_group, cent: np.ndarray, table_row, n_b: int, g: int) -> np.ndarray:
    """Vortex item 1 (indexer phase, Block Top-K): S(j) = max over the group's
    heads of q_h . centroid of page j, j < n_b."""
    qg = _f64(q_group)
    G, d = qg.shape
    n_pool, hkv = cent.shape[:2]
    tr = _i32(table_row)
    out = np.empty(max(n_b, 1))
    _load().orc_centroid_scores(_p(qg, _f64p), G, _p(cent, _f64p), n_pool, hkv, g, d, _p(tr, _i32p), n_b,
                                _p(out, _f64p))
    return out[:n_b]


SCORERS = {"bound": 0, "centroid": 1}


def select(scores, top_k: int) -> tuple[np.ndarray, int]:
    """TinyServe s2.3: top_k pages by score (ties -> lower index), ascending, -1 padded."""
    s = _f64(scores)
    sel = np.empty(max(top_k, 1), dtype=np.int32)
    n = _load().orc_select(_p(s, _f64p), len(s), top_k, _p(sel, _i32p))
    return sel[:top_k], n


def splitmix64(seed: int, i: int) -> int:
    """Output i of SplitMix64 started at `seed` (Steele, Lea and Flood 2014)."""
    return int(_load().orc_splitmix64(seed & (2 ** 64 - 1), i & (2 ** 64 - 1)))


def need_max(top_k: int, epsilon: float) -> int:
    """Early-exit threshold of the approximate top-K: floor(epsilon * K), the
    product taken as one IEEE double multiplication (epsilon is a double)."""
    return int(math.floor(float(epsilon) * float(top_k)))


def select_approx(scores_f32, top_k: int, epsilon: float, seed: int, row: int) -> tuple[np.ndarray, int]:
    """Vortex item 3: lossy radix top-K over fp32 scores -- exact radix passes
    over the key's four 8-bit digits (most significant first) until at most
    floor(epsilon * K) keys are undecided, then those drawn by systematic
    random sampling from the threshold bin.  epsilon = 0 is the exact rule.
    Returns (ascending indices, -1 padded to top_k; count)."""
    s = np.ascontiguousarray(scores_f32, dtype=np.float32)
    sel = np.empty(max(top_k, 1), dtype=np.int32)
    n = _load().orc_select_approx(s.ctypes.data_as(ctypes.POINTER(ctypes.c_float)), len(s), top_k,
                                  need_max(top_k, epsilon), seed & (2 ** 64 - 1), row, _p(sel, _i32p))
    return sel[:top_k], n


def attend_row(inputs: dict, b: int, g: int, pages, sm_scale: float | None = None):
    """CS336 s2.3/s9.2 + TinyServe s2.3: softmax attention of the G heads of
    KV head g of sequence b over the tokens (< seq_len) of the listed logical
    pages.  Returns (out [G][d], lse [G])."""
    spec = inputs["spec"]
    G, d = spec.group, spec.head_dim
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    qg = _f64(inputs["q"][b, g * G:(g + 1) * G])
    kp, dt = _pool(inputs["k_pool"])
    vp, _ = _pool(inputs["v_pool"])
    table_row = _i32(inputs["page_table"][b])
    seq_len = int(inputs["seq_lens"][b])
    n_b = (seq_len + spec.page_size - 1) // spec.page_size
    pl = _i32(pages)
    out = np.zeros((G, d))
    lse = np.zeros(G)
    n_pool = inputs["k_pool"].shape[0]
    rc = _load().orc_attend_row(_p(qg, _f64p), G, kp, vp, dt, n_pool, spec.num_kv_heads, g, spec.page_size, d,
                                _p(table_row, _i32p), n_b, seq_len, _p(pl, _i32p), len(pl), sm_scale,
                                _p(out, _f64p), _p(lse, _f64p))
    if rc < 0:
        raise IndexError("oracle attend: page index out of range")
    return out, lse


def step(inputs: dict, rows=None, top_k: int | None = "spec", meta_arr: np.ndarray | None = None,
         sm_scale: float | None = None, q=None, threads: int | None = None, scorer: str = "bound") -> dict:
    """One full decode step (scores -> top-K -> attention) over ``rows``
    (row = b * Hkv + g; default all).  ``top_k=None`` (or a dense spec) means
    every page.  ``scorer`` is "bound" (TinyServe s2.2, meta_arr = min/max
    rows) or "centroid" (Vortex Block Top-K, meta_arr = centroids).  Returns
    numpy arrays keyed selected, n_sel, scores, out, lse, plus the OpenMP
    thread count used."""
    spec = inputs["spec"]
    if isinstance(top_k, str):
        top_k = spec.top_k
    B, Hq, Hkv, d, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    G = spec.group
    max_pages = inputs["page_table"].shape[1]
    n_pool = inputs["k_pool"].shape[0]
    if rows is None:
        rows = np.arange(B * Hkv, dtype=np.int32)
    rows = _i32(rows)
    n_rows = len(rows)
    dense = top_k is None or top_k <= 0
    if not dense and meta_arr is None:
        ids, vt = _all_pages(inputs)
        meta_arr = (centroids if scorer == "centroid" else meta)(inputs["k_pool"], ids, vt)
    if sm_scale is None:
        sm_scale = 1.0 / math.sqrt(d)
    qd = _f64(inputs["q"] if q is None else q)
    kp, dt = _pool(inputs["k_pool"])
    vp, _ = _pool(inputs["v_pool"])
    table = _i32(inputs["page_table"])
    sl = _i32(inputs["seq_lens"])
    kk = 0 if dense else int(top_k)
    selected = np.full((n_rows, max(kk, 1)), -1, dtype=np.int32)
    n_sel = np.zeros(n_rows, dtype=np.int32)
    scores = None if dense else np.empty((n_rows, max_pages))
    out = np.zeros((n_rows, G, d))
    lse = np.zeros((n_rows, G))
    meta_p = _p(meta_arr, _f64p) if meta_arr is not None else _p(np.zeros(1), _f64p)
    lib = _load()
    if threads is not None:
        lib.orc_set_threads(int(threads))
    nthr = lib.orc_step(_p(qd, _f64p), kp, vp, dt, meta_p, SCORERS[scorer], _p(table, _i32p), _p(sl, _i32p), B,
                        Hq, Hkv, d, P,
                        max_pages, n_pool, kk, sm_scale, _p(rows, _i32p), n_rows, _p(selected, _i32p),
                        _p(n_sel, _i32p), _p(scores, _f64p) if scores is not None else None, _p(out, _f64p),
                        _p(lse, _f64p))
    if nthr < 0:
        raise IndexError("oracle step: an index was out of range")
    return dict(selected=selected[:, :kk] if not dense else None, n_sel=n_sel, scores=scores, out=out, lse=lse,
                rows=rows, threads=nthr, meta=meta_arr)


def _all_pages(inputs: dict):
    P = inputs["spec"].page_size
    table = inputs["page_table"].numpy()
    sl = inputs["seq_lens"].numpy().astype(np.int64)
    nb = (sl + P - 1) // P
    ids, valid = [], []
    seen = {}
    for b in range(table.shape[0]):
        for j in range(int(nb[b])):
            p = int(table[b, j])
            v = int(min(P, sl[b] - j * P))
            if p not in seen:
                seen[p] = v
    ids = np.array(sorted(seen), dtype=np.int32)
    valid = np.array([seen[int(p)] for p in ids], dtype=np.int32)
    return ids, valid


def all_pages(inputs: dict):
    """(physical ids, valid-token counts) of every referenced pool page."""
    return _all_pages(inputs)
