"""Parity rules between the CUDA path and the CPU oracle (shared by the GPU
tests, the package smoke check and the benchmark's sampled checks).

* metadata: bit-exact, with -0 and +0 treated as equal;
* selection: same size min(top_k, n_b); every page in the symmetric
  difference of the GPU and oracle sets has an oracle score within
  1e-3 * max(|S_K|, 1) of the oracle's K-th score S_K (tie band);
* output: the GPU output against oracle attention over the GPU's own
  selection, max-abs <= 1e-4 for fp32 KV and 1e-2 for bf16 KV (lse too).
"""
from __future__ import annotations

import math

import numpy as np
import torch

TIE_BAND = 1e-3


def out_tolerance(kv_dtype) -> float:
    return 1e-4 if kv_dtype == torch.float32 else 1e-2


def canon(x: np.ndarray) -> np.ndarray:
    x = np.array(x, dtype=np.float64)
    x[x == 0] = 0.0
    return x


def assert_meta_equal(gpu_meta: torch.Tensor, oracle_meta: np.ndarray, pages) -> None:
    g = gpu_meta.detach().cpu().double().numpy()
    pages = np.asarray(pages, dtype=np.int64)
    a, b = canon(g[pages]), canon(oracle_meta[pages])
    bad = np.argwhere(a != b)
    assert bad.size == 0, f"metadata differs at {len(bad)} places, first {bad[:3].tolist()}: {a[tuple(bad[0])]} vs {b[tuple(bad[0])]}"


def assert_scores_close(gpu_scores: np.ndarray, oracle_scores: np.ndarray, n_b: int, what: str = "") -> None:
    g, o = gpu_scores[:n_b].astype(np.float64), oracle_scores[:n_b]
    scale = max(1.0, float(np.abs(o[np.isfinite(o)]).max(initial=0.0)))
    err = np.abs(g - o)
    err[np.isinf(g) & np.isinf(o) & (np.sign(g) == np.sign(o))] = 0.0
    assert err.max(initial=0.0) <= 2e-5 * scale, f"{what} score error {err.max()} (scale {scale})"


def assert_selection_valid(gpu_sel, gpu_n: int, oracle_scores: np.ndarray, n_b: int, top_k: int, what: str = ""):
    """The tie-band rule; also: ascending, unique, in range, -1 padded."""
    n = min(top_k, n_b)
    assert gpu_n == n, f"{what} n_selected {gpu_n} != {n}"
    sel = np.asarray(gpu_sel[:n], dtype=np.int64)
    assert (np.asarray(gpu_sel[n:top_k]) == -1).all(), f"{what} padding is not -1"
    assert (sel >= 0).all() and (sel < n_b).all(), f"{what} selected index out of range"
    assert (np.diff(sel) > 0).all(), f"{what} selection not strictly ascending"
    if top_k >= n_b:
        assert sel.tolist() == list(range(n_b))
        return
    s = oracle_scores[:n_b]
    order = sorted(range(n_b), key=lambda j: (-s[j], j))
    oracle_set = set(order[:n])
    s_k = s[order[n - 1]]
    band = TIE_BAND * max(abs(s_k), 1.0)
    diff = oracle_set.symmetric_difference(sel.tolist())
    for j in diff:
        assert abs(s[j] - s_k) <= band, f"{what} page {j} (score {s[j]}) outside the tie band of S_K={s_k}"


def assert_output_close(gpu_out, gpu_lse, oracle_out, oracle_lse, tol: float, what: str = ""):
    go = np.asarray(gpu_out, dtype=np.float64)
    assert np.isfinite(go).all(), f"{what} non-finite output"
    err = np.abs(go - oracle_out).max(initial=0.0)
    assert err <= tol, f"{what} output max-abs error {err} > {tol}"
    if gpu_lse is not None:
        gl = np.asarray(gpu_lse, dtype=np.float64)
        both_inf = np.isneginf(gl) & np.isneginf(oracle_lse)
        e = np.abs(np.where(both_inf, 0.0, gl - oracle_lse)).max(initial=0.0)
        assert e <= tol, f"{what} lse max-abs error {e} > {tol}"


U32 = 2.0 ** -24  # unit roundoff of fp32


def centroid_tolerance(k_pool: torch.Tensor, pages, valid) -> np.ndarray:
    """Per-element bound of |fp32 centroid - exact mean| for the listed pages:
    a sum of n fp32 values in any order is within (n - 1) u sum|k| of the
    exact sum, and the division adds u |c|, so (sum/n) is within
    n u max|k| of the mean.  Returns [Npool][Hkv][d] (0 for unlisted pages)."""
    kp = k_pool.double().numpy()
    tol = np.zeros((kp.shape[0], kp.shape[1], kp.shape[3]))
    for p, v in zip(np.asarray(pages), np.asarray(valid)):
        tol[p] = int(v) * U32 * np.abs(kp[p, :, :int(v), :]).max(axis=1)
    return tol


def assert_centroids_close(gpu_cent: torch.Tensor, oracle_cent: np.ndarray, tol: np.ndarray, pages) -> None:
    g = gpu_cent.detach().cpu().double().numpy()
    pages = np.asarray(pages, dtype=np.int64)
    err = np.abs(g[pages] - oracle_cent[pages])
    bound = tol[pages] + 1e-30
    worst = np.unravel_index(np.argmax(err / bound), err.shape)
    assert (err <= bound).all(), f"centroid error {err[worst]} > bound {bound[worst]} at {worst}"


def centroid_score_tolerance(q_group: np.ndarray, cent: np.ndarray, cent_tol: np.ndarray, table_row, n_b: int,
                             g: int) -> np.ndarray:
    """Per-page bound of |fp32 score - exact score|: the centroid error
    propagated (sum_i |q_i| tol_i) plus the d-term fp32 dot-product bound
    (d u sum_i |q_i c_i|), the larger over the group's heads."""
    d = q_group.shape[1]
    out = np.zeros(n_b)
    for j in range(n_b):
        p = int(table_row[j])
        c, t = cent[p, g], cent_tol[p, g]
        out[j] = max(float(np.abs(qh) @ t + d * U32 * (np.abs(qh) @ np.abs(c))) for qh in q_group) * 1.01 + 1e-30
    return out


def n_pages_of(inputs: dict, b: int) -> int:
    P = inputs["spec"].page_size
    return (int(inputs["seq_lens"][b]) + P - 1) // P


def check_rows(inputs: dict, dec, rows, oracle, oracle_meta=None, check_scores=None, dense: bool = False,
               sm_scale=None, scorer: str = "bound", cent_tol=None):
    """Compare the decoder's last results on `rows` (b * Hkv + g) with the
    oracle.  `dec` is a PagedDecoder whose select/decode already ran;
    check_scores is the [B][Hkv][max_pages] GPU score tensor or None.  With
    scorer="centroid", oracle_meta holds the oracle's centroids and cent_tol
    their error bounds (centroid_tolerance)."""
    spec = inputs["spec"]
    Hkv, G = spec.num_kv_heads, spec.group
    tol = out_tolerance(spec.kv_dtype)
    out = dec.out.cpu().double().numpy()
    lse = dec.lse.cpu().double().numpy()
    sel = dec.selected.cpu().numpy()
    nsel = dec.n_selected.cpu().numpy()
    q = inputs["q"].double().numpy()
    for r in rows:
        b, g = divmod(int(r), Hkv)
        n_b = n_pages_of(inputs, b)
        what = f"[row b={b} g={g}]"
        if dense or spec.top_k is None:
            pages = list(range(n_b))
        else:
            qg = q[b, g * G:(g + 1) * G]
            if scorer == "centroid":
                o_scores = oracle.centroid_row_scores(qg, oracle_meta, inputs["page_table"][b], n_b, g)
                if check_scores is not None:
                    stol = centroid_score_tolerance(qg, oracle_meta, cent_tol, inputs["page_table"][b], n_b, g)
                    err = np.abs(check_scores[b, g].cpu().double().numpy()[:n_b] - o_scores)
                    assert (err <= stol).all(), f"{what} centroid score error {err.max()} (bound {stol[np.argmax(err)]})"
            else:
                o_scores = oracle.row_scores(qg, oracle_meta, inputs["page_table"][b], n_b, g)
                if check_scores is not None:
                    assert_scores_close(check_scores[b, g].cpu().numpy(), o_scores, n_b, what)
            assert_selection_valid(sel[b, g], int(nsel[b, g]), o_scores, n_b, spec.top_k, what)
            pages = sel[b, g, :int(nsel[b, g])].tolist()
        o_out, o_lse = oracle.attend_row(inputs, b, g, pages, sm_scale=sm_scale)
        assert_output_close(out[b, g * G:(g + 1) * G], lse[b, g * G:(g + 1) * G], o_out, o_lse, tol, what)


def sample_rows(n_rows: int, k: int, seed: int = 0) -> list:
    rng = np.random.default_rng(seed)
    if n_rows <= k:
        return list(range(n_rows))
    pick = set(rng.choice(n_rows, size=k - 2, replace=False).tolist()) | {0, n_rows - 1}
    return sorted(pick)


def inv_sqrt(d: int) -> float:
    return 1.0 / math.sqrt(d)
