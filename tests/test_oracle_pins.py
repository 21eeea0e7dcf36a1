"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- a hand-worked closed form, brute force over tokens, a textbook
softmax, an invariant or an identity stated by the pages.

Passages: TinyServe query-aware page selection article s2.1 (per-page min/max
metadata), s2.2 (bound score and its upper-bound property), s2.3 (top-K pages,
attention over only those); CS336 Lecture 10 "Inference" s2.3 (decode
attention) and s9.2 (PagedAttention block table, shared prefixes); Quail
AI-SQL engine article (partial results merged by log-sum-exp rescaling).
"""

import math

import numpy as np
import pytest
import scipy.special
import torch

from query_aware_sparse_kv_gb300 import workloads as W

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _small(kind="iid", kv=torch.float32, q=torch.float32, seq_lens=(37, 64, 5), hq=4, hkv=2, d=16, P=8,
           top_k=3, seed=7, extra=3, **kw):
    spec = W.Spec(name="t", batch=len(seq_lens), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, page_size=P,
                  seq_lens=seq_lens, top_k=top_k, q_dtype=q, kv_dtype=kv, kind=kind, extra_pool_pages=extra,
                  seed=seed, **kw)
    return W.make_inputs(spec)


def _valid_keys(inp, b, g):
    """Contiguous [n_tok][d] keys / values of sequence b, KV head g, gathered
    through the page table with torch indexing (independent of the oracle)."""
    P = inp["spec"].page_size
    L = int(inp["seq_lens"][b])
    pos = torch.arange(L)
    phys = inp["page_table"][b, pos // P].long()
    k = inp["k_pool"][phys, g, pos % P].double().numpy()
    v = inp["v_pool"][phys, g, pos % P].double().numpy()
    return k, v


# ----------------------------------------------------------------- metadata --

@pytest.mark.parametrize("kv", [torch.float32, torch.bfloat16])
def test_meta_bounds_every_key_and_is_attained(oracle_lib, kv):
    """TinyServe s2.1: m_j / M_j are the element-wise min / max over the page's
    keys -- every valid key lies inside [m, M] and each bound is attained."""
    inp = _small(kv=kv)
    ids, vt = oracle_lib.all_pages(inp)
    meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    kp = inp["k_pool"].double().numpy()
    for p, v in zip(ids, vt):
        keys = kp[p, :, :v, :]  # [Hkv][v][d]
        m, M = meta[p, :, 0, :], meta[p, :, 1, :]
        assert np.isfinite(m).all() and np.isfinite(M).all()
        assert (keys >= m[:, None, :]).all() and (keys <= M[:, None, :]).all()
        assert (keys == m[:, None, :]).any(axis=1).all()
        assert (keys == M[:, None, :]).any(axis=1).all()


def test_meta_single_token_page_is_the_key(oracle_lib):
    inp = _small(seq_lens=(9,), P=8)  # last page holds one valid token
    last = int(inp["page_table"][0, 1])
    meta = oracle_lib.meta(inp["k_pool"], [last], [1])
    k0 = inp["k_pool"][last, :, 0, :].double().numpy()
    assert np.array_equal(meta[last, :, 0], k0) and np.array_equal(meta[last, :, 1], k0)


def test_meta_ignores_slots_past_the_valid_tokens(oracle_lib):
    """The generator puts NaN past seq_len; a valid-token bound off by one
    would read it."""
    inp = _small(seq_lens=(13,), P=8)
    last = int(inp["page_table"][0, 1])
    assert torch.isnan(inp["k_pool"][last, :, 5:]).all()
    meta = oracle_lib.meta(inp["k_pool"], [last], [5])
    assert np.isfinite(meta[last]).all()


def test_meta_rejects_bad_ids(oracle_lib):
    inp = _small()
    n_pool = inp["k_pool"].shape[0]
    with pytest.raises(IndexError):
        oracle_lib.meta(inp["k_pool"], [n_pool], [1])
    with pytest.raises(IndexError):
        oracle_lib.meta(inp["k_pool"], [0], [0])


# -------------------------------------------------------------------- score --

def test_bound_worked_example(oracle_lib):
    """A hand-worked case of TinyServe s2.2.  Keys (1,2,3,4) and (-1,0,5,2):
    m = (-1,0,3,2), M = (1,2,5,4).  q = (1,-2,0.5,0): positive components take
    M, negative take m:  1*1 + (-2)*0 + 0.5*5 + 0*(either) = 3.5.
    The two true dot products are -1.5 and 1.5, both below 3.5."""
    kp = torch.zeros((1, 1, 2, 4), dtype=torch.float32)
    kp[0, 0, 0] = torch.tensor([1.0, 2.0, 3.0, 4.0])
    kp[0, 0, 1] = torch.tensor([-1.0, 0.0, 5.0, 2.0])
    meta = oracle_lib.meta(kp, [0], [2])
    assert meta[0, 0, 0].tolist() == [-1.0, 0.0, 3.0, 2.0]
    assert meta[0, 0, 1].tolist() == [1.0, 2.0, 5.0, 4.0]
    q = np.array([1.0, -2.0, 0.5, 0.0])
    assert oracle_lib.bound(q, meta[0, 0, 0], meta[0, 0, 1]) == 3.5
    assert float(q @ kp[0, 0, 0].double().numpy()) == -1.5
    assert float(q @ kp[0, 0, 1].double().numpy()) == 1.5


@pytest.mark.parametrize("kv", [torch.float32, torch.bfloat16])
def test_bound_is_an_upper_bound_of_every_key(oracle_lib, kv):
    """TinyServe s2.2: the score is an upper bound of the page's true maximum
    q.k -- checked by brute force over every token, page and head."""
    inp = _small(kv=kv, seq_lens=(70, 33, 128), d=32, hq=8, hkv=2)
    ids, vt = oracle_lib.all_pages(inp)
    meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    q = inp["q"].double().numpy()
    kp = inp["k_pool"].double().numpy()
    for p, v in zip(ids, vt):
        for g in range(2):
            for h in range(g * 4, g * 4 + 4):
                for b in range(3):
                    qb = q[b, h]
                    s = oracle_lib.bound(qb, meta[p, g, 0], meta[p, g, 1])
                    true_max = (kp[p, g, :v] @ qb).max()
                    slack = 1e-9 * np.abs(qb).sum() * np.abs(kp[p, g, :v]).max()
                    assert s >= true_max - slack


def test_bound_equals_the_dot_product_on_a_single_token_page(oracle_lib):
    """With one key, m = M = k and the bound collapses to q.k exactly."""
    rng = np.random.default_rng(1)
    k = rng.standard_normal(64)
    q = rng.standard_normal(64)
    assert math.isclose(oracle_lib.bound(q, k, k), float(q @ k), rel_tol=1e-13, abs_tol=1e-13)


def test_bound_one_signed_query(oracle_lib):
    """All-positive q reads only M; all-negative q reads only m."""
    rng = np.random.default_rng(2)
    m = rng.standard_normal(32)
    M = m + rng.random(32)
    qp = rng.random(32) + 0.1
    assert math.isclose(oracle_lib.bound(qp, m, M), float(qp @ M), rel_tol=1e-13)
    assert math.isclose(oracle_lib.bound(-qp, m, M), float(-qp @ m), rel_tol=1e-13)


def test_swapped_comparator_fails_the_upper_bound_pin():
    """Shows the upper-bound pin catches the most likely misreading of the
    garbled comparator (q < 0 ? M : m): that variant is a lower bound."""
    rng = np.random.default_rng(3)
    keys = rng.standard_normal((16, 32))
    m, M = keys.min(0), keys.max(0)
    q = rng.standard_normal(32)
    wrong = float(np.sum(q * np.where(q > 0, m, M)))
    assert wrong < (keys @ q).max()


def test_group_score_is_the_max_head_bound(oracle_lib):
    """Reading for grouped-query attention: one score per (sequence, KV head)
    that bounds every head of the group; it is one of the heads' bounds."""
    inp = _small(seq_lens=(64, 40), hq=8, hkv=2, d=16)
    ids, vt = oracle_lib.all_pages(inp)
    meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    q = inp["q"].double().numpy()
    for b in range(2):
        nb = int(inp["n_pages"][b])
        for g in range(2):
            s = oracle_lib.row_scores(q[b, g * 4:(g + 1) * 4], meta, inp["page_table"][b], nb, g)
            for j in range(nb):
                p = int(inp["page_table"][b, j])
                v = min(8, int(inp["seq_lens"][b]) - j * 8)
                heads = [oracle_lib.bound(q[b, h], meta[p, g, 0], meta[p, g, 1]) for h in range(g * 4, g * 4 + 4)]
                assert s[j] in heads
                true_max = (inp["k_pool"][p, g, :v].double().numpy() @ q[b, g * 4:(g + 1) * 4].T).max()
                assert s[j] >= true_max - 1e-9


# ------------------------------------------------------------------- select --

def _count_rule(scores, k):
    """Brute force: page j is kept iff fewer than k pages beat it, where a page
    beats j if its score is higher, or equal with a lower index."""
    n = len(scores)
    keep = []
    for j in range(n):
        beaten = sum(1 for i in range(n) if scores[i] > scores[j] or (scores[i] == scores[j] and i < j))
        if beaten < k:
            keep.append(j)
    return keep


@pytest.mark.parametrize("n,k", [(50, 7), (64, 64), (10, 30), (33, 1), (100, 99)])
def test_select_matches_the_counting_rule(oracle_lib, n, k):
    rng = np.random.default_rng(n * 31 + k)
    scores = np.round(rng.standard_normal(n) * 4) / 4  # many ties
    sel, ns = oracle_lib.select(scores, k)
    want = _count_rule(scores, k)
    assert ns == min(n, k)
    assert sel[:ns].tolist() == want
    assert (sel[ns:] == -1).all()


def test_select_all_equal_scores_takes_the_first_pages(oracle_lib):
    sel, ns = oracle_lib.select(np.zeros(20), 5)
    assert sel.tolist() == [0, 1, 2, 3, 4]


def test_select_top1_is_the_first_argmax(oracle_lib):
    rng = np.random.default_rng(9)
    s = rng.integers(0, 5, 40).astype(float)
    sel, _ = oracle_lib.select(s, 1)
    assert sel[0] == int(np.argmax(s))


# ---------------------------------------------------------------- attention --

@pytest.mark.parametrize("kv,q", [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
                                  (torch.bfloat16, torch.float32)])
def test_all_pages_equals_dense_softmax_attention(oracle_lib, kv, q):
    """K = all pages is ordinary decode attention (CS336 s2.3): compared with
    scipy's softmax / logsumexp over the de-paged keys."""
    inp = _small(kv=kv, q=q, seq_lens=(37, 64, 5), hq=4, hkv=2, d=16, P=8)
    qd = inp["q"].double().numpy()
    scale = 1.0 / math.sqrt(16)
    for b in range(3):
        nb = int(inp["n_pages"][b])
        for g in range(2):
            out, lse = oracle_lib.attend_row(inp, b, g, list(range(nb)))
            k, v = _valid_keys(inp, b, g)
            for i, h in enumerate(range(g * 2, g * 2 + 2)):
                logits = scale * (k @ qd[b, h])
                w = scipy.special.softmax(logits)
                np.testing.assert_allclose(out[i], w @ v, rtol=1e-12, atol=1e-12)
                assert math.isclose(lse[i], scipy.special.logsumexp(logits), rel_tol=1e-12, abs_tol=1e-12)


def test_identical_keys_give_the_mean_value(oracle_lib):
    """All logits equal -> uniform weights -> the output is the mean of V."""
    inp = _small(seq_lens=(21,), hq=2, hkv=1, d=8, P=8)
    kp = inp["k_pool"]
    kp[:] = torch.tensor([0.5, -1.0, 2.0, 0.0, 1.0, 1.0, -3.0, 0.25])
    out, lse = oracle_lib.attend_row(inp, 0, 0, [0, 1, 2])
    _, v = _valid_keys(inp, 0, 0)
    np.testing.assert_allclose(out[0], v.mean(0), rtol=1e-12, atol=1e-13)
    logit = float(inp["q"][0, 0].double() @ kp[0, 0, 0].double()) / math.sqrt(8)
    assert math.isclose(lse[0], logit + math.log(21), rel_tol=1e-12)


def test_two_token_worked_example(oracle_lib):
    """Two keys with logits 0 and ln 3 (sm_scale 1): weights 1/4 and 3/4."""
    spec = W.Spec(name="t", batch=1, num_q_heads=1, num_kv_heads=1, head_dim=2, page_size=2, seq_lens=(2,),
                  top_k=1, q_dtype=torch.float32, kv_dtype=torch.float32, contiguous=True)
    inp = W.make_inputs(spec)
    inp["q"][:] = torch.tensor([1.0, 0.0])
    inp["k_pool"][0, 0] = torch.tensor([[0.0, 5.0], [math.log(3.0), -7.0]])
    inp["v_pool"][0, 0] = torch.tensor([[4.0, 8.0], [0.0, -4.0]])
    out, lse = oracle_lib.attend_row(inp, 0, 0, [0], sm_scale=1.0)
    ln3 = float(np.float32(math.log(3.0)))
    np.testing.assert_allclose(out[0], [0.25 * 4.0 + 0.75 * 0.0, 0.25 * 8.0 + 0.75 * -4.0], rtol=1e-6)
    assert math.isclose(lse[0], math.log(1.0 + math.exp(ln3)), rel_tol=1e-12)


def test_lse_merge_of_two_page_sets_equals_the_union(oracle_lib):
    """Quail's recursive attention / flash decoding: attention over A and over
    B, merged by log-sum-exp rescaling, equals attention over A u B."""
    inp = _small(kv=torch.bfloat16, seq_lens=(61,), hq=4, hkv=1, d=16, P=8)
    A, Bp = [0, 3, 5], [1, 2, 7]
    oa, la = oracle_lib.attend_row(inp, 0, 0, A)
    ob, lb = oracle_lib.attend_row(inp, 0, 0, Bp)
    ou, lu = oracle_lib.attend_row(inp, 0, 0, sorted(A + Bp))
    lse = np.logaddexp(la, lb)
    merged = np.exp(la - lse)[:, None] * oa + np.exp(lb - lse)[:, None] * ob
    np.testing.assert_allclose(merged, ou, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lu, rtol=1e-13)


@pytest.mark.parametrize("splits", [1, 2, 7])
def test_lse_merge_is_independent_of_the_split_count(oracle_lib, splits):
    """The split-K decode's merge: the row's pages cut into `splits`
    contiguous ranges (some ending inside the partial last page's range),
    each attended alone, then folded by log-sum-exp one piece at a time with
    a running maximum (the order the merge kernel uses), give attention over
    all pages: the result does not depend on the split count."""
    inp = _small(kv=torch.bfloat16, seq_lens=(61,), hq=4, hkv=1, d=16, P=8)
    pages = list(range(8))  # 61 tokens in 8-token pages: the last page holds 5
    cuts = np.linspace(0, len(pages), splits + 1).round().astype(int)
    pieces = [oracle_lib.attend_row(inp, 0, 0, pages[cuts[i]:cuts[i + 1]]) for i in range(splits)]
    mx = np.full(4, -np.inf)
    den = np.zeros(4)
    acc = np.zeros((4, 16))
    for o, lse in pieces:
        m = np.maximum(mx, lse)
        scale = np.exp(mx - m)
        w = np.exp(lse - m)
        den = den * scale + w
        acc = acc * scale[:, None] + w[:, None] * o
        mx = m
    ou, lu = oracle_lib.attend_row(inp, 0, 0, pages)
    np.testing.assert_allclose(acc / den[:, None], ou, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(mx + np.log(den), lu, rtol=1e-13)


def test_physical_layout_does_not_matter(oracle_lib):
    """PagedAttention (CS336 s9.2): moving pages to other physical slots and
    rewriting the table leaves the result unchanged."""
    inp = _small(seq_lens=(40, 17), hq=2, hkv=2, d=8, P=8)
    ref = oracle_lib.step(inp, top_k=None)
    n_pool = inp["k_pool"].shape[0]
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(5))
    moved = dict(inp)
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(n_pool)
    moved["k_pool"] = inp["k_pool"][inv].contiguous()  # page p now lives at slot perm[p]
    moved["v_pool"] = inp["v_pool"][inv].contiguous()
    t = inp["page_table"].clone()
    t[t >= 0] = perm[t[t >= 0].long()].to(torch.int32)
    moved["page_table"] = t
    got = oracle_lib.step(moved, top_k=None)
    np.testing.assert_array_equal(got["out"], ref["out"])


def test_shared_prefix_rows_share_physical_pages(oracle_lib):
    """Sequences whose tables alias the same prefix pages and the same q see
    the same prefix keys: attention over the prefix alone is identical."""
    spec = W.Spec(name="sp", batch=3, num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=8, kind="shared_prefix",
                  prefix_pages=4, suffix_pages=2, q_dtype=torch.float32, kv_dtype=torch.float32, seed=3)
    inp = W.make_inputs(spec)
    inp["q"][1:] = inp["q"][0]
    outs = [oracle_lib.attend_row(inp, b, 0, [0, 1, 2, 3])[0] for b in range(3)]
    np.testing.assert_array_equal(outs[0], outs[1])
    np.testing.assert_array_equal(outs[0], outs[2])


def test_garbage_past_seq_len_is_ignored(oracle_lib):
    inp = _small(seq_lens=(13, 30), d=8, P=8)
    ref = oracle_lib.step(inp, top_k=None)
    assert np.isfinite(ref["out"]).all()
    for b in range(2):
        nb = int(inp["n_pages"][b])
        p = int(inp["page_table"][b, nb - 1])
        valid = int(inp["seq_lens"][b]) - (nb - 1) * 8
        inp["k_pool"][p, :, valid:] = 1e30
        inp["v_pool"][p, :, valid:] = -1e30
    got = oracle_lib.step(inp, top_k=None)
    np.testing.assert_array_equal(got["out"], ref["out"])


def test_empty_attention_is_zero(oracle_lib):
    inp = _small(seq_lens=(8,), d=8, P=8)
    out, lse = oracle_lib.attend_row(inp, 0, 0, [])
    assert (out == 0).all() and np.isneginf(lse).all()


# --------------------------------------------------------------- full step --

def test_step_composes_scores_select_attend(oracle_lib):
    """The batch driver equals the three steps taken one by one."""
    inp = _small(kv=torch.bfloat16, q=torch.bfloat16, seq_lens=(100, 57, 8), hq=8, hkv=2, d=16, P=8, top_k=4)
    res = oracle_lib.step(inp)
    meta = res["meta"]
    q = inp["q"].double().numpy()
    for e, r in enumerate(res["rows"]):
        b, g = divmod(int(r), 2)
        nb = int(inp["n_pages"][b])
        s = oracle_lib.row_scores(q[b, g * 4:(g + 1) * 4], meta, inp["page_table"][b], nb, g)
        np.testing.assert_array_equal(res["scores"][e, :nb], s)
        sel, ns = oracle_lib.select(s, 4)
        assert res["n_sel"][e] == ns and res["selected"][e].tolist() == sel.tolist()
        out, lse = oracle_lib.attend_row(inp, b, g, sel[:ns])
        np.testing.assert_array_equal(res["out"][e], out)
        np.testing.assert_array_equal(res["lse"][e], lse)


def test_planted_pages_are_selected(oracle_lib):
    """Sanity of method + generator: the pages whose keys were pushed along the
    group's mean query (the planted 2 %) survive the bound-score top-K."""
    spec = W.spec_for("llama3_8b", batch=2, seq_len_range=(1600, 2000), max_pages=None, top_k=16)
    inp = W.make_inputs(spec)
    res = oracle_lib.step(inp)
    hits = total = 0
    for e, r in enumerate(res["rows"]):
        b, g = divmod(int(r), spec.num_kv_heads)
        pl = [int(x) for x in inp["planted"][b, g] if x >= 0]
        hits += len(set(pl) & set(res["selected"][e].tolist()))
        total += len(pl)
    assert total > 0 and hits == total


# ------------------------------------------- Block Top-K (centroid) scorer --
# Vortex sparse-attention digest, method overview item 1: the cache phase
# keeps each block's mean key; the indexer scores q . centroid and keeps the
# top-K blocks.

@pytest.mark.parametrize("kv", [torch.float32, torch.bfloat16])
def test_centroid_is_the_mean_of_the_valid_keys(oracle_lib, kv):
    """Brute force: the per-dimension mean of the page's valid keys, taken by
    numpy over the pool slice (fsum-accurate)."""
    inp = _small(kv=kv)
    ids, vt = oracle_lib.all_pages(inp)
    cent = oracle_lib.centroids(inp["k_pool"], ids, vt)
    kp = inp["k_pool"].double().numpy()
    for p, v in zip(ids, vt):
        want = np.array([[math.fsum(kp[p, g, :v, i]) / v for i in range(kp.shape[3])] for g in range(kp.shape[1])])
        np.testing.assert_allclose(cent[p], want, rtol=1e-14, atol=1e-14)


def test_centroid_special_cases(oracle_lib):
    """A one-token page's centroid is the key; a page of identical keys has
    that key as its centroid; NaN slots past the valid count never leak."""
    inp = _small(seq_lens=(17, 8, 3))
    kp = inp["k_pool"]
    P = inp["spec"].page_size
    p_one = int(inp["page_table"][0, 2])    # sequence 0, third page: 1 valid token
    p_same = int(inp["page_table"][1, 0])   # sequence 1, first page: made constant
    kp[p_same] = kp[p_same, :, :1, :].expand(-1, P, -1).clone()
    ids = np.array([p_one, p_same], dtype=np.int32)
    vt = np.array([1, P], dtype=np.int32)
    cent = oracle_lib.centroids(kp, ids, vt)
    np.testing.assert_array_equal(cent[p_one], kp[p_one, :, 0, :].double().numpy())
    np.testing.assert_allclose(cent[p_same], kp[p_same, :, 0, :].double().numpy(), rtol=1e-15, atol=0)
    p3 = int(inp["page_table"][2, 0])       # sequence 2: 3 valid tokens, NaN past them
    assert torch.isnan(kp[p3, :, 3:]).all()
    c3 = oracle_lib.centroids(kp, np.array([p3], dtype=np.int32), np.array([3], dtype=np.int32))
    assert np.isfinite(c3[p3]).all()


def test_centroid_score_is_the_mean_token_score(oracle_lib):
    """Linearity: q . mean_t k_t equals the mean over the page's tokens of the
    per-token logits q . k_t, computed token by token (brute force)."""
    inp = _small(kv=torch.bfloat16, seq_lens=(45, 30), hq=6, hkv=2, d=16, P=8)
    ids, vt = oracle_lib.all_pages(inp)
    cent = oracle_lib.centroids(inp["k_pool"], ids, vt)
    q = inp["q"].double().numpy()
    kp = inp["k_pool"].double().numpy()
    P, G = 8, 3
    for b in range(2):
        nb = int(inp["n_pages"][b])
        L = int(inp["seq_lens"][b])
        for g in range(2):
            s = oracle_lib.centroid_row_scores(q[b, g * G:(g + 1) * G], cent, inp["page_table"][b], nb, g)
            for j in range(nb):
                p = int(inp["page_table"][b, j])
                n = min(P, L - j * P)
                per_head = [math.fsum(float(q[b, g * G + h] @ kp[p, g, t]) for t in range(n)) / n for h in range(G)]
                assert abs(s[j] - max(per_head)) <= 1e-12 * (1 + abs(s[j]))


def test_centroid_score_never_exceeds_the_bound(oracle_lib):
    """Invariant tying the two scorers: a mean never exceeds a maximum, so for
    every page and head q . centroid <= max_t q . k_t <= the TinyServe bound."""
    inp = _small(kind="page_offset", kv=torch.bfloat16, seq_lens=(60, 33, 17), hq=4, hkv=2, d=16, P=8)
    ids, vt = oracle_lib.all_pages(inp)
    cent = oracle_lib.centroids(inp["k_pool"], ids, vt)
    meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    q = inp["q"].double().numpy()
    for b in range(3):
        nb = int(inp["n_pages"][b])
        for g in range(2):
            qg = q[b, g * 2:(g + 1) * 2]
            sc = oracle_lib.centroid_row_scores(qg, cent, inp["page_table"][b], nb, g)
            sb = oracle_lib.row_scores(qg, meta, inp["page_table"][b], nb, g)
            assert (sc <= sb + 1e-12 * (1 + np.abs(sb))).all()


def test_centroid_shift_equivariance(oracle_lib):
    """Adding a vector u to every key of the pool moves each centroid by u and
    each head's score by q_h . u."""
    inp = _small(kv=torch.float32, seq_lens=(24, 40), hq=2, hkv=1, d=8, P=8)
    ids, vt = oracle_lib.all_pages(inp)
    c0 = oracle_lib.centroids(inp["k_pool"], ids, vt)
    u = torch.linspace(-1.0, 2.0, 8, dtype=torch.float64)
    shifted = (inp["k_pool"].double() + u).to(torch.float32)
    c1 = oracle_lib.centroids(shifted, ids, vt)
    np.testing.assert_allclose(c1[ids] - c0[ids], np.broadcast_to(u.numpy(), c0[ids].shape), atol=1e-6)
    q = inp["q"].double().numpy()
    for b in range(2):
        nb = int(inp["n_pages"][b])
        for h in range(2):
            s0 = oracle_lib.centroid_row_scores(q[b, h:h + 1], c0, inp["page_table"][b], nb, 0)
            s1 = oracle_lib.centroid_row_scores(q[b, h:h + 1], c1, inp["page_table"][b], nb, 0)
            np.testing.assert_allclose(s1 - s0, float(q[b, h] @ u.numpy()), atol=1e-5)


def test_centroid_step_composes_and_finds_the_aligned_pages(oracle_lib):
    """The batch driver with the centroid scorer equals its three steps one by
    one; on the centroid workload (keys around 64 centroids, q near one) the
    kept pages are exactly the best-aligned ones by brute force."""
    spec = W.spec_for("long_context", batch=2, seq_len_range=(1500, 2500), max_pages=None, top_k=8)
    inp = W.make_inputs(spec)
    res = oracle_lib.step(inp, scorer="centroid")
    cent = res["meta"]
    q = inp["q"].double().numpy()
    G, Hkv, P = spec.group, spec.num_kv_heads, spec.page_size
    kp = inp["k_pool"].double().numpy()
    for e, r in enumerate(res["rows"]):
        b, g = divmod(int(r), Hkv)
        nb = int(inp["n_pages"][b])
        L = int(inp["seq_lens"][b])
        s = oracle_lib.centroid_row_scores(q[b, g * G:(g + 1) * G], cent, inp["page_table"][b], nb, g)
        np.testing.assert_array_equal(res["scores"][e, :nb], s)
        sel, ns = oracle_lib.select(s, 8)
        assert res["selected"][e].tolist() == sel.tolist() and res["n_sel"][e] == ns
        # brute force: mean per-token logit per page, best of the group's heads
        brute = []
        for j in range(nb):
            p = int(inp["page_table"][b, j])
            n = min(P, L - j * P)
            keys = kp[p, g, :n]
            brute.append(max(float((keys @ q[b, g * G + h]).mean()) for h in range(G)))
        order = sorted(range(nb), key=lambda j: (-brute[j], j))[:8]
        assert sorted(order) == sel[:ns].tolist()


# ------------------------------------------- approximate radix top-K (lossy) --
# Vortex digest, method overview item 3: radix Top-K that stops early once
# enough high-confidence candidates are collected and samples the rest at
# random from the threshold bin; recall@k > 0.97 across bimodal, normal,
# lognormal and uniform score distributions (item 3 of the evaluation list).

def test_splitmix64_reference_outputs(oracle_lib):
    """The counter-based generator is SplitMix64 as published (Steele, Lea and
    Flood 2014): its first outputs from seed 1234567 and from seed 0 are the
    generator's published reference values."""
    assert [oracle_lib.splitmix64(1234567, i) for i in range(1, 6)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423, 4593380528125082431,
        16408922859458223821]
    assert oracle_lib.splitmix64(0, 1) == 0xE220A8397B1DCDAF


def _scores(dist, n, rng):
    if dist == "normal":
        s = rng.standard_normal(n)
    elif dist == "uniform":
        s = rng.uniform(-1.0, 1.0, n)
    elif dist == "lognormal":
        s = rng.lognormal(0.0, 1.0, n)
    else:  # bimodal
        s = np.where(rng.random(n) < 0.3, rng.normal(4.0, 0.5, n), rng.normal(0.0, 1.0, n))
    return s.astype(np.float32)


def _exact_topk(s, k):
    """Brute force: the k largest, ties to the lower index, ascending."""
    order = sorted(range(len(s)), key=lambda j: (-float(s[j]), j))
    return sorted(order[:k])


@pytest.mark.parametrize("dist", ["bimodal", "normal", "lognormal", "uniform"])
def test_approx_select_with_eps0_is_exact(oracle_lib, dist):
    rng = np.random.default_rng(11)
    for n, k in [(300, 40), (2048, 154), (5000, 128)]:
        s = _scores(dist, n, rng)
        s[rng.integers(0, n, 20)] = s[0]  # some ties
        sel, cnt = oracle_lib.select_approx(s, k, 0.0, 7, 3)
        assert cnt == k and sel.tolist() == _exact_topk(s, k)


@pytest.mark.parametrize("dist", ["bimodal", "normal", "lognormal", "uniform"])
@pytest.mark.parametrize("eps", [0.01, 0.03, 0.1])
def test_approx_select_recall_bound(oracle_lib, dist, eps):
    """recall@K >= 1 - eps by construction (every key above the threshold bin
    is kept and at most floor(eps K) are drawn), K distinct indices,
    ascending, each drawn one from the threshold bin (score <= the exact K-th)."""
    rng = np.random.default_rng(hash((dist, eps)) % 2 ** 32)
    for n, k in [(512, 154), (2048, 128), (4096, 256), (20000, 128)]:
        s = _scores(dist, n, rng)
        exact = set(_exact_topk(s, k))
        for seed in range(3):
            sel, cnt = oracle_lib.select_approx(s, k, eps, seed, 5)
            sel = sel[:cnt].tolist()
            assert cnt == k and len(set(sel)) == k and sel == sorted(sel)
            missed = len(exact - set(sel))
            assert missed <= math.floor(eps * k)
            kth = sorted(s.astype(np.float64), reverse=True)[k - 1]
            assert all(float(s[j]) <= kth for j in set(sel) - exact)


def test_approx_sampling_is_uniform_over_the_threshold_bin(oracle_lib):
    """Systematic sampling with a random start: over many seeds every key of a
    tied threshold bin is kept with frequency need / m."""
    n, k = 1000, 100
    s = np.zeros(n, dtype=np.float32)
    s[:60] = 5.0  # 60 certain keys; the other 940 tie in the threshold bin
    need, m = k - 60, n - 60
    eps = need / k  # need_max = 40: stop after the first pass (top digit)
    hits = np.zeros(n)
    trials = 3000
    for seed in range(trials):
        sel, cnt = oracle_lib.select_approx(s, k, eps, seed, 0)
        assert cnt == k and set(range(60)) <= set(sel.tolist())
        hits[sel] += 1
    p = need / m
    freq = hits[60:] / trials
    sigma = math.sqrt(p * (1 - p) / trials)
    assert abs(freq.mean() - p) < 1e-9
    assert np.abs(freq - p).max() < 6 * sigma


def test_approx_select_is_deterministic_per_seed_and_row(oracle_lib):
    rng = np.random.default_rng(3)
    s = np.round(rng.standard_normal(3000), 1).astype(np.float32)  # many ties
    a, _ = oracle_lib.select_approx(s, 200, 0.2, 42, 9)
    b, _ = oracle_lib.select_approx(s, 200, 0.2, 42, 9)
    c, _ = oracle_lib.select_approx(s, 200, 0.2, 43, 9)
    d, _ = oracle_lib.select_approx(s, 200, 0.2, 42, 10)
    assert a.tolist() == b.tolist()
    assert a.tolist() != c.tolist() and a.tolist() != d.tolist()


def test_approx_need_max_is_the_double_product_floored(oracle_lib):
    """need_max = floor(epsilon * K) with epsilon and the product in IEEE
    double: 0.03 * 100 and 0.7 * 10 round to the integers 3 and 7, 0.57 * 100
    to 56.99999999999999 (so 56), and a single-precision epsilon would give
    2, 0 and 6 for the first three."""
    assert oracle_lib.need_max(100, 0.03) == 3
    assert oracle_lib.need_max(100, 0.01) == 1
    assert oracle_lib.need_max(10, 0.7) == 7
    assert oracle_lib.need_max(100, 0.57) == 56
    assert oracle_lib.need_max(128, 0.0) == 0
    f32 = lambda e, k: math.floor(float(np.float32(e)) * k)
    assert (f32(0.03, 100), f32(0.01, 100), f32(0.7, 10)) == (2, 0, 6)


def test_approx_digits_are_the_fixed_bytes_of_the_key(oracle_lib):
    """The radix digits are the key's fixed bytes (bits 31..24, 23..16, ...).
    Scores 1 + m/128 + r*2^-16 in [1, 2) share their top byte; their second
    byte is 0x80 + m.  Three keys sit in a higher second-byte bucket, five in
    bucket m = 10 whose lower bits differ; with K = 4 and need_max = 1 the
    select stops after the second byte, so the one missing key is drawn from
    all five (a start at the highest differing bit would split them by bit
    15 and draw from two only)."""
    high = [1 + 90 / 128, 1 + 91 / 128, 1 + 92 / 128]
    bucket = [1 + 10 / 128 + r * 2.0 ** -16 for r in (1, 2, 3, 257, 258)]
    s = np.array(high + bucket + [1.0, 1.01], dtype=np.float32)
    seen = set()
    for seed in range(400):
        sel, cnt = oracle_lib.select_approx(s, 4, 0.25, seed, 0)
        assert cnt == 4 and set(sel[:4].tolist()) >= {0, 1, 2}
        (extra,) = set(sel[:4].tolist()) - {0, 1, 2}
        assert 3 <= extra <= 7
        seen.add(extra)
    assert seen == {3, 4, 5, 6, 7}
