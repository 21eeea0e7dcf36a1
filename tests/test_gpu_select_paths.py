"""GPU parity of the ranking kernel (TinyServe query-aware page selection,
s2.3: top-K of the page scores by a radix pass; Vortex digest, method
overview item 3: the lossy variant).

The selected list must equal, index for index, the oracle's rule applied to
the GPU's own fp32 scores: the exact top-K with ties to the lower page index,
or the lossy top-K.  Cases cover clustered bound scores, heavy ties, rows
shorter than K, rows of 2048 to 4096 pages (compacted by per-thread runs
rather than warp ballots) and rows longer than the 4096 keys the kernel
keeps in shared memory (those read their keys from global memory in every
pass).
Each batch is ranked twice, with its own page table and with the table
padded by -1 columns: width must change nothing."""
import numpy as np
import pytest
import torch

import parity as PR
import query_aware_sparse_kv_gb300 as qskv
from query_aware_sparse_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu

PAD = 300  # extra page-table columns, all -1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from query_aware_sparse_kv_gb300 import build

    build.build()
    qskv.load()


def _ties(spec):
    inp = W.make_inputs(spec)
    inp["k_pool"] = (torch.round(inp["k_pool"].float() * 2) / 2).to(inp["k_pool"].dtype)  # many equal scores
    return inp


CASES = {
    "llama": lambda: W.make_inputs(W.spec_for("llama3_8b", batch=4, seq_len_range=(3000, 32000), max_pages=None,
                                              top_k=128)),
    "gpt2": lambda: W.make_inputs(W.spec_for("gpt2_345m", batch=2, seq_lens=(8192, 5000), top_k=154)),
    "long": lambda: W.make_inputs(W.spec_for("long_context", batch=2, seq_len_range=(20000, 65000), max_pages=None,
                                             top_k=128)),
    "ties": lambda: _ties(W.Spec(name="ties", batch=3, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                                 seq_lens=(16 * 2000, 16 * 700 + 5, 16 * 40), top_k=100, kind="iid", seed=41)),
    "long_rows": lambda: W.make_inputs(W.spec_for("long_context", batch=2, seq_len_range=(70000, 130000),
                                                  max_pages=None, top_k=128)),
    "beyond_smem": lambda: W.make_inputs(W.Spec(name="long_rows", batch=2, num_q_heads=8, num_kv_heads=2,
                                                head_dim=64, page_size=16, seq_lens=(16 * 4500 + 3, 16 * 4200),
                                                top_k=200, kind="iid", seed=43)),
    # many short rows (2200), some shorter than K: one ranking CTA per row
    "many_rows": lambda: W.make_inputs(W.Spec(name="many_rows", batch=1100, num_q_heads=4, num_kv_heads=2,
                                              head_dim=64, page_size=16, seq_len_range=(20, 700), top_k=12,
                                              kind="iid", seed=44)),
}


def _widen(inp, width):
    t = inp["page_table"]
    pad = torch.full((t.shape[0], width - t.shape[1]), -1, dtype=t.dtype)
    out = dict(inp)
    out["page_table"] = torch.cat([t, pad], dim=1)
    return out


def _rank(inp, oracle, scorer, eps, seed):
    dec = qskv.from_inputs(inp, scorer=scorer, approx_epsilon=eps, approx_seed=seed)
    ids, vt = oracle.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    sc = torch.full(tuple(dec.selected.shape[:2]) + (inp["page_table"].shape[1],), float("nan"), device="cuda")
    dec.select(scores=sc)
    dec.check()
    torch.cuda.synchronize()
    return sc.cpu().numpy(), dec.selected.cpu().numpy(), dec.n_selected.cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("scorer", ["bound", "centroid"])
@pytest.mark.parametrize("eps", [None, 0.03, 0.2])
def test_ranking_matches_the_oracle_rule(oracle_lib, name, scorer, eps):
    inp = CASES[name]()
    spec = inp["spec"]
    K, Hkv = spec.top_k, spec.num_kv_heads
    seed = 77
    s_n, sel_n, n_n = _rank(inp, oracle_lib, scorer, eps, seed)
    s_w, sel_w, n_w = _rank(_widen(inp, inp["page_table"].shape[1] + PAD), oracle_lib, scorer, eps, seed)
    for r in range(spec.batch * Hkv):
        b, g = divmod(r, Hkv)
        n_b = PR.n_pages_of(inp, b)
        s = s_n[b, g, :n_b]
        assert np.array_equal(s, s_w[b, g, :n_b]), f"row {r}: scores differ with the table width"
        want, cnt = oracle_lib.select_approx(s, K, eps or 0.0, seed, r)
        for sel, ns, kind in ((sel_n, n_n, "own table"), (sel_w, n_w, "padded table")):
            assert ns[b, g] == cnt, f"row {r} ({kind}): n_selected {ns[b, g]} != {cnt}"
            assert sel[b, g].tolist() == want.tolist(), f"row {r} ({kind}): selection differs from the oracle rule"


def test_exact_rule_is_the_oracle_select(oracle_lib):
    """Cross-check with the oracle's exact select (a full sort) on the GPU
    scores, for heavy ties and for rows read from global memory."""
    for name in ("ties", "beyond_smem"):
        _exact_vs_sort(CASES[name](), oracle_lib)


def _exact_vs_sort(inp, oracle_lib):
    spec = inp["spec"]
    s_w, sel_w, n_w = _rank(inp, oracle_lib, "bound", None, 0)
    for r in range(spec.batch * spec.num_kv_heads):
        b, g = divmod(r, spec.num_kv_heads)
        n_b = PR.n_pages_of(inp, b)
        want, cnt = oracle_lib.select(s_w[b, g, :n_b].astype(np.float64), spec.top_k)
        assert n_w[b, g] == cnt and sel_w[b, g].tolist() == want.tolist()


def test_ranking_repeats_exactly_on_one_workspace(oracle_lib):
    """Calls on one workspace, alternating two queries, give identical
    selections every time: nothing a call leaves in the workspace changes
    the next call's result."""
    inp = CASES["llama"]()
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    q2 = (inp["q"].float() * -1.0).to(inp["q"].dtype).cuda()
    first = {}
    for i in range(6):
        q = dec.q if i % 2 == 0 else q2
        dec.selected.fill_(-7)
        dec.select(q=q)
        dec.check()
        torch.cuda.synchronize()
        got = (dec.selected.clone(), dec.n_selected.clone())
        if i < 2:
            first[i % 2] = got
        else:
            assert torch.equal(got[0], first[i % 2][0]) and torch.equal(got[1], first[i % 2][1]), f"call {i}"
    assert not torch.equal(first[0][0], first[1][0])
