"""Metadata refresh of the last pages fused with page selection.

TinyServe query-aware page selection, s5.3: a page's metadata is refreshed
at every decode step (the new token's key went into each sequence's last
page); s2.1-2.3: min/max metadata, bound score, top-K.
qskv_page_select_refresh rebuilds the metadata of every sequence's last page
inside the scoring launch and scores that page with it.  Checked: the last
pages' metadata against the oracle's element-wise scan of the new keys (bit
for bit), every other page's metadata untouched, scores against the
oracle's, the selection by the tie band, and the whole result equal to
kv_meta_build over the last pages followed by page_select."""
import numpy as np
import pytest
import torch

import parity as PR
import query_aware_sparse_kv_gb300 as qskv
from query_aware_sparse_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from query_aware_sparse_kv_gb300 import build

    build.build()
    qskv.load()


CASES = {
    # GQA 4, d=128, page 16; ragged lengths, one row short enough to keep every page
    "llama": W.spec_for("llama3_8b", batch=5, seq_lens=(3001, 1999, 77, 4096, 2500), max_pages=None, top_k=64),
    # MHA, d=64, fp32 q
    "gpt2": W.spec_for("gpt2_345m", batch=3, seq_lens=(8192, 4001, 1000), top_k=154),
    # page 32, the row-major scoring grid (2 KV heads)
    "long": W.spec_for("long_context", batch=2, seq_lens=(9000, 12345), max_pages=None, top_k=64,
                       num_q_heads=8, num_kv_heads=2),
}


def _new_last_keys(inp, seed):
    """Overwrite the valid key rows of every sequence's last page (the page
    the new token went into) with fresh values, in place."""
    g = torch.Generator().manual_seed(seed)
    ids, valid = W.last_pages(inp)
    for p, v in zip(ids.tolist(), valid.tolist()):
        new = 3.0 * torch.randn((inp["k_pool"].shape[1], v, inp["k_pool"].shape[3]), generator=g)
        inp["k_pool"][p, :, :v] = new.to(inp["k_pool"].dtype)
    return ids.numpy(), valid.numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_refresh_in_select_matches_the_oracle_and_the_two_calls(oracle_lib, name):
    inp = W.make_inputs(CASES[name])
    spec = inp["spec"]
    ids, vt = oracle_lib.all_pages(inp)
    old_meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    dec = qskv.from_inputs(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    last_ids, last_valid = _new_last_keys(inp, seed=7)  # the step's new keys, host copy
    dec.k_pool.copy_(inp["k_pool"].cuda())
    sc = torch.full((spec.batch, spec.num_kv_heads, inp["page_table"].shape[1]), float("nan"), device="cuda")
    dec.select(scores=sc, refresh_last=True)
    dec.check()
    torch.cuda.synchronize()

    # metadata: last pages rebuilt from the new keys, the others untouched
    new_meta = oracle_lib.meta(inp["k_pool"], last_ids, last_valid, out=old_meta.copy())
    PR.assert_meta_equal(dec.meta, new_meta, ids)

    # scores, selection and outputs against the oracle with the new metadata
    dec.decode()
    dec.check()
    PR.check_rows(inp, dec, range(spec.batch * spec.num_kv_heads), oracle_lib, oracle_meta=new_meta,
                  check_scores=sc)

    # the same as the two calls: metadata build of the last pages, then selection
    two = qskv.from_inputs(inp)
    two.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    two.build_meta(torch.from_numpy(last_ids).cuda(), torch.from_numpy(last_valid).cuda())
    sc2 = torch.full_like(sc, float("nan"))
    two.select(scores=sc2)
    two.check()
    torch.cuda.synchronize()
    assert torch.equal(two.selected, dec.selected) and torch.equal(two.n_selected, dec.n_selected)
    nb = inp["n_pages"].long()
    for b in range(spec.batch):
        assert torch.equal(sc[b, :, :nb[b]], sc2[b, :, :nb[b]])


def test_refresh_in_select_needs_bf16_kv():
    inp = W.make_inputs(W.spec_for("tiny"))  # fp32 KV
    dec = qskv.from_inputs(inp)
    with pytest.raises(qskv.QskvError) as e:
        qskv.page_select_refresh(dec.q, dec.k_pool, dec.meta, dec.page_table, dec.seq_lens, dec.top_k, dec.selected,
                                 dec.n_selected, dec.shape, dec.workspace)
    assert e.value.status == 2
    # the engine falls back to the two calls there
    assert not dec.can_refresh_in_select
