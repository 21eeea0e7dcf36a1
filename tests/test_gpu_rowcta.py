"""One row per k decode CTAs.

When the (sequence, KV head) rows fit one wave of decode CTAs (bf16 KV), the
k CTAs of row r decode it alone: each CTA's warps take a fixed share of the
row's selected pages and fold their partial results in the CTA by
log-sum-exp rescaling (Quail AI-SQL engine article: partial attention
combined as in flash decoding); with k = 1 (one or two rows per SM) that is
the row's output, with k > 1 (fewer rows than SMs) the CTA drawing the row's
last ticket folds the k pieces.  No merge kernel either way.  Sparse rows --
some with fewer pages than top_k -- and dense batches, d = 128 and d = 64,
are checked row by row against the oracle, and repeated calls on one
workspace give identical results."""
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


def _sms():
    return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count


def row_blocks(rows, slots, sms):
    """CTAs per row the library picks (0: the stream-K split)."""
    ctas = 2 * sms
    if rows <= 0 or rows > ctas or slots > 1024:
        return 0
    if rows >= sms:
        return 1
    k = min(ctas // rows, 8, slots // 4)
    return k if k >= 2 and rows * k >= sms else 0


def _case(kind):
    sms = _sms()
    if kind == "blocks_gpt2":   # 128 MHA rows, d = 64, fp32 q: two CTAs per row
        return W.spec_for("gpt2_345m")
    if kind == "blocks_long":   # 24 rows of 32-token pages: eight CTAs per row
        return W.spec_for("long_context", batch=3, seq_len_range=(3000, 9000), max_pages=None, top_k=64)
    if kind == "blocks_dense":  # dense d = 64 rows, fewer rows than SMs
        return W.spec_for("gpt2_345m", batch=7, seq_lens=None, seq_len_range=(400, 1500), max_pages=None, top_k=None,
                          num_q_heads=16, num_kv_heads=16)
    if kind == "sparse_mid":    # about 1.3 rows per SM, lengths around top_k
        return W.spec_for("llama3_8b", batch=(4 * sms) // (3 * 8), seq_len_range=(200, 6000), max_pages=None)
    if kind == "sparse_low":    # one row per SM (the smallest row count of the mode)
        return W.spec_for("llama3_8b", batch=-(-sms // 8), seq_len_range=(1500, 4000), max_pages=None, top_k=64)
    if kind == "sparse_high":   # two rows per SM (the largest)
        return W.spec_for("llama3_8b", batch=(2 * sms) // 8, seq_len_range=(300, 2500), max_pages=None, top_k=40)
    return W.spec_for("llama3_8b", batch=(4 * sms) // (3 * 8), seq_len_range=(100, 1500), max_pages=None,
                      top_k=None)


@pytest.mark.parametrize("kind", ["sparse_mid", "sparse_low", "sparse_high", "dense", "blocks_gpt2", "blocks_long",
                                  "blocks_dense"])
def test_row_per_cta_matches_the_oracle(oracle_lib, kind):
    spec = _case(kind)
    rows = spec.batch * spec.num_kv_heads
    inp = W.make_inputs(spec)
    slots = spec.top_k if spec.top_k is not None else inp["page_table"].shape[1]
    k = row_blocks(rows, slots, _sms())
    if kind.startswith("blocks"):
        assert k > 1, f"the case must split its rows over several CTAs (k = {k})"
    else:
        assert k == 1, f"the case must give each row one CTA (k = {k})"
    dec = qskv.from_inputs(inp)
    dense = spec.top_k is None
    o_meta = None
    if not dense:
        ids, vt = oracle_lib.all_pages(inp)
        dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
        dec.select()
        dec.check()
        o_meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    first = None
    for it in range(3):
        dec.out.fill_(float("nan"))
        dec.lse.fill_(float("nan"))
        dec.decode()
        dec.check()
        torch.cuda.synchronize()
        if first is None:
            PR.check_rows(inp, dec, list(range(rows)), oracle_lib, oracle_meta=o_meta, dense=dense)
            first = (dec.out.clone(), dec.lse.clone())
        else:
            assert torch.equal(dec.out, first[0]) and torch.equal(dec.lse, first[1]), f"call {it} differs"


def _edge_spec(kind):
    """Rows of no, one, two and many pages in the one-row-per-CTA split:
    with k = 1 (one row per SM or more) and with k = 8 (CTAs left without
    units give empty pieces)."""
    sms = _sms()
    if kind == "edge_k1":
        batch = -(-sms // 8) + 1
        lens = [0, 1, 15, 16, 17, 33] + [3000 + 97 * i for i in range(batch - 6)]
        return W.spec_for("llama3_8b", batch=batch, seq_lens=tuple(lens), seq_len_range=None, max_pages=None,
                          top_k=64, kind="iid")
    return W.spec_for("long_context", batch=3, seq_lens=(0, 40, 5000), seq_len_range=None, max_pages=None,
                      top_k=64, kind="iid")


@pytest.mark.parametrize("kind", ["edge_k1", "edge_k8"])
def test_row_per_cta_short_and_empty_rows(oracle_lib, kind):
    spec = _edge_spec(kind)
    inp = W.make_inputs(spec)
    rows = spec.batch * spec.num_kv_heads
    k = row_blocks(rows, spec.top_k, _sms())
    assert k == (1 if kind == "edge_k1" else 8), f"unexpected split (k = {k})"
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.select()
    dec.out.fill_(float("nan"))
    dec.lse.fill_(float("nan"))
    dec.decode()
    dec.check()
    torch.cuda.synchronize()
    # the sequence with no token: output 0, lse -inf, nothing selected
    assert (dec.n_selected[0] == 0).all()
    assert (dec.out[0] == 0).all() and torch.isneginf(dec.lse[0]).all()
    check = [r for r in range(rows) if r >= spec.num_kv_heads]
    PR.check_rows(inp, dec, check, oracle_lib, oracle_meta=oracle_lib.meta(inp["k_pool"], ids, vt))
