"""One row per decode CTA.

When the (sequence, KV head) rows fit one wave of decode CTAs (at least one
and at most two per SM, d = 128, bf16 KV), CTA r decodes row r alone: its
warps take the row's selected pages from a shared-memory counter and the
warps' partial results are folded in the CTA by log-sum-exp rescaling
(Quail AI-SQL engine article: partial attention combined as in flash
decoding), with no merge kernel.  Sparse rows -- some with fewer pages than
top_k -- and a dense batch are checked row by row against the oracle, and
repeated calls on one workspace give identical results."""
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


def _case(kind):
    sms = _sms()
    if kind == "sparse_mid":    # about 1.3 rows per SM, lengths around top_k
        return W.spec_for("llama3_8b", batch=(4 * sms) // (3 * 8), seq_len_range=(200, 6000), max_pages=None)
    if kind == "sparse_low":    # one row per SM (the smallest row count of the mode)
        return W.spec_for("llama3_8b", batch=-(-sms // 8), seq_len_range=(1500, 4000), max_pages=None, top_k=64)
    if kind == "sparse_high":   # two rows per SM (the largest)
        return W.spec_for("llama3_8b", batch=(2 * sms) // 8, seq_len_range=(300, 2500), max_pages=None, top_k=40)
    return W.spec_for("llama3_8b", batch=(4 * sms) // (3 * 8), seq_len_range=(100, 1500), max_pages=None,
                      top_k=None)


@pytest.mark.parametrize("kind", ["sparse_mid", "sparse_low", "sparse_high", "dense"])
def test_row_per_cta_matches_the_oracle(oracle_lib, kind):
    spec = _case(kind)
    rows = spec.batch * spec.num_kv_heads
    assert _sms() <= rows <= 2 * _sms(), "the case must fall in the one-row-per-CTA range"
    inp = W.make_inputs(spec)
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
