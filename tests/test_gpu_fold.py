"""Split rows folded inside the decode grid.

When one warp can load all the partial outputs (o, log-sum-exp) of a split
row in one round, the last decode warp to finish the row folds them (a
per-row ticket counter decides which warp is last; no warp waits).  Other
split rows go to the merge kernel.  Both paths must give the oracle's attention (Quail AI-SQL engine
article: partial attention combined by log-sum-exp rescaling), and the
per-row counters must be back at zero after every call, so repeated calls on
one workspace keep giving the same result."""
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


# A split row is folded in the grid when its pieces fit one round of loads of
# one warp: pieces x G x D / 128 <= 16 (the decode grid has 1824 warps).
CASES = {
    # GPT2-345M-like at full size (fp32 q, d=64, MHA): 19712 units, 11 per warp,
    # rows in 15 pieces of 64 floats -> folded in the grid
    "gpt2_fold": W.spec_for("gpt2_345m"),
    # GQA 4, d=128, top-12 of short rows: 7680 units, 5 per warp, rows in at most
    # 4 pieces of 4 x 128 floats -> folded in the grid
    "llama_fold": W.spec_for("llama3_8b", batch=80, seq_len_range=(300, 3000), max_pages=None, top_k=12),
    # GQA 4, d=128, top-64: rows in ~23 pieces -> merge kernel
    "llama_merge": W.spec_for("llama3_8b", batch=8, seq_len_range=(1500, 9000), max_pages=None, top_k=64),
    # 4 rows of 512 pages of 32 tokens, each over ~250 warps -> merge kernel
    "long_merge": W.spec_for("long_context", batch=1, seq_len_range=(40000, 60000), max_pages=None, top_k=512,
                             num_q_heads=16, num_kv_heads=4),
}


@pytest.mark.parametrize("name", list(CASES))
def test_split_rows_match_the_oracle_on_repeated_calls(oracle_lib, name):
    inp = W.make_inputs(CASES[name])
    spec = inp["spec"]
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.select()
    dec.check()
    rows = list(range(spec.batch * spec.num_kv_heads))
    o_meta = oracle_lib.meta(inp["k_pool"], ids, vt)
    first = None
    for it in range(3):
        dec.out.fill_(float("nan"))
        dec.lse.fill_(float("nan"))
        dec.decode()
        dec.check()
        torch.cuda.synchronize()
        if first is None:
            PR.check_rows(inp, dec, rows, oracle_lib, oracle_meta=o_meta)
            first = (dec.out.clone(), dec.lse.clone())
        else:
            # same inputs, same workspace: bit-identical results every call
            assert torch.equal(dec.out, first[0]) and torch.equal(dec.lse, first[1]), f"call {it} differs"
