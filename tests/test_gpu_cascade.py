"""GPU parity of the shared-prefix cascade decode: the prefix attended once
per KV head on the tensor cores, each row's own pages through the paged
decode, merged by log-sum-exp.  The result is dense attention over every
token of each sequence, so it is compared with the oracle's dense attention
(same tolerance as the paged decode: max-abs 1e-2 with a bf16 cache)."""
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


def _cascade(inputs, prefix_pages=None):
    spec = inputs["spec"]
    pp = spec.prefix_pages if prefix_pages is None else prefix_pages
    dec = qskv.from_inputs(inputs, top_k=None, prefix_pages=pp)
    dec.decode()
    dec.check()
    torch.cuda.synchronize()
    return dec


def _check(inputs, dec, oracle, rows=None):
    spec = inputs["spec"]
    n_rows = spec.batch * spec.num_kv_heads
    PR.check_rows(inputs, dec, range(n_rows) if rows is None else rows, oracle, dense=True)


def _spec(G=4, d=128, P=16, batch=6, prefix=9, suffix=3, seq=None, q=torch.bfloat16, seed=11):
    return W.Spec(name="cascade", batch=batch, num_q_heads=2 * G, num_kv_heads=2, head_dim=d, page_size=P,
                  top_k=None, q_dtype=q, kv_dtype=torch.bfloat16, kind="shared_prefix", prefix_pages=prefix,
                  suffix_pages=suffix, seq_lens=seq, seed=seed)


def _ragged(batch, prefix, suffix, P, seed=0):
    """Sequence lengths from exactly the prefix to prefix + suffix pages,
    most ending inside a page."""
    rng = np.random.default_rng(seed)
    lo, hi = prefix * P, (prefix + suffix) * P
    s = rng.integers(lo, hi + 1, size=batch)
    s[0], s[-1] = lo, hi
    return tuple(int(x) for x in s)


def test_small_shared_prefix(oracle_lib):
    inp = W.make_inputs(W.spec_for("shared_prefix", batch=6, prefix_pages=8, suffix_pages=3))
    _check(inp, _cascade(inp), oracle_lib)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("P", [16, 32])
def test_shape_sweep(oracle_lib, G, d, P):
    # a prefix that is not a whole number of 128-key blocks, ragged rows,
    # and (G = 8) more than one 128-row query tile with a ragged last tile
    batch = 20 if G == 8 else 7
    prefix = 9 if P == 16 else 5
    spec = _spec(G=G, d=d, P=P, batch=batch, prefix=prefix, suffix=3, seq=_ragged(batch, prefix, 3, P, seed=G + d + P),
                 seed=G * 1000 + d + P)
    inp = W.make_inputs(spec)
    _check(inp, _cascade(inp), oracle_lib)


def test_fp32_queries(oracle_lib):
    for d in (64, 128):
        spec = _spec(d=d, batch=5, prefix=10, suffix=2, seq=_ragged(5, 10, 2, 16, seed=d), q=torch.float32, seed=d)
        inp = W.make_inputs(spec)
        _check(inp, _cascade(inp), oracle_lib)


def test_long_prefix_many_splits(oracle_lib):
    # few rows and a 2048-token prefix: the prefix is split over many CTAs
    spec = _spec(G=4, batch=2, prefix=128, suffix=4, seq=(128 * 16 + 3, 132 * 16), seed=21)
    inp = W.make_inputs(spec)
    _check(inp, _cascade(inp), oracle_lib)


def test_persistent_prefix_grid_all_rows(oracle_lib):
    """The prefix grid is persistent (about 43 % of the SMs): at 64 sequences,
    8 KV heads and a 64-page prefix there are 128 work items, so each prefix
    CTA takes two of them in turn (mbarriers re-armed in between) while the
    paged decode runs on the other SMs.  Every row is checked."""
    spec = W.Spec(name="cascade", batch=64, num_q_heads=32, num_kv_heads=8, head_dim=128, page_size=16,
                  top_k=None, q_dtype=torch.bfloat16, kv_dtype=torch.bfloat16, kind="shared_prefix",
                  prefix_pages=64, suffix_pages=4, seq_lens=_ragged(64, 64, 4, 16, seed=5), seed=24)
    inp = W.make_inputs(spec)
    _check(inp, _cascade(inp), oracle_lib)


def test_prefix_is_the_whole_sequence(oracle_lib):
    # no private pages at all: max_pages == prefix_pages, the paged decode has no work
    spec = _spec(batch=4, prefix=6, suffix=0, seq=(96,) * 4, seed=22)
    inp = W.make_inputs(spec)
    assert inp["max_pages"] == 6
    _check(inp, _cascade(inp), oracle_lib)


def test_zero_prefix_is_plain_dense(oracle_lib):
    spec = _spec(batch=4, prefix=5, suffix=2, seq=_ragged(4, 5, 2, 16, seed=3), seed=23)
    inp = W.make_inputs(spec)
    dec = _cascade(inp, prefix_pages=0)
    _check(inp, dec, oracle_lib)


def test_matches_the_paged_dense_decode(oracle_lib):
    spec = _spec(G=4, batch=40, prefix=12, suffix=4, seq=_ragged(40, 12, 4, 16, seed=5), seed=24)
    inp = W.make_inputs(spec)
    dec = _cascade(inp)
    plain = qskv.from_inputs(inp, top_k=None)
    plain.decode()
    plain.check()
    assert (dec.out - plain.out).abs().max().item() <= 1e-2
    assert (dec.lse - plain.lse).abs().max().item() <= 1e-2
    _check(inp, dec, oracle_lib, rows=PR.sample_rows(80, 12, seed=2))


def test_repeat_calls_are_identical(oracle_lib):
    spec = _spec(G=4, batch=9, prefix=20, suffix=3, seq=_ragged(9, 20, 3, 16, seed=6), seed=25)
    inp = W.make_inputs(spec)
    dec = _cascade(inp)
    out1, lse1 = dec.out.clone(), dec.lse.clone()
    for _ in range(3):
        dec.decode()
    dec.check()
    assert torch.equal(out1, dec.out) and torch.equal(lse1, dec.lse)


def test_contract_violations_are_flagged(oracle_lib):
    spec = _spec(batch=4, prefix=6, suffix=2, seq=_ragged(4, 6, 2, 16, seed=7), seed=26)
    inp = W.make_inputs(spec)
    dec = qskv.from_inputs(inp, top_k=None, prefix_pages=6)
    # row 2 names a different page inside the prefix
    good = dec.page_table[2, 3].item()
    dec.page_table[2, 3] = dec.page_table[1, 7]
    dec.decode()
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    dec.page_table[2, 3] = good
    # row 1 shorter than the prefix
    keep = dec.seq_lens[1].item()
    dec.seq_lens[1] = 6 * 16 - 1
    dec.decode()
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    dec.seq_lens[1] = keep
    # a prefix page outside the pool
    n_pool = inp["k_pool"].shape[0]
    saved = dec.page_table[:, 0].clone()
    dec.page_table[:, 0] = n_pool + 3
    dec.decode()
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    dec.page_table[:, 0] = saved
    dec.decode()
    dec.check()
    torch.cuda.synchronize()
    _check(inp, dec, oracle_lib)


def test_host_checks():
    spec = _spec(batch=2, prefix=4, suffix=1, seq=(70, 80), seed=27)
    inp = W.make_inputs(spec)
    dec = qskv.from_inputs(inp, top_k=None, prefix_pages=4)
    for bad_prefix in (-1, dec.shape.max_pages + 1):
        with pytest.raises(qskv.QskvError) as e:
            qskv.cascade_paged_decode(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seq_lens, dec.out,
                                      dec.shape, dec.workspace, bad_prefix)
        assert e.value.status == 1
    with pytest.raises(qskv.QskvError) as e:  # too small a workspace
        qskv.cascade_paged_decode(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seq_lens, dec.out, dec.shape,
                                  dec.workspace[:256], 4)
    assert e.value.status == 3
    kf, vf = dec.k_pool.float(), dec.v_pool.float()
    with pytest.raises(qskv.QskvError) as e:  # fp32 KV
        qskv.cascade_paged_decode(dec.q, kf, vf, dec.page_table, dec.seq_lens, dec.out, dec.shape, dec.workspace, 4)
    assert e.value.status == 2


def test_cuda_graph_capture(oracle_lib):
    spec = _spec(G=4, batch=12, prefix=16, suffix=3, seq=_ragged(12, 16, 3, 16, seed=8), seed=28)
    inp = W.make_inputs(spec)
    dec = _cascade(inp)
    ref = dec.out.clone()
    replay = dec.capture_step(dec.q)
    dec.out.zero_()
    replay()
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(ref, dec.out)


def test_full_size_shared_prefix_sampled(oracle_lib):
    inp = W.make_inputs(W.spec_for("shared_prefix"))
    dec = _cascade(inp)
    assert torch.isfinite(dec.out).all() and torch.isfinite(dec.lse).all()
    spec = inp["spec"]
    _check(inp, dec, oracle_lib, rows=PR.sample_rows(spec.batch * spec.num_kv_heads, 10, seed=3))
