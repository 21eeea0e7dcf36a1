"""GPU parity of the Block Top-K scorer (Vortex sparse-attention digest,
method overview item 1): per-page fp32 mean keys, scores q . centroid (best
head of the group), then the shared top-K and sparse decode.

Rules: centroids within the fp32 summation bound of the oracle's exact
means; scores within the propagated bound; selection by the tie-band rule
on the oracle's centroid scores; outputs against oracle attention over the
GPU's own selection (max-abs 1e-4 fp32 KV, 1e-2 bf16 KV)."""
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


def _run(inputs, oracle, rows=None, scores=True, top_k="spec"):
    dec = qskv.from_inputs(inputs, top_k=top_k, scorer="centroid")
    ids, vt = oracle.all_pages(inputs)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    sc = None
    if scores:
        sc = torch.full(tuple(dec.selected.shape[:2]) + (inputs["page_table"].shape[1],), float("nan"),
                        device="cuda")
    dec.select(scores=sc)
    dec.decode()
    dec.check()
    torch.cuda.synchronize()
    o_cent = oracle.centroids(inputs["k_pool"], ids, vt)
    tol = PR.centroid_tolerance(inputs["k_pool"], ids, vt)
    PR.assert_centroids_close(dec.meta, o_cent, tol, ids)
    spec = inputs["spec"]
    n_rows = spec.batch * spec.num_kv_heads
    PR.check_rows(inputs, dec, range(n_rows) if rows is None else rows, oracle, o_cent, sc, scorer="centroid",
                  cent_tol=tol)
    return dec


SMALL = {
    "tiny": W.spec_for("tiny"),
    "gpt2_small": W.spec_for("gpt2_345m", batch=2, seq_lens=(1024, 1000), top_k=20),
    "llama_small": W.spec_for("llama3_8b", batch=3, seq_len_range=(300, 1500), max_pages=None, top_k=16),
    "long_small": W.spec_for("long_context", batch=2, seq_len_range=(2000, 5000), max_pages=None, top_k=16),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_configs_end_to_end(oracle_lib, name):
    _run(W.make_inputs(SMALL[name]), oracle_lib)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("kv", [torch.bfloat16, torch.float32])
def test_shape_sweep(oracle_lib, G, d, P, kv):
    q = torch.float32 if G in (1, 8) else torch.bfloat16
    spec = W.Spec(name="sweep", batch=3, num_q_heads=2 * G, num_kv_heads=2, head_dim=d, page_size=P,
                  seq_lens=(P * 41 + 5, 3, P * 4), top_k=5, q_dtype=q, kv_dtype=kv, kind="page_offset",
                  extra_pool_pages=2, seed=G * 100 + d + P + 7)
    _run(W.make_inputs(spec), oracle_lib)


def test_centroid_workload_keeps_the_aligned_pages(oracle_lib):
    """On the centroid workload (keys around 64 centroids per KV head, q near
    one) the selected pages are the ones whose centroid is q's: the GPU keeps
    the same set as the oracle up to the tie band, and the kept pages carry
    almost all the attention mass."""
    spec = W.spec_for("long_context", batch=2, seq_len_range=(4000, 6000), max_pages=None, top_k=32)
    inp = W.make_inputs(spec)
    dec = _run(inp, oracle_lib)
    assert (dec.n_selected == 32).all()


def test_flags_bad_page_ids(oracle_lib):
    inp = W.make_inputs(SMALL["llama_small"])
    dec = qskv.from_inputs(inp, scorer="centroid")
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.check()
    n_pool = inp["k_pool"].shape[0]
    good = dec.page_table[0, 1].item()
    dec.page_table[0, 1] = n_pool + 5
    dec.step()
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    assert torch.isfinite(dec.out).all()
    dec.page_table[0, 1] = good
    dec.build_meta(torch.tensor([0, n_pool], dtype=torch.int32, device="cuda"),
                   torch.tensor([4, 4], dtype=torch.int32, device="cuda"))
    with pytest.raises(qskv.QskvError):
        dec.check()


def test_repeat_calls_are_identical(oracle_lib):
    inp = W.make_inputs(SMALL["long_small"])
    dec = _run(inp, oracle_lib)
    cent1, sel1, out1 = dec.meta.clone(), dec.selected.clone(), dec.out.clone()
    ids, vt = oracle_lib.all_pages(inp)
    for _ in range(2):
        dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
        dec.select()
        dec.decode()
    dec.check()
    assert torch.equal(cent1, dec.meta) and torch.equal(sel1, dec.selected) and torch.equal(out1, dec.out)


def test_cuda_graph_step(oracle_lib):
    inp = W.make_inputs(SMALL["llama_small"])
    dec = _run(inp, oracle_lib)
    ref_sel, ref_out = dec.selected.clone(), dec.out.clone()
    replay = dec.capture_step(dec.q)
    dec.out.zero_()
    replay()
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(ref_sel, dec.selected) and torch.equal(ref_out, dec.out)


@pytest.mark.parametrize("name", ["llama3_8b", "long_context"])
def test_full_size_sampled(oracle_lib, name):
    inp = W.make_inputs(W.spec_for(name))
    spec = inp["spec"]
    rows = PR.sample_rows(spec.batch * spec.num_kv_heads, 8, seed=4)
    dec = _run(inp, oracle_lib, rows=rows)
    assert torch.isfinite(dec.out).all()
    nb = inp["n_pages"].cuda()
    want = torch.clamp(nb, max=spec.top_k)[:, None].expand_as(dec.n_selected)
    assert torch.equal(dec.n_selected, want.to(torch.int32))
