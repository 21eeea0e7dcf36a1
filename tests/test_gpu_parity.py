"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Rules (tests/parity.py): metadata bit-exact; selection equal up to the
1e-3 tie band around the K-th score; outputs within max-abs 1e-4 (fp32 KV)
or 1e-2 (bf16 KV) of oracle attention over the GPU's own selection.
"""
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


def _run(inputs, oracle, top_k="spec", rows=None, scores=True, dense=False):
    """Meta for every referenced page, select (with scores), decode; then
    compare `rows` (default all) with the oracle."""
    dec = qskv.from_inputs(inputs, top_k=top_k)
    ids, vt = oracle.all_pages(inputs)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    sc = None
    if dec.top_k is not None and not dense:
        sc = torch.full(tuple(dec.selected.shape[:2]) + (inputs["page_table"].shape[1],), float("nan"),
                        device="cuda") if scores else None
        dec.select(scores=sc)
    dec.decode(dense=dense)
    dec.check()
    torch.cuda.synchronize()
    o_meta = oracle.meta(inputs["k_pool"], ids, vt)
    PR.assert_meta_equal(dec.meta, o_meta, ids)
    spec = inputs["spec"]
    n_rows = spec.batch * spec.num_kv_heads
    PR.check_rows(inputs, dec, range(n_rows) if rows is None else rows, oracle, o_meta, sc, dense=dense)
    return dec


SMALL = {
    "tiny": W.spec_for("tiny"),
    "gpt2_small": W.spec_for("gpt2_345m", batch=2, seq_lens=(1024, 1000), top_k=20),
    "llama_small": W.spec_for("llama3_8b", batch=3, seq_len_range=(300, 1500), max_pages=None, top_k=16),
    "long_small": W.spec_for("long_context", batch=2, seq_len_range=(2000, 5000), max_pages=None, top_k=16),
    "prefix_small": W.spec_for("shared_prefix", batch=6, prefix_pages=8, suffix_pages=3),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_small_configs_end_to_end(oracle_lib, name):
    _run(W.make_inputs(SMALL[name]), oracle_lib)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("P", [16, 32])
@pytest.mark.parametrize("kv", [torch.bfloat16, torch.float32])
def test_shape_sweep(oracle_lib, G, d, P, kv):
    q = torch.float32 if (G + d + P) % 2 == 0 and kv == torch.bfloat16 and G == 2 else kv
    spec = W.Spec(name="sweep", batch=3, num_q_heads=2 * G, num_kv_heads=2, head_dim=d, page_size=P,
                  seq_lens=(P * 9 + 5, 3, P * 4), top_k=5, q_dtype=q, kv_dtype=kv, kind="page_offset",
                  extra_pool_pages=2, seed=G * 100 + d + P)
    _run(W.make_inputs(spec), oracle_lib)


def test_fp32_query_with_bf16_cache(oracle_lib):
    spec = W.spec_for("gpt2_345m", batch=2, seq_lens=(700, 333), top_k=9, num_q_heads=8, num_kv_heads=2,
                      head_dim=128)
    _run(W.make_inputs(spec), oracle_lib)


def test_dense_equals_oracle_dense(oracle_lib):
    spec = SMALL["llama_small"]
    _run(W.make_inputs(spec), oracle_lib, dense=True)


def test_top_k_covers_every_page(oracle_lib):
    spec = W.spec_for("llama3_8b", batch=2, seq_len_range=(100, 400), max_pages=None, top_k=64)
    inp = W.make_inputs(spec)
    dec = _run(inp, oracle_lib)
    nb = inp["n_pages"].numpy()
    sel = dec.selected.cpu().numpy()
    for b in range(2):
        assert sel[b, 0, :nb[b]].tolist() == list(range(nb[b]))


def test_top1(oracle_lib):
    spec = W.spec_for("llama3_8b", batch=2, seq_len_range=(500, 900), max_pages=None, top_k=1)
    _run(W.make_inputs(spec), oracle_lib)


def test_short_and_empty_sequences(oracle_lib):
    spec = W.Spec(name="edge", batch=4, num_q_heads=8, num_kv_heads=2, head_dim=128, page_size=16,
                  seq_lens=(1, 15, 17, 40), top_k=2, kind="iid", seed=5)
    inp = W.make_inputs(spec)
    _run(inp, oracle_lib)
    # a sequence with no token: output 0, lse -inf, nothing selected
    inp["seq_lens"][1] = 0
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.step()
    dec.check()
    assert (dec.n_selected[1] == 0).all()
    assert (dec.out[1] == 0).all() and torch.isneginf(dec.lse[1]).all()
    PR.check_rows(inp, dec, [0, 1, 4, 5, 6, 7], oracle_lib, oracle_lib.meta(inp["k_pool"], ids, vt))


def test_ties_take_the_lower_page_index(oracle_lib):
    """Logical pages that alias one physical page have bit-identical scores;
    the kept ones must be the lowest-indexed (the oracle's rule)."""
    spec = W.Spec(name="ties", batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, page_size=16,
                  seq_lens=(16 * 12,), top_k=5, kind="iid", seed=8)
    inp = W.make_inputs(spec)
    t = inp["page_table"]
    t[0, 1::2] = t[0, 0]  # pages 0, 1, 3, 5, ... share one physical page
    dec = _run(inp, oracle_lib)
    res = oracle_lib.step(inp)
    assert dec.selected[0, 0].cpu().tolist() == res["selected"][0].tolist()


def test_zero_and_negative_zero_keys(oracle_lib):
    spec = W.Spec(name="zeros", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64, page_size=16,
                  seq_lens=(70, 64), top_k=3, kind="iid", seed=9)
    inp = W.make_inputs(spec)
    kp = inp["k_pool"]
    kp[:, :, :, ::3] = 0.0
    kp[:, :, :, 1::3] = -0.0
    _run(inp, oracle_lib)


def test_same_row_alone_and_in_a_batch(oracle_lib):
    """The split of a row over warps depends on the batch; the result must not."""
    spec = W.spec_for("llama3_8b", batch=8, seq_len_range=(3000, 6000), max_pages=None, top_k=64)
    inp = W.make_inputs(spec)
    dec = _run(inp, oracle_lib, rows=[0, 1, 2])
    one = {k: (v[:1].contiguous() if k in ("q", "page_table", "seq_lens", "n_pages") else v) for k, v in inp.items()}
    one["spec"] = W.spec_for("llama3_8b", batch=1, seq_lens=(int(inp["seq_lens"][0]),), max_pages=None, top_k=64)
    dec1 = _run(one, oracle_lib)
    assert torch.equal(dec1.selected[0], dec.selected[0])
    assert (dec1.out[0] - dec.out[0]).abs().max().item() <= 1e-2


def test_repeat_calls_are_identical(oracle_lib):
    inp = W.make_inputs(SMALL["llama_small"])
    dec = _run(inp, oracle_lib)
    out1, lse1, sel1 = dec.out.clone(), dec.lse.clone(), dec.selected.clone()
    for _ in range(3):
        dec.select()
        dec.decode()
    dec.check()
    assert torch.equal(sel1, dec.selected) and torch.equal(out1, dec.out) and torch.equal(lse1, dec.lse)


def test_device_index_errors_are_flagged_not_fatal(oracle_lib):
    inp = W.make_inputs(SMALL["llama_small"])
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.check()
    n_pool = inp["k_pool"].shape[0]
    good = dec.page_table[0, 0].item()
    dec.page_table[0, 0] = n_pool + 7  # out of the pool
    dec.step()
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    assert torch.isfinite(dec.out).all()
    dec.page_table[0, 0] = good
    dec.step()
    dec.check()
    PR.check_rows(inp, dec, range(8), oracle_lib, oracle_lib.meta(inp["k_pool"], ids, vt))
    # metadata build with a bad id and a bad valid-token count
    bad_ids = torch.tensor([0, n_pool], dtype=torch.int32, device="cuda")
    bad_valid = torch.tensor([17, 3], dtype=torch.int32, device="cuda")
    dec.build_meta(bad_ids, bad_valid)
    with pytest.raises(qskv.QskvError):
        dec.check()
    dec.check()  # flags were cleared


def test_host_checks_reject_bad_arguments():
    inp = W.make_inputs(SMALL["llama_small"])
    dec = qskv.from_inputs(inp)
    with pytest.raises(qskv.QskvError) as e:
        qskv.sparse_paged_decode(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seq_lens, dec.out, dec.shape,
                                 dec.workspace[:64])
    assert e.value.status == 3
    shifted = torch.empty(dec.out.numel() + 4, device="cuda")[1:1 + dec.out.numel()].view_as(dec.out)
    with pytest.raises(qskv.QskvError) as e:
        qskv.sparse_paged_decode(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seq_lens, shifted, dec.shape,
                                 dec.workspace)
    assert e.value.status == 1
    with pytest.raises(qskv.QskvError) as e:
        qskv.page_select(dec.q, dec.meta, dec.page_table, dec.seq_lens, 0, dec.selected, dec.n_selected, dec.shape,
                         dec.workspace)
    assert e.value.status == 1


def test_cuda_graph_capture_of_a_step(oracle_lib):
    inp = W.make_inputs(SMALL["llama_small"])
    dec = _run(inp, oracle_lib)
    ref = dec.out.clone()
    dec.out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dec.step()  # warm-up outside capture (sets kernel attributes)
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        dec.step()
    dec.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    dec.check()
    assert torch.equal(ref, dec.out)


# ---------------------------------------------------------------- full size --
FULL_ROWS = 10


@pytest.mark.parametrize("name", ["tiny", "gpt2_345m", "llama3_8b", "long_context", "shared_prefix"])
def test_full_size_config_sampled(oracle_lib, name):
    """The named workloads at their full sizes: every row is checked for
    structure (size, order, range, finiteness); sampled rows against the oracle."""
    inp = W.make_inputs(W.spec_for(name))
    spec = inp["spec"]
    n_rows = spec.batch * spec.num_kv_heads
    rows = PR.sample_rows(n_rows, FULL_ROWS, seed=1)
    dec = _run(inp, oracle_lib, rows=rows, scores=True)
    assert torch.isfinite(dec.out).all() and torch.isfinite(dec.lse).all()
    if spec.top_k is not None:
        nb = inp["n_pages"].cuda()
        want = torch.clamp(nb, max=spec.top_k)[:, None].expand_as(dec.n_selected)
        assert torch.equal(dec.n_selected, want.to(torch.int32))
        sel = dec.selected
        assert (sel[..., 1:] > sel[..., :-1]).all()  # every row keeps >= top_k pages here
        assert (sel >= 0).all() and (sel < nb[:, None, None]).all()


@pytest.mark.parametrize("case", ["centroid_lossy", "cascade"])
def test_zero_copy_step_matches_the_device_path(oracle_lib, case):
    """The zero-copy captured step (kernels reading q from and writing out to
    pinned host memory) gives bit-identical outputs to the device-resident
    calls, for the Block Top-K scorer with the lossy top-K and for the
    shared-prefix cascade (whose prefix kernel reads q too)."""
    if case == "cascade":
        spec = W.spec_for("shared_prefix", batch=6, prefix_pages=9, suffix_pages=4)
        inp = W.make_inputs(spec)
        dec = qskv.from_inputs(inp, top_k=None, prefix_pages=9)
    else:
        inp = W.make_inputs(SMALL["long_small"])
        dec = qskv.from_inputs(inp, scorer="centroid", approx_epsilon=0.05, approx_seed=4)
        ids, vt = oracle_lib.all_pages(inp)
        dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    qv = W.q_variants(inp, 2)
    want = []
    for v in range(2):
        dec.step(q=qv[v].cuda())
        torch.cuda.synchronize()
        want.append(dec.out.cpu().clone())
    q_host = [qv[v].pin_memory() for v in range(2)]
    out_host = torch.zeros(dec.out.shape, dtype=dec.out.dtype).pin_memory()
    graphs = [dec.capture_step(torch.empty_like(dec.q), q_host=q_host[v], out_host=out_host) for v in range(2)]
    for v in (0, 1, 0):
        out_host.zero_()
        graphs[v]()
        dec.wait()  # event poll: returns only once the output is in host memory
        assert torch.equal(out_host, want[v])
    dec.check()


@pytest.mark.parametrize("zero_copy", [True, False])
def test_captured_step_with_host_copies(oracle_lib, zero_copy):
    """capture_step(q_host=, out_host=): one graph takes the query from pinned
    memory, runs the step and puts the output in pinned memory (the kernels
    reading and writing host memory directly, or copy nodes); replays with two
    different queries give the outputs of the direct calls."""
    inp = W.make_inputs(SMALL["llama_small"])
    dec = _run(inp, oracle_lib)
    qv = W.q_variants(inp, 2)
    want = []
    for v in range(2):
        dec.step(q=qv[v].cuda())
        torch.cuda.synchronize()
        want.append(dec.out.cpu().clone())
    q_dev = torch.empty_like(dec.q)
    out_host = torch.zeros(dec.out.shape, dtype=dec.out.dtype).pin_memory()
    q_host = [qv[v].pin_memory() for v in range(2)]
    graphs = [dec.capture_step(q_dev, q_host=q_host[v], out_host=out_host, zero_copy=zero_copy) for v in range(2)]
    for v in (1, 0, 1):
        out_host.zero_()
        graphs[v]()
        torch.cuda.current_stream().synchronize()
        assert torch.equal(out_host, want[v])
    dec.check()
    with pytest.raises(ValueError):
        dec.capture_step(q_dev, q_host=qv[0])  # not pinned
    with pytest.raises(ValueError):
        dec.capture_step(q_dev, q_host=qv[0][:1].pin_memory())  # wrong shape
