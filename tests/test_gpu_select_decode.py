"""One call per decode step: qskv_select_decode.

TinyServe query-aware page selection, s5.3 (the last page's metadata is
refreshed every step), s2.1-2.3 (min/max metadata, bound score, top-K) and
s3.2 (attention over the selected pages only).  The call is the scoring
launch (with the last-page refresh inside) followed by the decode launch;
when the rows go one row per k decode CTAs, the decode CTAs rank their own
row's scores before they stream its pages (no ranking launch), and with
k >= 2, when a CTA's share of a full row's pages fits its staging memory at
once, they also score the row themselves, the k CTAs of a row forming one
thread-block cluster (the step is one launch).

Checked, on cases with k = 1, k = 2, k = 4 and k = 8 scored in the decode
launch (d = 64 with fp32 q, d = 128 with bf16 q), k = 8 with shares too
long for that (the scoring launch runs; d = 64 and d = 128), k = 1 and a
batch too large for the split (the ranking launch runs): the refreshed
metadata bit for bit against
the oracle's scan of the new keys, scores and selections against the
oracle's, outputs against the oracle's attention over the selected pages,
and every result (metadata, scores, selection, out, lse) equal bit for bit
to the separate calls kv_meta_build, page_select and sparse_paged_decode;
repeated calls give identical results."""
import numpy as np
import pytest
import torch

import parity as PR
import query_aware_sparse_kv_gb300 as qskv
from query_aware_sparse_kv_gb300 import binding as B
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
    """CTAs per row the library picks (0: the stream-K split and a ranking launch)."""
    ctas = 2 * sms
    if rows <= 0 or rows > ctas or slots > 1024:
        return 0
    if rows >= sms:
        return 1
    k = min(ctas // rows, 8, slots // 4)
    return k if k >= 2 and rows * k >= sms else 0


def _case(kind):
    sms = _sms()
    if kind == "llama_k1":   # about 1.3 rows per SM, GQA 4, d = 128, lengths around top_k
        return W.spec_for("llama3_8b", batch=(4 * sms) // (3 * 8), seq_len_range=(200, 6000), max_pages=None)
    if kind == "gpt2_k2":    # 128 MHA rows, d = 64, fp32 q, 30 % of 512 pages
        return W.spec_for("gpt2_345m")
    if kind == "long_k8":    # 24 rows of 32-token pages
        return W.spec_for("long_context", batch=3, seq_len_range=(3000, 9000), max_pages=None, top_k=64)
    if kind == "long_rounds_k8":  # the long-context batch: 256-512 pages per CTA, d = 128
        return W.spec_for("long_context")
    if kind == "gpt2_rounds_k8":  # 32 MHA rows of 4096 pages: 512 per CTA, d = 64, fp32 q
        return W.spec_for("gpt2_345m", batch=2, seq_lens=(65536, 61000))
    if kind == "edges_k4":   # 64 rows of no, one, two and many pages, split over 4 CTAs each
        return W.spec_for("llama3_8b", batch=8, seq_lens=(0, 1, 15, 16, 17, 33, 3000, 5000), seq_len_range=None,
                          max_pages=None, top_k=64, kind="iid")
    if kind == "edges_k1":   # rows of no, one, two and many pages
        batch = -(-sms // 8) + 1
        lens = [0, 1, 15, 16, 17, 33] + [3000 + 97 * i for i in range(batch - 6)]
        return W.spec_for("llama3_8b", batch=batch, seq_lens=tuple(lens), seq_len_range=None, max_pages=None,
                          top_k=64, kind="iid")
    # more rows than two per SM: scoring, ranking launch, stream-K decode
    return W.spec_for("llama3_8b", batch=(2 * sms) // 8 + 8, seq_len_range=(100, 2500), max_pages=None, top_k=48,
                      kind="iid")


def _new_last_keys(inp, seed):
    """Overwrite the valid key rows of every non-empty sequence's last page
    with fresh values, in place; returns those pages' ids and valid counts."""
    g = torch.Generator().manual_seed(seed)
    ids, valid = W.last_pages(inp)
    keep = inp["n_pages"] > 0
    ids, valid = ids[keep], valid[keep]
    for p, v in zip(ids.tolist(), valid.tolist()):
        new = 3.0 * torch.randn((inp["k_pool"].shape[1], v, inp["k_pool"].shape[3]), generator=g)
        inp["k_pool"][p, :, :v] = new.to(inp["k_pool"].dtype)
    return ids.numpy(), valid.numpy()


def _nan_like(t):
    return torch.full_like(t, float("nan"))


KINDS = {"llama_k1": 1, "gpt2_k2": 2, "long_k8": 8, "long_rounds_k8": 8, "gpt2_rounds_k8": 8, "edges_k1": 1,
         "edges_k4": 4, "many_rows": 0}


@pytest.mark.parametrize("kind", list(KINDS))
def test_select_decode_matches_the_oracle_and_the_separate_calls(oracle_lib, kind):
    spec = _case(kind)
    inp = W.make_inputs(spec)
    rows = spec.batch * spec.num_kv_heads
    k = row_blocks(rows, spec.top_k, _sms())
    want = KINDS[kind]
    assert k == want, f"unexpected split (k = {k})"
    ids, vt = oracle_lib.all_pages(inp)
    old_meta = oracle_lib.meta(inp["k_pool"], ids, vt)

    # fused: metadata of every page from the old keys, then the step's new keys
    dec = qskv.from_inputs(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    last_ids, last_valid = _new_last_keys(inp, seed=11)
    dec.k_pool.copy_(inp["k_pool"].cuda())
    sc = torch.full((spec.batch, spec.num_kv_heads, inp["page_table"].shape[1]), float("nan"), device="cuda")
    dec.out.fill_(float("nan"))
    dec.lse.fill_(float("nan"))
    qskv.select_decode(dec.q, dec.k_pool, dec.v_pool, dec.meta, dec.page_table, dec.seq_lens, dec.top_k,
                       dec.selected, dec.n_selected, dec.out, dec.shape, dec.workspace, lse=dec.lse, scores=sc)
    dec.check()
    torch.cuda.synchronize()

    # against the oracle: metadata, scores, selection by the tie band, outputs
    new_meta = oracle_lib.meta(inp["k_pool"], last_ids, last_valid, out=old_meta.copy())
    PR.assert_meta_equal(dec.meta, new_meta, ids)
    check = list(range(rows)) if rows <= 256 else PR.sample_rows(rows, 96, seed=5)
    if kind.startswith("edges"):
        check = [r for r in check if r >= spec.num_kv_heads]
    PR.check_rows(inp, dec, check, oracle_lib, oracle_meta=new_meta, check_scores=sc)
    if kind.startswith("edges"):  # the sequence with no token: nothing selected, output 0, lse -inf
        assert (dec.n_selected[0] == 0).all()
        assert (dec.out[0] == 0).all() and torch.isneginf(dec.lse[0]).all()

    # the separate calls on the same state give the same bits
    sep = qskv.from_inputs(inp)
    sep.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    sep.build_meta(torch.from_numpy(last_ids).cuda(), torch.from_numpy(last_valid).cuda())
    sc2 = _nan_like(sc)
    sep.select(scores=sc2)
    sep.out.fill_(float("nan"))
    sep.lse.fill_(float("nan"))
    sep.decode()
    sep.check()
    torch.cuda.synchronize()
    assert torch.equal(sep.meta, dec.meta)
    assert torch.equal(sep.selected, dec.selected) and torch.equal(sep.n_selected, dec.n_selected)
    nb = inp["n_pages"].long()
    for b in range(spec.batch):
        assert torch.equal(sc[b, :, :nb[b]], sc2[b, :, :nb[b]]), f"scores of sequence {b} differ"
    assert torch.equal(sep.out, dec.out) and torch.equal(sep.lse, dec.lse)

    # repeated steps (the refresh of unchanged keys is idempotent) and the
    # engine's step, which takes this call, give the same bits again
    first = (dec.out.clone(), dec.lse.clone(), dec.selected.clone())
    for _ in range(2):
        dec.out.fill_(float("nan"))
        dec.selected.fill_(-7)
        dec.step(refresh_last=True)
        dec.check()
        torch.cuda.synchronize()
        assert torch.equal(dec.out, first[0]) and torch.equal(dec.lse, first[1])
        assert torch.equal(dec.selected, first[2])


def test_select_decode_needs_bf16_kv():
    inp = W.make_inputs(W.spec_for("tiny"))  # fp32 KV
    dec = qskv.from_inputs(inp)
    with pytest.raises(qskv.QskvError) as e:
        B.select_decode(dec.q, dec.k_pool, dec.v_pool, dec.meta, dec.page_table, dec.seq_lens, dec.top_k,
                        dec.selected, dec.n_selected, dec.out, dec.shape, dec.workspace, lse=dec.lse)
    assert e.value.status == 2
    np.testing.assert_equal(dec.can_refresh_in_select, False)  # the engine takes the separate calls there


@pytest.mark.parametrize("kind", ["gpt2_k2", "long_k8"])
def test_one_launch_step_flags_device_index_errors(oracle_lib, kind):
    """The one-launch step (the decode CTAs of a row score it): an out-of-pool
    page id and an out-of-range sequence length are flagged
    (QSKV_ERR_DEVICE_INDEX), skipped, and the call stays usable; after the
    table is repaired the next step matches the oracle again."""
    spec = _case(kind)
    inp = W.make_inputs(spec)
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.check()
    n_pool = inp["k_pool"].shape[0]
    good = dec.page_table[0, 3].item()
    dec.page_table[0, 3] = n_pool + 5
    dec.step(refresh_last=True)
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    assert torch.isfinite(dec.out).all()
    dec.page_table[0, 3] = good
    seq0 = dec.seq_lens[1].item()
    dec.seq_lens[1] = dec.page_table.shape[1] * spec.page_size + 1  # beyond the table row
    dec.step(refresh_last=True)
    with pytest.raises(qskv.QskvError) as e:
        dec.check()
    assert e.value.status == 5
    dec.seq_lens[1] = seq0
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.step(refresh_last=True)
    dec.check()
    torch.cuda.synchronize()
    PR.check_rows(inp, dec, PR.sample_rows(spec.batch * spec.num_kv_heads, 12, seed=3), oracle_lib,
                  oracle_meta=oracle_lib.meta(inp["k_pool"], ids, vt))


def test_one_launch_step_in_a_cuda_graph(oracle_lib):
    """The clustered one-launch step captured in a CUDA graph replays to the
    same bits as the eager call."""
    spec = _case("gpt2_k2")
    inp = W.make_inputs(spec)
    dec = qskv.from_inputs(inp)
    ids, vt = oracle_lib.all_pages(inp)
    dec.build_meta(torch.from_numpy(ids).cuda(), torch.from_numpy(vt).cuda())
    dec.step(refresh_last=True)
    dec.check()
    torch.cuda.synchronize()
    ref = (dec.out.clone(), dec.lse.clone(), dec.selected.clone())
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dec.step(refresh_last=True)
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        dec.step(refresh_last=True)
    for _ in range(2):
        dec.out.fill_(float("nan"))
        dec.selected.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        dec.check()
        assert torch.equal(dec.out, ref[0]) and torch.equal(dec.lse, ref[1]) and torch.equal(dec.selected, ref[2])
