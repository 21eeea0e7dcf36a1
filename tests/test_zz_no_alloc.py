"""The decode entry point that allocates nothing.

Some callers cannot allocate device memory at decode time: serving engines
whose memory planner hands out all of HBM up front and forbids further
cudaMalloc calls, or latency-critical loops where the allocator (which may
synchronise the device) must not be called.  qskv_sparse_paged_decode_noalloc
serves them: it takes the same inputs and outputs as qskv_sparse_paged_decode
but keeps its scratch in a fixed 8 MiB array built into the library.  Its
output is checked against the workspace entry point and, row by row, against
the CPU oracle.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""
import ctypes

import pytest
import torch

import parity as PR
import query_aware_sparse_kv_gb300 as qskv
from query_aware_sparse_kv_gb300 import binding
from query_aware_sparse_kv_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"
    from query_aware_sparse_kv_gb300 import build

    build.build()
    qskv.load()


def _noalloc(dec, out, lse, dense=False):
    """Calls the entry point through the C ABI with raw pointers."""
    lib = binding.load()
    sel = None if dense else dec.selected
    st = lib.qskv_sparse_paged_decode_noalloc(
        binding._ptr(dec.q), binding._dtype(dec.q), binding._ptr(dec.k_pool), binding._ptr(dec.v_pool),
        binding._dtype(dec.k_pool), binding._ptr(dec.page_table), binding._ptr(dec.seq_lens),
        ctypes.byref(dec.shape), binding._ptr(sel), binding._ptr(None if dense else dec.n_selected),
        int(dec.top_k or 0), ctypes.c_float(0.0), binding._ptr(out), binding._ptr(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.last_error_message()


def _check_against_oracle(inp, dec, out, lse, dense, oracle):
    """Every row of the entry point's output against the oracle's attention
    over the same pages (the selection when sparse, every page when dense)."""
    spec = inp["spec"]
    Hkv, G = spec.num_kv_heads, spec.group
    tol = PR.out_tolerance(spec.kv_dtype)
    o, l = out.cpu().double().numpy(), lse.cpu().double().numpy()
    sel, nsel = dec.selected.cpu().numpy(), dec.n_selected.cpu().numpy()
    for r in range(spec.batch * Hkv):
        b, g = divmod(r, Hkv)
        n_b = PR.n_pages_of(inp, b)
        pages = list(range(n_b)) if dense else sel[b, g, :int(nsel[b, g])].tolist()
        o_out, o_lse = oracle.attend_row(inp, b, g, pages)
        PR.assert_output_close(o[b, g * G:(g + 1) * G], l[b, g * G:(g + 1) * G], o_out, o_lse, tol, f"row {r}")


@pytest.mark.parametrize("name,dense", [("llama", False), ("llama", True), ("tiny", False)])
def test_noalloc_matches_the_workspace_entry_point_twice(oracle_lib, name, dense):
    spec = (W.spec_for("llama3_8b", batch=4, seq_len_range=(900, 3000), max_pages=None, top_k=32)
            if name == "llama" else W.spec_for("tiny"))
    inp = W.make_inputs(spec)
    dec = qskv.from_inputs(inp)
    ids, vt = W.all_pages(inp)
    dec.build_meta(ids.cuda(), vt.cuda())
    if not dense:
        dec.select()
    dec.decode(dense=dense)
    dec.check()
    ref_out, ref_lse = dec.out.clone(), dec.lse.clone()
    tol = PR.out_tolerance(spec.kv_dtype)
    out = torch.full_like(dec.out, float("nan"))
    lse = torch.full_like(dec.lse, float("nan"))
    for _ in range(2):  # the scratch keeps the previous call's contents
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        _noalloc(dec, out, lse, dense=dense)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out - ref_out).abs().max().item() <= tol
        assert (lse - ref_lse).abs().max().item() <= tol
        _check_against_oracle(inp, dec, out, lse, dense, oracle_lib)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A shape whose partials would not fit the built-in scratch fails
    before any launch, with a message naming the alternative."""
    small = torch.zeros(64, dtype=torch.bfloat16, device="cuda")
    ints = torch.zeros(16, dtype=torch.int32, device="cuda")
    out = torch.zeros(64, dtype=torch.float32, device="cuda")
    shape = qskv.make_shape(4096, 64, 8, 128, 16, 4, 1024)  # 32768 rows: ~140 MB of partials
    with pytest.raises(qskv.QskvError) as e:
        qskv.sparse_paged_decode_noalloc(small, small, small, ints, ints, out, shape)
    assert e.value.status == 3
    assert "workspace" in str(e.value)
