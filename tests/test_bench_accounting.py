"""The benchmark's algorithmic byte counts against hand-worked sizes."""
import numpy as np
import torch

import bench
from query_aware_sparse_kv_gb300 import workloads as W


def test_tiny_step_bytes():
    """tiny: 2 sequences x 2 KV heads, 16 full pages of 16 tokens, d=64,
    fp32, top-4.  decode reads 4 rows x 4 pages x (16 x 64 x 4 B) x (K, V)
    = 131072 B of KV; select reads 4 rows x 16 pages x 2 x 64 x 4 B = 32768 B
    of metadata."""
    inp = W.make_inputs(W.spec_for("tiny"))
    sel = np.tile(np.arange(4, dtype=np.int32), (2, 2, 1))
    nsel = np.full((2, 2), 4, dtype=np.int32)
    nb = bench.step_bytes(inp, sel, nsel)
    assert nb["kv"] == 4 * 4 * 16 * 64 * 4 * 2
    q = 2 * 4 * 64 * 4
    out = 2 * 4 * 64 * 4 + 2 * 4 * 4
    selb = 2 * 2 * 4 * 4 + 2 * 2 * 4
    assert nb["decode"] == nb["kv"] + q + out + selb + 16 * 4
    assert nb["select"] == 4 * 16 * (2 * 64 * 4 + 4 + 8) + q + selb
    assert nb["meta"] == 2 * 2 * (16 * 64 * 4 + 2 * 64 * 4)


def test_partial_last_page_counts_only_loaded_subtiles():
    """A 32-token page with 5 valid tokens is read as one 16-token sub-tile."""
    spec = W.Spec(name="p", batch=1, num_q_heads=2, num_kv_heads=1, head_dim=128, page_size=32, seq_lens=(37,),
                  top_k=2, kind="iid")
    inp = W.make_inputs(spec)
    nb = bench.step_bytes(inp, np.array([[[0, 1]]]), np.array([[2]]))
    assert nb["kv"] == (2 + 1) * 16 * 128 * 2 * 2


def test_dense_counts_every_page():
    spec = W.spec_for("shared_prefix", batch=3, prefix_pages=2, suffix_pages=1)
    inp = W.make_inputs(spec)
    nb = bench.step_bytes(inp, None, None)
    assert nb["kv"] == 3 * 8 * 3 * 16 * 128 * 2 * 2
    assert nb["meta"] == 0 and nb["select"] == 0  # a dense step reads no metadata
    assert nb["select"] == 0


def test_cascade_counts_the_prefix_once():
    """3 sequences x 8 KV heads share 2 prefix pages and own 1 page each:
    the cascade reads (2 + 3 x 1) page-heads of K and V per KV head."""
    spec = W.spec_for("shared_prefix", batch=3, prefix_pages=2, suffix_pages=1)
    inp = W.make_inputs(spec)
    nb = bench.step_bytes(inp, None, None, prefix_pages=2)
    assert nb["kv"] == 8 * (2 + 3 * 1) * 16 * 128 * 2 * 2


def test_reference_arm_json_line():
    """`bench.py --impl reference` runs the oracle on the host cores (no GPU)
    and prints the contract's JSON line for the reference arm."""
    import json
    import subprocess
    import sys

    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "2",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600,
                       cwd=str(__import__("pathlib").Path(bench.__file__).parent))
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([x for x in r.stdout.splitlines() if x.startswith("{")][-1])
    assert line["impl"] == "reference" and line["unit"] == "steps/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["steps"] == 2 and line["warmup"] == 3
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "steps/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert line["config"]["l2"].startswith("inputs fit in L2")


def test_l2_note_states_what_holds():
    llama = W.make_inputs(W.spec_for("llama3_8b", batch=2, seq_len_range=(30000, 32000)))
    assert "both exceed L2" not in bench.l2_note(llama)  # 2 x 8 rows x 128 pages x 8 KB = 17 MB a step
    assert "exceeds L2" in bench.l2_note(llama)


def _shape_only(name, **kw):
    """A workload's shapes without its values: the pool is a broadcast view
    (no memory), which is all the replica count reads."""
    spec = W.spec_for(name, **kw)
    g = torch.Generator().manual_seed(5)
    if spec.seq_lens is not None:
        seq = torch.tensor(list(spec.seq_lens), dtype=torch.int32)
    elif spec.kind == "shared_prefix":
        seq = torch.full((spec.batch,), (spec.prefix_pages + spec.suffix_pages) * spec.page_size, dtype=torch.int32)
    else:
        lo, hi = spec.seq_len_range
        seq = torch.randint(lo, hi + 1, (spec.batch,), generator=g).to(torch.int32)
    nb = (seq + spec.page_size - 1) // spec.page_size
    n_pool = int(nb.sum()) if spec.kind != "shared_prefix" else spec.prefix_pages + spec.batch * spec.suffix_pages
    pool = torch.zeros(1, dtype=spec.kv_dtype).expand(n_pool, spec.num_kv_heads, spec.page_size, spec.head_dim)
    return {"spec": spec, "k_pool": pool, "n_pages": nb, "seq_lens": seq}


def test_pool_copies_make_the_rotating_kv_exceed_four_l2():
    """Steps rotate over enough copies of the pool that the K/V they read
    together exceeds 4 x 129 MB: Llama-like 268 MB a step -> 2 copies,
    GPT2-like 81 MB -> 8, long context 67 MB -> 8; the shared-prefix batch
    (545 MB of unique K/V) and the tiny batch (fits in L2) need none."""
    for name, want in (("llama3_8b", 2), ("gpt2_345m", 8), ("long_context", 8), ("shared_prefix", 1),
                       ("tiny", 1)):
        inp = _shape_only(name)
        r = bench.replica_count(inp)
        assert r == want, (name, r, bench.step_kv_bytes(inp))
        if r > 1:
            assert r * bench.step_kv_bytes(inp) >= 4 * bench.L2_BYTES
            assert (r // 2) * bench.step_kv_bytes(inp) < 4 * bench.L2_BYTES
            assert "copies of the pool" in bench.l2_note(inp, r)


def test_source_hash_ignores_comments(tmp_path):
    a, b, c = tmp_path / "a.cu", tmp_path / "b.cu", tmp_path / "c.cu"
    a.write_text("int f() { return 1; }  // one\n/* block\n comment */\n")
    b.write_text("// another comment\nint f() { return 1; }\n\n")
    c.write_text("int f() { return 2; }\n")
    assert bench.source_hash([a]) == bench.source_hash([b]) != bench.source_hash([c])


def test_launches_per_step_of_each_workload():
    """The bench line's gpu_launches claim, per step on a 152-SM GB300: one
    launch for the GPT2-like step (its rows fit one wave split 2 ways, and a
    CTA's 256 pages of metadata one staging round), two for the Llama-like
    (k = 1) and long-context (512 pages per CTA: too many for one round)
    steps, two for the cascade, five for the fp32 tiny batch; the separate
    calls take three for the bf16 sparse steps."""
    import torch

    want = {"llama3_8b": 2, "gpt2_345m": 1, "long_context": 2, "shared_prefix": 2, "tiny": 5}
    for name, n in want.items():
        spec = W.spec_for(name)
        pages = spec.max_pages or (spec.prefix_pages + spec.suffix_pages if spec.kind == "shared_prefix"
                                   else -(-max(spec.seq_lens) // spec.page_size))
        inputs = {"page_table": torch.empty((spec.batch, pages), dtype=torch.int32)}
        prefix = spec.prefix_pages if spec.kind == "shared_prefix" else 0
        assert bench.kernels_per_step(spec, inputs, prefix, sms=152) == n, name
        if spec.top_k is not None and spec.kv_dtype == torch.bfloat16:
            assert bench.kernels_per_step(spec, inputs, prefix, one_call=False, sms=152) == 3, name
