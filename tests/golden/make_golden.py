"""Writes oracle_micro.json: a micro decode batch and the oracle's answers.

Run from the repository root:  python tests/golden/make_golden.py
Inputs come from the seeded generator; every expected value is computed by
the CPU oracle (``oracle/``) alone.  The fixture stores the inputs too, so the
regression test does not depend on the random number generator's stream.
"""
import json
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from query_aware_sparse_kv_gb300 import workloads as W  # noqa: E402


def main():
    spec = W.Spec(name="micro", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4,
                  seq_lens=(22, 7), top_k=2, q_dtype=torch.float32, kv_dtype=torch.bfloat16, kind="iid",
                  extra_pool_pages=1, seed=11)
    inp = W.make_inputs(spec)
    res = oracle.step(inp)
    doc = {
        "about": "Oracle regression fixture (query-aware sparse paged decode). Inputs from the seeded "
                 "generator, expected values from oracle.step; written by tests/golden/make_golden.py.",
        "source": "TinyServe query-aware page selection article s2.1-2.3; CS336 Lecture 10 s2.3, s9.2",
        "shape": dict(batch=2, num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4, top_k=2),
        "q": inp["q"].tolist(),
        "k_pool": inp["k_pool"].float().tolist(),
        "v_pool": inp["v_pool"].float().tolist(),
        "page_table": inp["page_table"].tolist(),
        "seq_lens": inp["seq_lens"].tolist(),
        "meta": res["meta"].tolist(),
        "scores": [[None if x == float("-inf") else x for x in r] for r in res["scores"].tolist()],
        "selected": res["selected"].tolist(),
        "n_sel": res["n_sel"].tolist(),
        "out": res["out"].tolist(),
        "lse": res["lse"].tolist(),
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_micro.json")
    with open(path, "w") as f:
        json.dump(doc, f, allow_nan=True)
    print("wrote", path)


if __name__ == "__main__":
    main()
