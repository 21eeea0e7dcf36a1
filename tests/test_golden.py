"""Oracle regression against tests/golden/oracle_micro.json (written by
tests/golden/make_golden.py from the oracle alone).  Guards the oracle's
arithmetic against accidental change; its correctness is pinned by
test_oracle_pins.py."""
import json
import os

import numpy as np
import torch

from query_aware_sparse_kv_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_micro_regression(oracle_lib):
    with open(os.path.join(HERE, "golden", "oracle_micro.json")) as f:
        doc = json.load(f)
    s = doc["shape"]
    spec = W.Spec(name="micro", batch=s["batch"], num_q_heads=s["num_q_heads"], num_kv_heads=s["num_kv_heads"],
                  head_dim=s["head_dim"], page_size=s["page_size"], seq_lens=tuple(doc["seq_lens"]),
                  top_k=s["top_k"], q_dtype=torch.float32, kv_dtype=torch.bfloat16)
    inp = dict(spec=spec, q=torch.tensor(doc["q"], dtype=torch.float32),
               k_pool=torch.tensor(doc["k_pool"], dtype=torch.float32).to(torch.bfloat16),
               v_pool=torch.tensor(doc["v_pool"], dtype=torch.float32).to(torch.bfloat16),
               page_table=torch.tensor(doc["page_table"], dtype=torch.int32),
               seq_lens=torch.tensor(doc["seq_lens"], dtype=torch.int32))
    inp["n_pages"] = (inp["seq_lens"] + s["page_size"] - 1) // s["page_size"]
    res = oracle_lib.step(inp)
    np.testing.assert_array_equal(res["meta"], np.array(doc["meta"], dtype=np.float64))
    want_scores = np.array([[-np.inf if x is None else x for x in r] for r in doc["scores"]])
    np.testing.assert_allclose(res["scores"], want_scores, rtol=1e-13)
    assert res["selected"].tolist() == doc["selected"]
    assert res["n_sel"].tolist() == doc["n_sel"]
    np.testing.assert_allclose(res["out"], np.array(doc["out"]), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(res["lse"], np.array(doc["lse"]), rtol=1e-12)
