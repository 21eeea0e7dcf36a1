"""Benchmark: query-aware sparse paged decode steps on GB300.

A step is one pass of the whole hot path over one batch: refresh the
metadata of the page each sequence appends to, select the top-K pages per
(sequence, KV head), and run sparse paged decode over them (one library
call, qskv_select_decode, for the bf16 workloads with a top-K: one to three
launches by shape; the dense shared-prefix batch is the cascade decode alone;
the fp32 tiny batch takes the separate calls).  Inputs are synthetic and resident in HBM.  The
query rotates over 16 variants, and where one step's K/V would fit in a few
L2s the steps also rotate over copies of the KV pool and its metadata, so
that a step never finds its K/V in the 129 MB L2.

The JSON line's headline is the Llama-3-8B-like workload; `per_workload`
carries the same measurement for the GPT2-345M-like, long-context,
shared-prefix and tiny workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...     # the CPU oracle on the host cores

One JSON line on stdout (rank 0).  Under torchrun each rank decodes its own
batch (weak scaling, no collective on the data path); the timed region is
bracketed by barriers and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from query_aware_sparse_kv_gb300 import workloads as W  # noqa: E402

METRIC = "sparse paged decode: steps/s and effective HBM GB/s (% of GB300 peak)"
DEFAULT_WORKLOAD = "llama3_8b"
N_Q_VARIANTS = 16
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------ accounting --
def _es(dtype) -> int:
    return torch.tensor([], dtype=dtype).element_size()


def step_bytes(inputs: dict, selected: np.ndarray | None, n_selected: np.ndarray | None,
               prefix_pages: int = 0, scorer: str = "bound") -> dict:
    """Algorithmic bytes of one step, per kernel.

    decode: K and V of every 16-token sub-tile holding a valid token of a
            selected page (a whole page when P = 16), q, out, lse, the
            selected list and one page-table entry per selected page; with
            a shared prefix of `prefix_pages` pages (cascade decode), the
            prefix pages once per KV head instead of once per sequence;
    select: the metadata of every page of every row (2 d values in the KV
            dtype for the bound scorer, d fp32 for the centroid scorer), q,
            one page-table entry per page, the fp32 score written and read
            back, the selected list written;
    meta:   the valid key rows of each sequence's last page, its metadata
            written (sparse decode only: a dense decode reads no metadata,
            so its step has no refresh).
    """
    spec = inputs["spec"]
    B, Hq, Hkv, d, P = spec.batch, spec.num_q_heads, spec.num_kv_heads, spec.head_dim, spec.page_size
    s = _es(spec.kv_dtype)
    qs = _es(spec.q_dtype)
    seq = inputs["seq_lens"].numpy().astype(np.int64)
    nb = (seq + P - 1) // P
    sub_bytes = 16 * d * s * 2  # K + V of one 16-token sub-tile
    kv = 0
    n_pages_read = 0
    for b in range(B):
        for g in range(Hkv):
            if selected is None:
                pages = range(int(nb[b]))
            else:
                pages = selected[b, g, :int(n_selected[b, g])]
            for j in pages:
                if b > 0 and int(j) < prefix_pages:
                    continue  # read once, for the whole batch
                valid = min(P, int(seq[b]) - int(j) * P)
                kv += ((valid + 15) // 16) * sub_bytes
                n_pages_read += 1
    q_bytes = B * Hq * d * qs
    out_bytes = B * Hq * d * 4 + B * Hq * 4
    top_k = spec.top_k
    sel_bytes = 0 if top_k is None else B * Hkv * top_k * 4 + B * Hkv * 4
    decode = kv + q_bytes + out_bytes + sel_bytes + n_pages_read * 4
    meta_row = d * 4 if scorer == "centroid" else 2 * d * s
    if top_k is None:
        select = 0
    else:
        total_pages = int(nb.sum()) * Hkv
        select = total_pages * (meta_row + 4 + 8) + q_bytes + sel_bytes
    last_valid = seq - (nb - 1) * P
    meta = 0 if top_k is None else int(sum(int(v) * d * s + meta_row for v in last_valid)) * Hkv
    return dict(decode=decode, select=select, meta=meta, total=decode + select + meta, kv=kv)


# ---------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [s for t, s in self.samples if t0 - 0.15 <= t <= t1 + 0.15]
        window = "timed"
        if not rows:
            rows = [s for _, s in self.samples]
            window = "run"
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows), "window": window}


# ------------------------------------------------------------ references --
def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured (MEASURED_PEAKS.json)"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "fallback"}


# ------------------------------------------------------------ distributed --
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def shard_spec(spec: W.Spec, rank: int) -> W.Spec:
    """Rank r decodes its own batch of the same shape (weak scaling)."""
    import dataclasses

    return dataclasses.replace(spec, seed=spec.seed + 1000 * rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# --------------------------------------------------------------- oracle --
def cpu_model() -> str:
    """The host CPU's model name (x86 "model name", or Arm implementer/part)."""
    try:
        info = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in info:
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    impl = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU implementer")]
    part = [l.split(":", 1)[1].strip() for l in info if l.startswith("CPU part")]
    if impl and part:
        return f"Arm implementer {impl[0]} part {part[0]} x {len(part)}"
    return "unknown"


def oracle_sample(inputs: dict, qv_cpu, budget_s: float, threads: int, step_target_s: float | None = None,
                  scorer: str = "bound"):
    """Times the CPU oracle (scores, top-K, attention) on a bounded sample of
    rows.  Returns (steps/s, cores, sample description, rows per step used)."""
    import oracle

    spec = inputs["spec"]
    n_rows = spec.batch * spec.num_kv_heads
    meta = None
    if spec.top_k is not None:
        ids, vt = oracle.all_pages(inputs)
        meta = (oracle.centroids if scorer == "centroid" else oracle.meta)(inputs["k_pool"], ids, vt)
    rng = np.random.default_rng(0)
    # calibrate on a small sample
    calib = rng.choice(n_rows, size=min(n_rows, max(threads, 8)), replace=False).astype(np.int32)
    t0 = time.perf_counter()
    res = oracle.step(inputs, rows=calib, meta_arr=meta, q=qv_cpu[0], threads=threads, scorer=scorer)
    dt = time.perf_counter() - t0
    rows_per_s = len(calib) / max(dt, 1e-9)
    cores = int(res["threads"])
    per_step = step_target_s if step_target_s is not None else budget_s
    n = int(min(n_rows, max(1, rows_per_s * per_step)))
    done_rows, t_total, steps = 0, 0.0, 0
    while t_total < budget_s or steps == 0:
        rows = rng.choice(n_rows, size=n, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        oracle.step(inputs, rows=rows, meta_arr=meta, q=qv_cpu[steps % len(qv_cpu)], threads=threads, scorer=scorer)
        t_total += time.perf_counter() - t0
        done_rows += n
        steps += 1
        if step_target_s is not None:
            break
    steps_per_s = (done_rows / n_rows) / t_total
    sample = (f"{steps} samples of {n} random rows out of the {n_rows} (sequence, KV head) rows of a step "
              f"(scores + top-K + attention per row), {done_rows / n_rows:.2f} full steps in {t_total:.2f} s "
              f"on {cores} OpenMP threads")
    return steps_per_s, cores, sample, n


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    spec = W.spec_for(args.workload)
    inputs = W.make_inputs(spec)
    qv = W.q_variants(inputs, N_Q_VARIANTS)
    threads = os.cpu_count() or 1
    # each of the K steps is a bounded sample sized so the run lasts about two minutes
    per_step = max(0.02, 120.0 / max(1, args.steps + args.warmup))
    import oracle

    meta = None
    if spec.top_k is not None:
        ids, vt = oracle.all_pages(inputs)
        meta = (oracle.centroids if args.scorer == "centroid" else oracle.meta)(inputs["k_pool"], ids, vt)
    n_rows = spec.batch * spec.num_kv_heads
    rng = np.random.default_rng(0)
    calib = np.arange(min(n_rows, max(threads, 8)), dtype=np.int32)
    t0 = time.perf_counter()
    res = oracle.step(inputs, rows=calib, meta_arr=meta, q=qv[0], threads=threads, scorer=args.scorer)
    rows_per_s = len(calib) / (time.perf_counter() - t0)
    n = int(min(n_rows, max(1, rows_per_s * per_step)))
    for i in range(args.warmup):
        oracle.step(inputs, rows=rng.choice(n_rows, size=n, replace=False).astype(np.int32), meta_arr=meta,
                    q=qv[i % N_Q_VARIANTS], threads=threads, scorer=args.scorer)
    t_total = 0.0
    for i in range(args.steps):
        rows = rng.choice(n_rows, size=n, replace=False).astype(np.int32)
        t0 = time.perf_counter()
        oracle.step(inputs, rows=rows, meta_arr=meta, q=qv[i % N_Q_VARIANTS], threads=threads, scorer=args.scorer)
        t_total += time.perf_counter() - t0
    steps_per_s = (args.steps * n / n_rows) / t_total
    cores = int(res["threads"])
    sample = (f"each step: {n} of {n_rows} random (sequence, KV head) rows (scores + top-K + attention), "
              f"scaled to full steps; {cores} OpenMP threads")
    line = {
        "impl": "reference", "metric": METRIC, "value": steps_per_s, "unit": "steps/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / steps_per_s,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, args.scorer, args.approx_eps, inputs),
        "cpu_baseline": {"value": steps_per_s, "unit": "steps/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": steps_per_s, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6  # GB300 L2
MAX_REPLICAS = 16


def step_kv_bytes(inputs: dict) -> float:
    """K+V bytes one step reads: the selected pages (sparse; top-K whole
    pages per row), or every page once (dense; the shared prefix counted
    once)."""
    spec = inputs["spec"]
    P, d, Hkv = spec.page_size, spec.head_dim, spec.num_kv_heads
    page = 2 * P * d * inputs["k_pool"].element_size()
    nb = inputs["n_pages"].long()
    pages = (torch.clamp(nb, max=spec.top_k) if spec.top_k is not None else nb).sum().item() * Hkv
    if spec.kind == "shared_prefix" and spec.top_k is None:
        pages = (nb.sum().item() - (spec.batch - 1) * spec.prefix_pages) * Hkv  # unique pages
    return float(pages * page)


def replica_count(inputs: dict) -> int:
    """Copies of the KV pool (and its metadata) the timed steps rotate over so
    that consecutive steps never find their K/V in L2: enough that the K/V
    the rotating steps read together exceeds 4 x L2 (a power of two, so the
    16 query variants and the copies cycle together).  A workload whose
    whole pool fits in L2 (the correctness case) is not replicated."""
    pool = 2 * inputs["k_pool"].numel() * inputs["k_pool"].element_size()
    if pool <= L2_BYTES:
        return 1
    r = 1
    while r < MAX_REPLICAS and r * step_kv_bytes(inputs) < 4 * L2_BYTES:
        r *= 2
    return r


def l2_note(inputs: dict, replicas: int = 1) -> str:
    """How the timed steps relate to the 129 MB L2."""
    pool = 2 * inputs["k_pool"].numel() * inputs["k_pool"].element_size()
    step = step_kv_bytes(inputs)
    if pool <= L2_BYTES:
        return f"inputs fit in L2 (KV pool {pool / 1e6:.1f} MB; correctness workload), no flush"
    if replicas > 1:
        return (f"KV pool {pool / 1e9:.2f} GB; one step reads {step / 1e6:.0f} MB of K/V, so the steps rotate over "
                f"{replicas} copies of the pool and its metadata ({replicas * step / 1e6:.0f} MB of K/V >= 4 x L2): "
                f"a step never finds its K/V in L2; 16 rotating query variants")
    if step > 4 * L2_BYTES:
        return (f"KV pool {pool / 1e9:.2f} GB and one step's K/V {step / 1e6:.0f} MB both exceed 4 x L2; "
                f"16 rotating query variants")
    return (f"KV pool {pool / 1e9:.2f} GB exceeds L2; one step's K/V ({step / 1e6:.0f} MB) is below 4 x L2 and "
            f"partly repeats across the 16 rotating query variants (no pool copies)")


def workload_config(spec: W.Spec, scorer: str = "bound", approx_eps=None, inputs=None, replicas: int = 1) -> dict:
    desc = {
        "llama3_8b": "Llama-3-8B-like GQA decode, query-aware top-K paged KV",
        "gpt2_345m": "GPT2-345M-like MHA decode at 8K, query-aware top-K paged KV",
        "long_context": "long-context GQA decode, 64K-128K tokens, query-aware top-K paged KV",
        "shared_prefix": "shared-prefix dense decode (all pages), cascade: prefix once per KV head",
        "tiny": "tiny correctness batch",
    }.get(spec.name, spec.name)
    if spec.top_k is not None and scorer == "centroid":
        desc += " (Block Top-K centroid scorer)"
    if spec.top_k is not None and approx_eps is not None:
        desc += f" (lossy top-K, eps {approx_eps:g})"
    return {"workload": desc, "batch": spec.batch, "num_q_heads": spec.num_q_heads,
            "num_kv_heads": spec.num_kv_heads, "head_dim": spec.head_dim, "page_size": spec.page_size,
            "seq_len": list(spec.seq_len_range) if spec.seq_len_range else
            (list(spec.seq_lens)[:1] if spec.seq_lens else None),
            "top_k": spec.top_k, "kv_dtype": str(spec.kv_dtype).replace("torch.", ""),
            "q_dtype": str(spec.q_dtype).replace("torch.", ""), "pool_copies": replicas,
            "l2": l2_note(inputs, replicas) if inputs is not None else
            "KV pool larger than L2, 16 rotating query variants"}


def source_hash(paths) -> str:
    """Hash of the kernel sources with comments and blank lines removed, so a
    comment-only edit keeps a profile's counters valid and a code edit does
    not."""
    h = hashlib.sha256()
    for p in paths:
        text = open(p).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update("\n".join(l.strip() for l in text.splitlines() if l.strip()).encode())
    return h.hexdigest()[:16]


DECODE_SOURCES = [os.path.join(ROOT, "query_aware_sparse_kv_gb300", "csrc", n)
                  for n in ("decode.cu", "merge.cu", "qskv_device.cuh", "qskv_internal.h", "qskv_select.cuh")]


def ncu_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, or None if
    the decode kernel's code changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.md")
    try:
        text = open(path).read()
        sha = source_hash(DECODE_SOURCES)
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    h = re.search(r"decode_src_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != sha:
        return None
    return int(m.group(1))


# ---------------------------------------------------------------- recall --
def true_page_max_logits(inputs: dict, b: int, g: int, q) -> np.ndarray:
    """max over the group's heads and the page's valid tokens of q_h . k_t,
    per logical page of sequence b, KV head g (torch on the CPU, fp32): the
    ground truth the bound's ranking is judged against."""
    spec = inputs["spec"]
    P, G = spec.page_size, spec.group
    L = int(inputs["seq_lens"][b])
    nb = (L + P - 1) // P
    phys = inputs["page_table"][b, :nb].long()
    keys = inputs["k_pool"][phys, g].float().reshape(nb * P, -1)[:L]  # tokens past seq_len dropped
    logits = keys @ q[b, g * G:(g + 1) * G].float().T  # [L][G]
    best = torch.full((nb * P,), float("-inf"))
    best[:L] = logits.max(dim=1).values
    return best.view(nb, P).max(dim=1).values.numpy()


def selection_recall(inputs: dict, q, selected: np.ndarray, n_selected: np.ndarray, max_rows: int = 64) -> dict:
    """Recall figures of the GPU's selection (one query variant):
    true_topk: |selected & T| / K, T = the K pages with the largest true max
               logit (TinyServe s2.2 states its recall this way), over rows
               with more than K pages;
    planted / aligned: share of the planted pages (Llama-like) or of the pages
               drawn around the query's own centroid (long context) that are
               kept, up to K."""
    spec = inputs["spec"]
    K, Hkv = spec.top_k, spec.num_kv_heads
    rows = [(b, g) for b in range(spec.batch) for g in range(Hkv)]
    rng = np.random.default_rng(0)
    if len(rows) > max_rows:
        rows = [rows[i] for i in sorted(rng.choice(len(rows), size=max_rows, replace=False))]
    true_r, struct_r = [], []
    struct = inputs.get("planted") if inputs.get("planted") is not None else inputs.get("aligned")
    for b, g in rows:
        sel = set(selected[b, g, :int(n_selected[b, g])].tolist())
        nb = int(inputs["n_pages"][b])
        if nb > K:
            m = true_page_max_logits(inputs, b, g, q)
            top = np.argsort(-m, kind="stable")[:K]
            true_r.append(len(sel & set(top.tolist())) / K)
        if struct is not None:
            pages = [int(x) for x in struct[b, g].tolist() if x >= 0]
            if pages:
                struct_r.append(len(sel & set(pages)) / min(len(pages), K))
    out = {"rows": len(rows), "true_topk": float(np.mean(true_r)) if true_r else None}
    if struct is not None:
        out["planted" if inputs.get("planted") is not None else "aligned"] = float(np.mean(struct_r))
    return out


# ------------------------------------------------------------------ main --
class Bench:
    """One workload's decode step on the GPU: inputs (replicated to defeat L2),
    a PagedDecoder, one CUDA graph per query variant for the whole step and
    split graphs (selection part, decode part) for the decode call alone."""

    def __init__(self, spec: W.Spec, args, dev, prefix: int):
        import query_aware_sparse_kv_gb300 as qskv

        self.spec, self.args, self.dev, self.prefix = spec, args, dev, prefix
        t0 = time.perf_counter()
        inputs = W.make_inputs(spec)
        self.inputs = inputs
        self.qv_cpu = W.q_variants(inputs, N_Q_VARIANTS)
        self.qv = self.qv_cpu.to(dev)
        self.replicas = R = replica_count(inputs) if not args.no_replicas else 1
        n_pool = inputs["num_pool_pages"]
        k = inputs["k_pool"].to(dev)
        v = inputs["v_pool"].to(dev)
        if R > 1:
            k, v = k.repeat(R, 1, 1, 1), v.repeat(R, 1, 1, 1)
        pt = inputs["page_table"].to(dev)
        self.tables = [torch.where(pt >= 0, pt + r * n_pool, pt).contiguous() for r in range(R)]
        top_k = inputs["top_k"]
        self.dec = qskv.PagedDecoder(inputs["q"].to(dev), k, v, self.tables[0], inputs["seq_lens"].to(dev), top_k,
                                     prefix_pages=prefix, scorer=args.scorer, approx_epsilon=args.approx_eps,
                                     approx_seed=args.seed)
        ids, vt = W.all_pages(inputs)
        ids_all = torch.cat([ids + r * n_pool for r in range(R)]).to(dev)
        self.dec.build_meta(ids_all, vt.repeat(R).to(dev))
        li, lv = W.last_pages(inputs)
        self.last = [((li + r * n_pool).to(dev), lv.to(dev)) for r in range(R)]
        self.dec.check()
        self.setup_s = time.perf_counter() - t0

    def table_for(self, v: int) -> int:
        return v % self.replicas

    def use(self, v: int):
        self.dec.page_table = self.tables[self.table_for(v)]

    def select_part(self, v: int):
        if self.spec.top_k is not None:  # a dense decode reads no metadata: no refresh
            self.use(v)
            if self.dec.can_refresh_in_select:  # the last pages' refresh inside the scoring launch
                self.dec.select(q=self.qv[v], refresh_last=True)
            else:
                self.dec.build_meta(*self.last[self.table_for(v)])
                self.dec.select(q=self.qv[v])

    def decode_part(self, v: int):
        self.use(v)
        self.dec.decode(q=self.qv[v])

    @property
    def one_call(self) -> bool:
        """Whether a step is PagedDecoder.step's single call (qskv_select_decode:
        one to three launches by shape)."""
        return (self.spec.top_k is not None and self.dec.can_refresh_in_select
                and not self.args.separate_calls)

    def step_part(self, v: int):
        if self.one_call:
            self.use(v)
            self.dec.step(q=self.qv[v], refresh_last=True)
        else:
            self.select_part(v)
            self.decode_part(v)

    @staticmethod
    def capture(fn):
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()  # first use outside capture (kernel attributes, descriptors)
        torch.cuda.current_stream().wait_stream(side)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    def bytes_and_recall(self, want_recall: bool):
        acc, recall = [], None
        spec = self.spec
        for v in range(N_Q_VARIANTS):
            if spec.top_k is None:
                acc.append(step_bytes(self.inputs, None, None, prefix_pages=self.prefix))
                break
            self.use(v)
            self.dec.select(q=self.qv[v])
            torch.cuda.synchronize()
            sel, ns = self.dec.selected.cpu().numpy(), self.dec.n_selected.cpu().numpy()
            acc.append(step_bytes(self.inputs, sel, ns, scorer=self.args.scorer))
            if v == 0 and want_recall:
                recall = selection_recall(self.inputs, self.qv_cpu[0], sel, ns)
        self.nbytes = {k: sum(a[k] for a in acc) / len(acc) for k in acc[0]}
        return recall

    def build_graphs(self, warmup: int):
        for i in range(warmup):
            self.step_part(i % N_Q_VARIANTS)
        self.dec.check()
        torch.cuda.synchronize()
        self.step_graphs = [self.capture(lambda v=v: self.step_part(v)) for v in range(N_Q_VARIANTS)]
        self.sel_graphs = [self.capture(lambda v=v: self.select_part(v)) for v in range(N_Q_VARIANTS)]
        self.dec_graphs = [self.capture(lambda v=v: self.decode_part(v)) for v in range(N_Q_VARIANTS)]
        for i in range(warmup):
            self.step_graphs[i % N_Q_VARIANTS].replay()
        self.dec.check()
        torch.cuda.synchronize()

    def time_steps(self, steps: int, world: int) -> float:
        """Device time (ms) of `steps` graph replays, events on the launching stream."""
        stream = torch.cuda.current_stream()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(steps):
            self.step_graphs[i % N_Q_VARIANTS].replay()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        return start.elapsed_time(stop)

    def time_decode_call(self, n: int) -> float:
        """Mean device time (ms) of the decode call alone: events around the
        decode graph, each replayed right after its own selection graph."""
        stream = torch.cuda.current_stream()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            v = i % N_Q_VARIANTS
            self.sel_graphs[v].replay()
            ev[i][0].record(stream)
            self.dec_graphs[v].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        self.dec.check()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    def build_decode_stream(self):
        """One graph of N_Q_VARIANTS decode calls back to back: call v decodes
        query variant v over its own selection (computed beforehand and kept
        in a buffer of its own) and the pool copy of step v.  Nothing else
        runs between the calls, so the graph measures the decode call's own
        duration in a stream of calls (launches overlapped by programmatic
        dependent launch, as inside a step), without a graph launch per call."""
        dec = self.dec
        sels = []
        for v in range(N_Q_VARIANTS):
            self.use(v)
            if self.spec.top_k is not None:
                dec.select(q=self.qv[v])
                sels.append((dec.selected.clone(), dec.n_selected.clone()))
            else:
                sels.append(None)
        torch.cuda.synchronize()
        keep = (dec.selected, dec.n_selected)

        def body():
            for v in range(N_Q_VARIANTS):
                self.use(v)
                if sels[v] is not None:
                    dec.selected, dec.n_selected = sels[v]
                dec.decode(q=self.qv[v])
        try:
            self.stream_graph = self.capture(body)
        finally:
            dec.selected, dec.n_selected = keep
        self.stream_sels = sels

    def time_decode_stream(self, n: int) -> float:
        """Mean device time (ms) of one decode call: events around replays of
        the back-to-back graph (N_Q_VARIANTS calls each)."""
        reps = max(1, n // N_Q_VARIANTS)
        stream = torch.cuda.current_stream()
        self.stream_graph.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            self.stream_graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        self.dec.check()
        return e0.elapsed_time(e1) / (reps * N_Q_VARIANTS)

    def time_eager(self, n: int) -> float:
        stream = torch.cuda.current_stream()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            self.step_part(i % N_Q_VARIANTS)
        e1.record(stream)
        torch.cuda.synchronize()
        self.dec.check()
        return e0.elapsed_time(e1) / n

    def e2e(self, steps: int, warmup: int, world: int, zero_copy: bool) -> float:
        """Steps/s through the public API: one graph per step recorded by
        PagedDecoder.capture_step with pinned host q / out (a copy node brings
        q in; the decode writes out to host memory when zero_copy, else a copy
        node takes it out), the host waiting
        for every step's output (PagedDecoder.wait)."""
        dec, spec = self.dec, self.spec
        q_host = self.qv_cpu.pin_memory()
        q_dev = torch.empty_like(self.qv[0])
        q_dev.copy_(self.qv[0])
        out_host = torch.empty(dec.out.shape, dtype=dec.out.dtype).pin_memory()
        graphs = []
        for v in range(N_Q_VARIANTS):
            self.use(v)
            fused = spec.top_k is not None and dec.can_refresh_in_select and not self.args.separate_calls
            refresh = self.last[self.table_for(v)] if spec.top_k is not None and not fused else (None, None)
            graphs.append(dec.capture_step(q_dev, *refresh, q_host=q_host[v], out_host=out_host,
                                           zero_copy=zero_copy, refresh_last=fused))
        for i in range(min(steps, warmup)):
            graphs[i % N_Q_VARIANTS]()
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            graphs[i % N_Q_VARIANTS]()
            dec.wait()
        s = max_over_ranks(time.perf_counter() - t0, world, self.dev)
        dec.check()
        self.e2e_h2d = int(q_dev.numel() * q_dev.element_size())
        self.e2e_d2h = int(out_host.numel() * out_host.element_size())
        return world * steps / s


def kernels_per_step(spec: W.Spec, inputs: dict, prefix: int, scorer: str = "bound", approx: bool = False,
                     one_call: bool = True, sms: int | None = None) -> int:
    """The library's launches in one step: metadata refresh (inside the
    scoring launch for the exact bound top-K on bf16 KV), scoring, ranking
    (sparse only; inside the decode launch when the step is one call and the
    rows go one row per k CTAs, and the scoring with the refresh too when
    k >= 2 and a CTA's share of the pages fits one staging round), decode,
    and the merge kernel unless the decode folds the
    rows' pieces itself: bf16 KV without a shared prefix, and either the rows
    fit one wave of decode CTAs (one row per k CTAs: k = 1 for one or two rows
    per SM, else min(2 SMs / rows, 8, units / 4) when that gives every SM a
    CTA) or a row's stream-K pieces fit one warp's single round of loads
    (pieces x G x d / 128 <= 16, with the grid's 2 CTAs x 6 warps per SM); a
    cascade adds the prefix kernel."""
    if sms is None:
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    rows = spec.batch * spec.num_kv_heads
    spr = spec.top_k if spec.top_k is not None else inputs["page_table"].shape[1] - prefix
    upw = max(1, -(-rows * spr // (2 * sms * 6)))
    pieces = -(-spr // upw) + 1
    ctas = 2 * sms
    k = 0
    if spec.kv_dtype == torch.bfloat16 and prefix == 0 and 0 < rows <= ctas and spr <= 1024:
        k = 1 if rows >= sms else min(ctas // rows, 8, spr // 4)
        k = k if k == 1 or (k >= 2 and rows * k >= sms) else 0
    row_per_cta = k > 0
    per_lane = max(1, spec.group * spec.head_dim // 128)
    fold = row_per_cta or (spec.kv_dtype == torch.bfloat16 and prefix == 0 and pieces * per_lane <= 16)
    if prefix and spec.kv_dtype == torch.bfloat16:
        # the cascade: its decode grid is sized to the SMs the prefix grid
        # leaves, and a row also holds the prefix kernel's E pieces
        # (prefix_splits / prefix_ctas in prefix_attend.cu)
        tiles = -(-spec.batch * spec.group // 128) * spec.num_kv_heads
        nblk = -(-prefix * spec.page_size // 128)
        e = max(1, min(sms // tiles, nblk, 64)) if nblk else 0
        items = tiles * e
        share = max(1, int(sms * 0.43))
        rounds = -(-items // share)
        pctas = -(-items // rounds) if items else 0
        warps = 2 * max(1, sms - pctas) * 6
        upw_c = max(1, -(-rows * spr // warps))
        fold = spr > 0 and (-(-spr // upw_c) + 1 + e) * per_lane <= 16
    # the refresh runs inside the scoring launch for the exact bound top-K on bf16 KV
    fused_refresh = spec.kv_dtype == torch.bfloat16 and scorer == "bound" and not approx
    ranked_in_decode = fused_refresh and one_call and row_per_cta
    # ... and scored there too when each CTA's share of a full row fits its
    # staging memory at once (fused_score_pages_per_round in decode.cu)
    ring = (spec.head_dim // 64) * 16 * 128 * 2 * (1 if spec.head_dim == 128 else 2) * 2 * 6
    per_round = ring // (16 * (4 * spec.head_dim + 4)) * 16
    scored_in_decode = ranked_in_decode and k >= 2 and -(-inputs["page_table"].shape[1] // k) <= per_round
    n = ((2 if fused_refresh else 3) - (1 if ranked_in_decode else 0) - (1 if scored_in_decode else 0)
         if spec.top_k is not None else 0) + 1 + (0 if fold else 1)
    return n + (1 if prefix else 0)


def _prefix_for(spec: W.Spec, args) -> int:
    return spec.prefix_pages if (spec.kind == "shared_prefix" and not args.no_cascade) else 0


def cpu_baseline(inputs, qv_cpu, args, budget: float, single: bool) -> dict:
    sps, cores, sample, _ = oracle_sample(inputs, qv_cpu, budget_s=budget, threads=os.cpu_count() or 1,
                                          scorer=args.scorer)
    cpu = {"value": sps, "unit": "steps/s", "cores": cores, "kind": "oracle", "sample": sample,
           "cpu_model": cpu_model()}
    if single:
        sps1, _, sample1, _ = oracle_sample(inputs, qv_cpu, budget_s=max(1.0, budget / 4), threads=1,
                                            scorer=args.scorer)
        cpu["single_thread"] = {"value": sps1, "unit": "steps/s", "sample": sample1}
    return cpu


def summary(bn: Bench, ms_per_step: float, decode_ms: float, peak: float) -> dict:
    decode_gbs = bn.nbytes["decode"] / (decode_ms * 1e-3) / 1e9
    step_gbs = bn.nbytes["total"] / (ms_per_step * 1e-3) / 1e9
    return {"steps_per_s": 1000.0 / ms_per_step, "ms_per_step": ms_per_step, "effective_gbs": step_gbs,
            "hbm_frac_step": step_gbs / peak, "decode_ms": decode_ms, "decode_gbs": decode_gbs,
            "decode_frac": decode_gbs / peak, "bytes_per_step": bn.nbytes}


def run_gpu(args):
    import query_aware_sparse_kv_gb300 as qskv
    from query_aware_sparse_kv_gb300 import build as qbuild

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    if rank == 0:
        qbuild.build()
    barrier(world)
    qskv.load()
    peaks = measured_peaks()

    spec = W.spec_for(args.workload)
    if args.batch:
        spec = W.spec_for(args.workload, batch=args.batch,
                          seq_lens=spec.seq_lens[:1] * args.batch if spec.seq_lens else None)
    spec = shard_spec(spec, rank)
    prefix = _prefix_for(spec, args)
    main = Bench(spec, args, dev, prefix)
    recall = main.bytes_and_recall(want_recall=spec.top_k is not None and rank == 0 and not args.no_recall)
    main.build_graphs(args.warmup)

    gpu_id = str(local)
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    wall0 = time.time()
    elapsed_ms = main.time_steps(args.steps, world)
    wall1 = time.time()
    clocks = None
    main.build_decode_stream()
    decode_ms = main.time_decode_stream(min(args.steps, 1600))
    decode_isolated_ms = main.time_decode_call(min(args.steps, 1000))
    eager_ms = main.time_eager(min(args.steps, 300))
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    ms_per_step = elapsed_ms / args.steps
    value = world * args.steps / (elapsed_ms / 1000.0)

    # end to end through the public API (zero-copy default; copy nodes as a diagnostic)
    e2e_steps = 0 if args.no_e2e else min(args.steps, 500)
    e2e_value = main.e2e(e2e_steps, args.warmup, world, True) if e2e_steps else None
    e2e_copy_nodes = main.e2e(e2e_steps, args.warmup, world, False) if e2e_steps else None

    # the other workloads, each timed the same way (step graphs, decode call)
    per_workload = {}
    if args.per_workload and world == 1:
        for name in [n for n in PER_WORKLOAD_ORDER if n != args.workload]:
            ws = W.spec_for(name)
            bn = Bench(ws, args, dev, _prefix_for(ws, args))
            rec = bn.bytes_and_recall(want_recall=ws.top_k is not None and not args.no_recall)
            bn.build_graphs(args.warmup)
            t0 = time.time()
            ms = bn.time_steps(args.sub_steps, 1) / args.sub_steps
            t1 = time.time()
            bn.build_decode_stream()
            dms = bn.time_decode_stream(min(args.sub_steps, 1600))
            ent = summary(bn, ms, dms, peaks["hbm_gbs"])
            ent["decode_isolated_ms"] = bn.time_decode_call(min(args.sub_steps, 1000))
            ent["config"] = workload_config(ws, args.scorer, args.approx_eps, bn.inputs, bn.replicas)
            ent["steps"] = args.sub_steps
            ent["recall"] = rec
            ent["kernels_per_step"] = kernels_per_step(ws, bn.inputs, bn.prefix, args.scorer, args.approx_eps is not None,
                                               not args.separate_calls)
            if sampler:
                ent["clocks"] = sampler.summary(t0, t1)
            if not args.no_cpu_baseline:
                ent["cpu_baseline"] = cpu_baseline(bn.inputs, bn.qv_cpu, args, args.cpu_budget / 2, single=False)
            per_workload[name] = ent
            del bn
            torch.cuda.empty_cache()
    if sampler:
        time.sleep(0.25)
        sampler.stop()
        clocks = sampler.summary(wall0, wall1)

    if rank != 0:
        return 0
    main_sum = summary(main, ms_per_step, decode_ms, peaks["hbm_gbs"])
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        cpu = cpu_baseline(main.inputs, main.qv_cpu, args, args.cpu_budget, single=True)
    line = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if spec.kv_dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": workload_config(spec, args.scorer, args.approx_eps, main.inputs, main.replicas),
        "effective_gbs": main_sum["effective_gbs"],
        "hbm_frac_step": main_sum["hbm_frac_step"],
        "bytes_per_step": main.nbytes,
        "roofline": {"kernel": ("decode_bf16_kernel + prefix_attend_kernel (qskv_cascade_paged_decode)" if prefix
                                else "decode_bf16_kernel + merge (qskv_sparse_paged_decode)"), "bound": "hbm",
                     "achieved": main_sum["decode_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": main_sum["decode_frac"], "peak_source": peaks["source"],
                     "decode_ms": decode_ms, "bytes_per_launch": main.nbytes["decode"],
                     "timing": ("mean of back-to-back decode calls (one graph of 16 calls, each over its own "
                                "query variant, selection and pool copy; events around the replays)"),
                     "decode_isolated_ms": decode_isolated_ms,
                     "traffic": ncu_traffic(args.workload), "decode_src_sha256_16": source_hash(DECODE_SOURCES)},
        "cpu_baseline": cpu,
        "recall": recall,
        "step_launch": ("CUDA graph replay, one graph per query variant: " +
                        ("qskv_select_decode (one launch where the decode CTAs of a row also refresh and score "
                         "it; else the scoring launch with the last-page metadata refresh inside, then the "
                         "decode launch, which ranks its own rows when they go one row per k CTAs)" if main.one_call
                         else "scoring (last-page metadata refresh inside where it can be) + ranking + decode")
                        if spec.top_k is not None else
                        "CUDA graph replay, one graph per query variant (dense decode: no metadata refresh or selection)"),
        "eager_ms_per_step": eager_ms,
        "e2e": {"value": e2e_value, "unit": "steps/s", "steps": e2e_steps,
                "path": "PagedDecoder.capture_step(q_host, out_host) replay: a copy node brings q in from pinned "
                        "host memory, the decode writes out straight to pinned host memory (zero-copy), host "
                        "waits for every step (PagedDecoder.wait)",
                "copy_nodes_value": e2e_copy_nodes,
                "h2d_bytes_per_step": getattr(main, "e2e_h2d", 0), "d2h_bytes_per_step": getattr(main, "e2e_d2h", 0)},
        # kernels per step: metadata refresh (fused into scoring where it can be), scoring, ranking
        # (inside the decode for one-call steps of one row per k CTAs), decode, merge (dense: decode
        # and merge only; cascade: + the shared-prefix kernel; no merge when the decode folds its rows)
        "gpu_launches": kernels_per_step(spec, main.inputs, prefix, args.scorer, args.approx_eps is not None,
                                         not args.separate_calls) * args.steps,
        "clocks": clocks,
        "per_workload": per_workload or None,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


PER_WORKLOAD_ORDER = ["llama3_8b", "gpt2_345m", "long_context", "shared_prefix", "tiny"]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["qskv", "reference"], default="qskv")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=8.0, help="seconds of oracle timing for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch (profiling runs)")
    ap.add_argument("--scorer", choices=["bound", "centroid"], default="bound",
                    help="page score: TinyServe min/max bound (default) or Block Top-K centroid")
    ap.add_argument("--approx-eps", type=float, default=None,
                    help="lossy top-K: stop once floor(eps * K) pages are undecided and sample them")
    ap.add_argument("--seed", type=int, default=0, help="seed of the lossy top-K's sampling")
    ap.add_argument("--no-replicas", action="store_true",
                    help="do not rotate over copies of the KV pool (study of the warm-L2 case)")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --workload (profiling runs); by default the other workloads follow")
    ap.add_argument("--sub-steps", type=int, default=1000, help="timed steps of each other workload")
    ap.add_argument("--no-recall", action="store_true", help="skip the recall figures of the selection")
    ap.add_argument("--separate-calls", action="store_true",
                    help="a step as the separate selection and decode calls instead of qskv_select_decode")
    ap.add_argument("--no-cascade", action="store_true",
                    help="shared-prefix workload: plain paged dense decode instead of the cascade")
    args = ap.parse_args(argv)
    args.per_workload = not args.no_per_workload
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
