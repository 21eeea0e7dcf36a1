"""Buffer plumbing around the three C-ABI calls for one paged KV cache.

``PagedDecoder`` owns the device buffers a decode step needs (metadata,
workspace, selection, outputs) and issues the calls in order.  It only
allocates and passes pointers; every step of the computation runs in
libqskv.so's kernels.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import binding as B


class PagedDecoder:
    """One decode batch over a paged KV cache resident on the GPU.

    q           [batch][Hq][d]            fp32 or bf16
    k_pool      [Npool][Hkv][P][d]        fp32 or bf16 (v_pool the same)
    page_table  [batch][max_pages] int32  physical page ids
    seq_lens    [batch] int32
    top_k       pages kept per (sequence, KV head); None = dense decode
    prefix_pages  logical pages [0, prefix_pages) every row shares (the same
                physical pages): dense decodes then run as a cascade, the
                prefix attended once per KV head for the whole batch
    scorer      "bound" (TinyServe min/max metadata, the default) or
                "centroid" (Block Top-K: fp32 mean key per page, q . centroid)
    approx_epsilon  None: exact top-K; else the lossy top-K stops refining
                once at most floor(epsilon * top_k) pages are undecided and
                samples them from the threshold bucket (seed approx_seed)
    """

    def __init__(self, q, k_pool, v_pool, page_table, seq_lens, top_k: Optional[int], sm_scale: float = 0.0,
                 prefix_pages: int = 0, scorer: str = "bound", approx_epsilon: Optional[float] = None,
                 approx_seed: int = 0):
        self.approx_epsilon, self.approx_seed = approx_epsilon, approx_seed
        if scorer not in ("bound", "centroid"):
            raise ValueError(f"unknown scorer {scorer!r}")
        dev = k_pool.device
        self.q, self.k_pool, self.v_pool = q, k_pool, v_pool
        self.page_table, self.seq_lens = page_table, seq_lens
        n_pool, hkv, P, d = k_pool.shape
        batch, hq, _ = q.shape
        self.top_k = top_k
        self.sm_scale = sm_scale
        self.shape = B.make_shape(batch, hq, hkv, d, P, page_table.shape[1], n_pool)
        self.prefix_pages = int(prefix_pages)
        self.scorer = scorer
        if scorer == "centroid":
            self.meta = torch.empty((n_pool, hkv, d), dtype=torch.float32, device=dev)
        else:
            self.meta = torch.empty((n_pool, hkv, 2, d), dtype=k_pool.dtype, device=dev)
        ws = B.workspace_size(self.shape)
        if self.prefix_pages > 0:
            ws = max(ws, B.cascade_workspace_size(self.shape, self.prefix_pages))
        self.workspace = torch.zeros(ws, dtype=torch.uint8, device=dev)
        k = max(int(top_k or 1), 1)
        self.selected = torch.full((batch, hkv, k), -1, dtype=torch.int32, device=dev)
        self.n_selected = torch.zeros((batch, hkv), dtype=torch.int32, device=dev)
        self.out = torch.empty((batch, hq, d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((batch, hq), dtype=torch.float32, device=dev)

    # -- cache phase ---------------------------------------------------------
    def build_meta(self, page_ids: torch.Tensor, valid_tokens: torch.Tensor, stream=None):
        if self.scorer == "centroid":
            B.kv_centroid_build(self.k_pool, page_ids, valid_tokens, self.meta, self.shape, self.workspace, stream)
        else:
            B.kv_meta_build(self.k_pool, page_ids, valid_tokens, self.meta, self.shape, self.workspace, stream)

    # -- indexer phase -------------------------------------------------------
    @property
    def can_refresh_in_select(self) -> bool:
        """Whether select(refresh_last=True) runs as one launch (bound scorer,
        exact top-K, bf16 KV); otherwise it is a metadata build of the last
        pages followed by the selection."""
        return self.scorer == "bound" and self.approx_epsilon is None and self.k_pool.dtype == torch.bfloat16

    def select(self, q=None, scores: Optional[torch.Tensor] = None, stream=None, refresh_last: bool = False):
        """Top-K pages per (sequence, KV head).  refresh_last: first rebuild
        the metadata of every sequence's last page (the page the new token
        went into)."""
        if refresh_last and self.can_refresh_in_select:
            B.page_select_refresh(self.q if q is None else q, self.k_pool, self.meta, self.page_table, self.seq_lens,
                                  self.top_k, self.selected, self.n_selected, self.shape, self.workspace, scores,
                                  stream)
            return
        if refresh_last:
            self.build_meta(*self._last_pages(), stream)
        if self.approx_epsilon is not None:
            B.page_select_approx(self.q if q is None else q, self.meta, self.page_table, self.seq_lens, self.top_k,
                                 self.selected, self.n_selected, self.shape, self.workspace, self.approx_epsilon,
                                 self.approx_seed, scorer=self.scorer, scores=scores, stream=stream)
            return
        fn = B.page_select_centroid if self.scorer == "centroid" else B.page_select
        fn(self.q if q is None else q, self.meta, self.page_table, self.seq_lens, self.top_k, self.selected,
           self.n_selected, self.shape, self.workspace, scores, stream)

    def _last_pages(self):
        """(physical id, valid tokens) of every sequence's last page, gathered
        on the device from the page table and the lengths (plumbing for the
        two-call refresh; no arithmetic of the method)."""
        P = self.shape.page_size
        nb = torch.clamp((self.seq_lens.long() + P - 1) // P, min=1)
        ids = self.page_table.gather(1, (nb - 1)[:, None]).squeeze(1).to(torch.int32)
        valid = (self.seq_lens.long() - (nb - 1) * P).clamp(min=1).to(torch.int32)
        return ids, valid

    def decode(self, q=None, dense: bool = False, out=None, lse=None, stream=None):
        sel = None if (dense or self.top_k is None) else self.selected
        if sel is None and self.prefix_pages > 0:
            B.cascade_paged_decode(self.q if q is None else q, self.k_pool, self.v_pool, self.page_table,
                                   self.seq_lens, self.out if out is None else out, self.shape, self.workspace,
                                   self.prefix_pages, lse=self.lse if lse is None else lse, sm_scale=self.sm_scale,
                                   stream=stream)
            return
        B.sparse_paged_decode(self.q if q is None else q, self.k_pool, self.v_pool, self.page_table, self.seq_lens,
                              self.out if out is None else out, self.shape, self.workspace, selected=sel,
                              n_selected=self.n_selected if sel is not None else None,
                              top_k=self.top_k or 0, lse=self.lse if lse is None else lse, sm_scale=self.sm_scale,
                              stream=stream)

    def step(self, q=None, last_ids=None, last_valid=None, stream=None, out=None, refresh_last: bool = False):
        """Metadata refresh of the pages being appended to, selection, decode
        (into ``out`` if given, else ``self.out``).  The refresh is either
        the listed pages (last_ids, last_valid) or, with refresh_last, every
        sequence's last page inside the selection's launch; then, where the
        selection can take the refresh (bound scorer, exact top-K, bf16 KV),
        the whole step is one call (qskv_select_decode)."""
        if refresh_last and last_ids is None and self.top_k is not None and self.can_refresh_in_select:
            B.select_decode(self.q if q is None else q, self.k_pool, self.v_pool, self.meta, self.page_table,
                            self.seq_lens, self.top_k, self.selected, self.n_selected,
                            self.out if out is None else out, self.shape, self.workspace, lse=self.lse,
                            sm_scale=self.sm_scale, stream=stream)
            return
        if last_ids is not None:
            self.build_meta(last_ids, last_valid, stream)
        if self.top_k is not None:
            self.select(q, stream=stream, refresh_last=refresh_last)
        self.decode(q, out=out, stream=stream)

    def capture_step(self, q: torch.Tensor, last_ids=None, last_valid=None, q_host: Optional[torch.Tensor] = None,
                     out_host: Optional[torch.Tensor] = None, zero_copy: bool = True, refresh_last: bool = False):
        """Record one step (metadata refresh, selection, decode) reading the
        query from the device buffer `q` into a CUDA graph, and return a
        function that replays it on the current stream.  Refill `q` in place
        before each replay; results land in ``out`` / ``lse``.

        With pinned host tensors ``q_host`` (shaped like q) and/or
        ``out_host`` (shaped like out) the graph also moves the query in and
        the output out, so a serving loop launches one graph per step and
        synchronises once: a copy node brings ``q_host`` into ``q`` first
        (the scoring grid reads the query once per page chunk, so it is read
        from device memory), refill ``q_host`` before each replay.
        zero_copy=True (default): the decode writes the output straight into
        ``out_host`` (pinned host memory is device-accessible; on GB300 the
        NVLink-C2C link makes this faster than a copy node), and ``out`` is
        not written.  zero_copy=False: a copy node from ``out`` into
        ``out_host`` last."""
        def body():
            if q_host is not None:
                q.copy_(q_host, non_blocking=True)
            if zero_copy:
                self.step(q, last_ids, last_valid, out=out_host, refresh_last=refresh_last)
                return
            self.step(q, last_ids, last_valid, refresh_last=refresh_last)
            if out_host is not None:
                out_host.copy_(self.out, non_blocking=True)

        for t in (q_host, out_host):
            if t is not None and not t.is_pinned():
                raise ValueError("host buffers of a captured step must be pinned")
        if q_host is not None and (q_host.shape != q.shape or q_host.dtype != q.dtype):
            raise ValueError("q_host must have the shape and dtype of q")
        if out_host is not None and (out_host.shape != self.out.shape or out_host.dtype != self.out.dtype):
            raise ValueError("out_host must have the shape and dtype of out")
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            body()  # first use outside capture (device set-up)
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            body()
        return graph.replay

    def wait(self, stream=None):
        """Block the host until all work issued so far on ``stream`` (the
        current stream by default) has run, by polling an event recorded
        behind it (a busy wait on the host), which returns slightly sooner
        than a stream synchronisation; for serving loops that wait for every
        step's output."""
        st = torch.cuda.current_stream() if stream is None else stream
        ev = getattr(self, "_wait_event", None)
        if ev is None:
            ev = self._wait_event = torch.cuda.Event()
        ev.record(st)
        while not ev.query():
            pass

    def check(self, stream=None):
        """Raise if the device flagged an out-of-range index or a timeout."""
        st = B.get_error(self.workspace, stream)
        if st != 0:
            raise B.QskvError(st, B.last_error_message())


def from_inputs(inputs: dict, device="cuda", top_k="spec", prefix_pages: int = 0,
                scorer: str = "bound", approx_epsilon: Optional[float] = None, approx_seed: int = 0) -> PagedDecoder:
    """A PagedDecoder over a workloads.make_inputs() batch copied to `device`."""
    if isinstance(top_k, str):
        top_k = inputs["top_k"]
    t = {k: inputs[k].to(device) for k in ("q", "k_pool", "v_pool", "page_table", "seq_lens")}
    return PagedDecoder(t["q"], t["k_pool"], t["v_pool"], t["page_table"], t["seq_lens"], top_k,
                        prefix_pages=prefix_pages, scorer=scorer, approx_epsilon=approx_epsilon,
                        approx_seed=approx_seed)
