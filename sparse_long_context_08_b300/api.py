"""A decoder object over the C ABI: owns the device buffers of one decode
configuration and runs score -> select -> decode on the current stream.

Marshalling only; every stage runs in libentmaxkv.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import entmaxkv as E


class _HostStepGraphs:
    """Replays a host-buffer step as one CUDA graph: the pinned H2D copy of q,
    the step's kernels and the D2H copy of out are captured on the first call
    with a given set of buffers, so later calls cost one graph launch instead
    of one launch per copy and kernel.  The graph keeps the buffers it was
    captured with: the same tensors must stay alive and be reused."""

    def _host_graph_replay(self, eager, q_host, out_host, q_dev, stream=None) -> None:
        last = self.__dict__.get("_host_last")
        if (last is not None and stream is None and last[0] is q_host and last[1] is out_host
                and last[2] is q_dev):
            last[3].replay()                      # same buffers as the last call
            return
        graphs = self.__dict__.setdefault("_host_graphs", {})
        key = (q_host.data_ptr(), out_host.data_ptr(), q_dev.data_ptr())
        g = graphs.get(key)
        if g is None:
            cs = torch.cuda.Stream()
            cs.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(cs):
                eager(q_host, out_host, q_dev, cs)          # warm-up outside the capture
            cs.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                eager(q_host, out_host, q_dev, cs)
            torch.cuda.current_stream().wait_stream(cs)
            graphs[key] = g
        self._host_last = (q_host, out_host, q_dev, g)
        if stream is None:
            g.replay()
        else:
            with torch.cuda.stream(stream):
                g.replay()


def upload_workload(w, device="cuda") -> tuple[E.PagedKV, torch.Tensor]:
    """Copy a workloads.Workload (host numpy arrays) to the GPU."""
    def pool(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if a.dtype == np.uint16:
            t = t.view(torch.bfloat16)
        return t.to(device)
    kv = E.PagedKV(pool(w.k_pool), pool(w.v_pool),
                   torch.from_numpy(np.ascontiguousarray(w.page_table)).to(device),
                   torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(device))
    q = torch.from_numpy(np.ascontiguousarray(w.q)).to(device)
    return kv, q


class EntmaxKVDecoder(_HostStepGraphs):
    """score_pages -> select -> decode for one (cache, policy) configuration."""

    def __init__(self, kv: E.PagedKV, num_q_heads: int, scale: float, alpha: float,
                 policy: str = "topk", budget_tokens: int = 4096, delta: float = 0.0):
        self.kv = kv
        self.Hq = int(num_q_heads)
        self.scale = float(scale)
        self.alpha = float(alpha)
        self.policy = {"topk": E.EKV_SELECT_TOPK, "gauss": E.EKV_SELECT_GAUSS,
                       "topk_shared": E.EKV_SELECT_TOPK_SHARED}[policy]
        self.budget = int(budget_tokens)
        self.delta = float(delta)
        self.cap = self.budget // kv.page_size
        dev = kv.k_pool.device
        B, Hq = kv.batch, self.Hq
        gauss = self.policy == E.EKV_SELECT_GAUSS
        self.meta = E.PageMeta.empty_like(kv, bbox=not gauss, gauss=gauss)
        self.page_scores = torch.empty((B, Hq, kv.max_pages) + ((2,) if gauss else ()),
                                       dtype=torch.float32, device=dev)
        self.sel = torch.empty((B, Hq, self.cap), dtype=torch.int32, device=dev)
        self.n_sel = torch.empty((B, Hq), dtype=torch.int32, device=dev)
        self.aux = torch.empty((B, Hq, 2), dtype=torch.float32, device=dev)
        self.out = torch.empty((B, Hq, kv.head_dim), dtype=torch.float32, device=dev)
        self.tau = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.support = torch.empty((B, Hq), dtype=torch.int32, device=dev)
        ws = E.entmaxkv_workspace_size(B, Hq, kv.num_kv_heads, kv.head_dim, kv.page_size,
                                       kv.max_pages, self.cap)
        if ws == 0:
            raise ValueError("invalid sizes for the decode workspace")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def build_meta(self, first_page: int = 0, num_pages: int | None = None, stream=None) -> None:
        gauss = self.policy == E.EKV_SELECT_GAUSS
        E.entmaxkv_build_page_meta(self.kv, first_page,
                                   self.kv.max_pages if num_pages is None else num_pages,
                                   self.meta, want_bbox=not gauss, want_gauss=gauss, stream=stream)

    def score(self, q: torch.Tensor, stream=None) -> None:
        E.entmaxkv_score_pages(q, self.Hq, self.scale, self.kv, self.meta, self.policy,
                               self.page_scores, stream)

    def select(self, stream=None) -> None:
        E.entmaxkv_select(self.page_scores, self.kv, self.Hq, self.policy, self.budget,
                          self.alpha, self.delta, self.sel, self.n_sel, self.aux, stream)

    def decode(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        E.entmaxkv_decode(q, self.Hq, self.scale, self.kv, self.sel, self.n_sel, self.cap,
                          self.alpha, self.out, self.tau, self.support, self.workspace, stream)
        return self.out

    def select_decode(self, q: torch.Tensor, stream=None, out: torch.Tensor | None = None):
        """select then decode in one library call (the selection also builds
        the decode's page union); the same results as select() and decode().
        out: where the result goes (default self.out; pinned host memory is
        written by the kernel directly)."""
        out = self.out if out is None else out
        E.entmaxkv_select_decode(self.page_scores, q, self.Hq, self.scale, self.kv, self.policy,
                                 self.budget, self.alpha, self.delta, self.sel, self.n_sel,
                                 self.aux, out, self.tau, self.support, self.workspace,
                                 stream)
        return out

    def step(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        """One decode step for device-resident q [B, Hq, d]; returns `out` (device)."""
        self.score(q, stream)
        return self.select_decode(q, stream)

    def _step_host_eager(self, q_host, out_host, q_dev, s) -> None:
        with torch.cuda.stream(s):
            E.entmaxkv_copy_in(q_dev, q_host, s)      # a kernel, no copy-engine hand-off
            self.score(q_dev, s)
            self.select_decode(q_dev, s, out=out_host)   # the result written to host memory

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        """One decode step from host memory: q_host (pinned) -> q_dev by a
        copy kernel, the stages, and the result written by the last kernel
        straight into out_host (pinned); self.out is not written.
        Asynchronous on `stream`; replayed as one CUDA graph per set of
        buffers (see _HostStepGraphs)."""
        self._host_graph_replay(self._step_host_eager, q_host, out_host, q_dev, stream)


class EntmaxKVFullDecoder(_HostStepGraphs):
    """Full-cache alpha-entmax decode: attention over every valid token, the
    exact result the sparse pipeline approximates."""

    def __init__(self, kv: E.PagedKV, num_q_heads: int, scale: float, alpha: float):
        self.kv = kv
        self.Hq = int(num_q_heads)
        self.scale = float(scale)
        self.alpha = float(alpha)
        dev = kv.k_pool.device
        B, Hq = kv.batch, self.Hq
        self.out = torch.empty((B, Hq, kv.head_dim), dtype=torch.float32, device=dev)
        self.tau = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        self.support = torch.empty((B, Hq), dtype=torch.int32, device=dev)
        ws = E.entmaxkv_full_workspace_size(B, Hq, kv.num_kv_heads, kv.head_dim, kv.page_size,
                                            kv.max_pages)
        if ws == 0:
            raise ValueError("invalid sizes for the full-cache workspace")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def decode(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        E.entmaxkv_decode_full(q, self.Hq, self.scale, self.kv, self.alpha, self.out, self.tau,
                               self.support, self.workspace, stream)
        return self.out

    def _step_host_eager(self, q_host, out_host, q_dev, s) -> None:
        with torch.cuda.stream(s):
            q_dev.copy_(q_host, non_blocking=True)
            self.decode(q_dev, s)
            out_host.copy_(self.out, non_blocking=True)

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        """q_host (pinned) -> device, the full-cache decode, out -> out_host
        (pinned).  Asynchronous on `stream`; replayed as one CUDA graph."""
        self._host_graph_replay(self._step_host_eager, q_host, out_host, q_dev, stream)


class EntmaxKVSoftmaxDecoder(_HostStepGraphs):
    """Softmax attention over the pages the EntmaxKV scoring and selection keep
    (the comparison method: a softmax whose dense tail is truncated to the kept
    pages), or over every token with full=True.  The selection stage is the
    entmax pipeline's own (alpha only matters for the Gaussian tau-hat)."""

    def __init__(self, kv: E.PagedKV, num_q_heads: int, scale: float, policy: str = "topk",
                 budget_tokens: int = 4096, delta: float = 0.0, alpha: float = 1.5,
                 full: bool = False):
        self.kv = kv
        self.Hq = int(num_q_heads)
        self.scale = float(scale)
        self.full = bool(full)
        dev = kv.k_pool.device
        B, Hq = kv.batch, self.Hq
        self.sparse = None if full else EntmaxKVDecoder(kv, num_q_heads, scale, alpha, policy,
                                                        budget_tokens, delta)
        self.cap = kv.max_pages if full else self.sparse.cap
        self.out = torch.empty((B, Hq, kv.head_dim), dtype=torch.float32, device=dev)
        self.lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
        ws = E.entmaxkv_softmax_workspace_size(B, Hq, kv.num_kv_heads, kv.head_dim, kv.page_size,
                                               kv.max_pages, self.cap)
        if ws == 0:
            raise ValueError("invalid sizes for the softmax workspace")
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)

    def build_meta(self, stream=None) -> None:
        if self.sparse is not None:
            self.sparse.build_meta(stream=stream)

    def decode(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        sel = None if self.full else self.sparse.sel
        n_sel = None if self.full else self.sparse.n_sel
        E.entmaxkv_decode_softmax(q, self.Hq, self.scale, self.kv, sel, n_sel, self.cap, self.out,
                                  self.lse, self.workspace, stream)
        return self.out

    def step(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        if self.sparse is not None:
            self.sparse.score(q, stream)
            self.sparse.select(stream)
        return self.decode(q, stream)

    def _step_host_eager(self, q_host, out_host, q_dev, s) -> None:
        with torch.cuda.stream(s):
            q_dev.copy_(q_host, non_blocking=True)
            self.step(q_dev, s)
            out_host.copy_(self.out, non_blocking=True)

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        """q_host (pinned) -> device, the step, out -> out_host (pinned);
        replayed as one CUDA graph."""
        self._host_graph_replay(self._step_host_eager, q_host, out_host, q_dev, stream)
