"""A decoder object over the C ABI: owns the device buffers of one decode
configuration and runs score -> select -> decode on the current stream.

Marshalling only; every stage runs in libentmaxkv.so.
"""
from __future__ import annotations

import numpy as np
import torch

from . import entmaxkv as E


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


class EntmaxKVDecoder:
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

    def step(self, q: torch.Tensor, stream=None) -> torch.Tensor:
        """One decode step for device-resident q [B, Hq, d]; returns `out` (device)."""
        self.score(q, stream)
        self.select(stream)
        return self.decode(q, stream)

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        """One decode step from host memory: q_host (pinned) -> device, the three
        stages, then out -> out_host (pinned).  Asynchronous on `stream`."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            q_dev.copy_(q_host, non_blocking=True)
            self.step(q_dev, s)
            out_host.copy_(self.out, non_blocking=True)


class EntmaxKVFullDecoder:
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

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        """q_host (pinned) -> device, the full-cache decode, out -> out_host
        (pinned).  Asynchronous on `stream`."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            q_dev.copy_(q_host, non_blocking=True)
            self.decode(q_dev, s)
            out_host.copy_(self.out, non_blocking=True)


class EntmaxKVSoftmaxDecoder:
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

    def step_host(self, q_host: torch.Tensor, out_host: torch.Tensor, q_dev: torch.Tensor,
                  stream=None) -> None:
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            q_dev.copy_(q_host, non_blocking=True)
            self.step(q_dev, s)
            out_host.copy_(self.out, non_blocking=True)
