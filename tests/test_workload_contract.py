"""The very-long-context workload's own contract, checked with the oracle on the
host: keys are clustered so that every query head's full-cache alpha-entmax
support spans at most 64 pages (the 1M-token decode configuration: batch 1,
32 query / 8 kv heads, d = 128, pages of 32 tokens, alpha = 1.5)."""
from __future__ import annotations

import numpy as np

import oracle
from sparse_long_context_08_b300.workloads import make_workload


def test_ctx1m_support_spans_at_most_64_pages():
    w = make_workload("ctx1m")
    assert w.params["context"] == 1048576 and w.page_size == 32 and w.alpha == 1.5
    kv = oracle.KV(w)
    heads = np.arange(w.batch * w.num_q_heads, dtype=np.int32)
    f = oracle.decode_full(kv, float(w.scale), w.alpha, heads=heads)
    assert np.all(f.support_pages >= 1)
    assert np.all(f.support_pages <= 64), f.support_pages.max()
    # the decode's budget (128 pages) can hold every head's support
    assert np.all(f.support_pages <= w.cap_pages)
