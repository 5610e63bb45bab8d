"""Discarded mass and support retention of the kept pages, alpha-entmax
against softmax ("Riepilogo Tecnico: EntmaxKV", §3 error bound and §4
comparison with truncated softmax), measured on the GPU.

For the pages I that the EntmaxKV scoring and selection keep, per query head:
- entmax: delta = the full-cache alpha-entmax's mass on tokens outside I.  The
  page bounds the output error by 2 B delta, and delta = 0 exactly when I
  holds the full-cache support (the sparse output is then exact);
- softmax: the full-cache softmax's mass outside I = 1 - e^(lse_I - lse_all).
  It is never 0, since every token has a positive weight.

Run as ``python -m sparse_long_context_08_b300.mass --workload long128k`` for a
JSON summary per workload.
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

from . import entmaxkv as E
from .api import EntmaxKVDecoder, EntmaxKVFullDecoder, upload_workload
from .workloads import CONFIGS, make_workload

# delta at or below this counts as "support kept" (fp32 scores and thresholds)
RECOVERED_TOL = 1e-5


def measure(w, device: str = "cuda") -> dict:
    """Per-head arrays: entmax delta, support kept, softmax mass outside the
    kept pages, kept tokens; plus the GPU's selection (sel, n_sel)."""
    kv, q = upload_workload(w, device)
    B, Hq, Hkv = w.batch, w.num_q_heads, w.num_kv_heads
    sp = EntmaxKVDecoder(kv, Hq, float(w.scale), w.alpha, w.policy, w.budget_tokens, w.delta)
    sp.build_meta()
    sp.step(q)
    full = EntmaxKVFullDecoder(kv, Hq, float(w.scale), w.alpha)
    full.decode(q)
    mass = torch.empty_like(full.tau)
    E.entmaxkv_kept_mass(sp.workspace, B, Hq, Hkv, w.head_dim, w.page_size, w.max_pages, sp.cap,
                         w.alpha, full.tau, mass)
    # softmax on the same kept pages, and over every token
    ws_s = torch.empty(E.entmaxkv_softmax_workspace_size(B, Hq, Hkv, w.head_dim, w.page_size,
                                                         w.max_pages, sp.cap),
                       dtype=torch.uint8, device=kv.k_pool.device)
    out_s = torch.empty_like(sp.out)
    lse_kept = torch.empty_like(full.tau)
    E.entmaxkv_decode_softmax(q, Hq, float(w.scale), kv, sp.sel, sp.n_sel, sp.cap, out_s, lse_kept,
                              ws_s)
    ws_f = torch.empty(E.entmaxkv_softmax_workspace_size(B, Hq, Hkv, w.head_dim, w.page_size,
                                                         w.max_pages, w.max_pages),
                       dtype=torch.uint8, device=kv.k_pool.device)
    lse_all = torch.empty_like(full.tau)
    E.entmaxkv_decode_softmax(q, Hq, float(w.scale), kv, None, None, w.max_pages, out_s, lse_all,
                              ws_f)
    torch.cuda.synchronize()
    BH = B * Hq
    delta = np.clip(1.0 - mass.cpu().numpy().astype(np.float64).reshape(BH), 0.0, 1.0)
    sm_out = np.clip(-np.expm1(lse_kept.cpu().numpy().astype(np.float64)
                               - lse_all.cpu().numpy().astype(np.float64)).reshape(BH), 0.0, 1.0)
    n_sel = sp.n_sel.cpu().numpy().reshape(BH)
    kept = np.array([min(int(n_sel[bh]) * w.page_size, int(w.seq_lens[bh // Hq]))
                     for bh in range(BH)])
    return {"delta": delta, "recovered": delta <= RECOVERED_TOL, "softmax_outside": sm_out,
            "kept_tokens": kept, "sel": sp.sel.cpu().numpy().reshape(BH, -1), "n_sel": n_sel,
            "support_full": full.support.cpu().numpy().reshape(BH)}


def summary(w, m: dict) -> dict:
    def stats(x):
        return {"mean": float(np.mean(x)), "median": float(np.median(x)),
                "p95": float(np.percentile(x, 95)), "max": float(np.max(x))}
    ctx = int(max(w.seq_lens))
    return {"workload": w.name, "heads": int(len(m["delta"])), "context": ctx,
            "policy": w.policy, "alpha": w.alpha,
            "kept_tokens_per_head": stats(m["kept_tokens"]),
            "entmax": {"support_kept_fraction": float(np.mean(m["recovered"])),
                       "full_support_tokens": stats(m["support_full"]),
                       "delta": stats(m["delta"])},
            "softmax": {"mass_outside": stats(m["softmax_outside"])}}


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", action="append", choices=sorted(CONFIGS))
    ap.add_argument("--alpha", type=float, default=None)
    args = ap.parse_args()
    for name in args.workload or ["tiny", "gqa32k", "long128k", "ctx1m", "gauss64k"]:
        w = make_workload(name, **({"alpha": args.alpha} if args.alpha else {}))
        print(json.dumps(summary(w, measure(w))), flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
