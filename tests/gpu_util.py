"""Helpers shared by the GPU parity tests: run the CUDA path through the binding,
run the fp64 oracle on the same seeded inputs, and compare with the stated
tolerances.

Tolerances (fp32 kernels against the fp64 oracle; bf16 K/V widened exactly on
both sides):
  kmin/kmax             bit-exact
  mean, var             |d| <= 1e-5 * (mean |k| resp. var + 1e-6)
  page bound / (m, s)   |d| <= 1e-5 * s * sum_j |q_j| max(|kmin_j|, |kmax_j|)
  page selection        identical sets, except pages whose fp64 score lies within
                        2e-5 (relative to that scale) of the decision boundary
                        (k-th bound, or tau-hat - delta); such ties are reported
  tau                   |d| <= 1e-5 * max(|tau|, 1)
  out                   |d| <= 1e-4 + 2e-3 |out|
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_long_context_08_b300 import entmaxkv as E
from sparse_long_context_08_b300.api import EntmaxKVDecoder, upload_workload
from sparse_long_context_08_b300.workloads import bf16_bits_to_f32

TAU_RTOL = 1e-5
OUT_RTOL, OUT_ATOL = 2e-3, 1e-4
SCORE_RTOL = 1e-5
TIE_RTOL = 2e-5


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return bf16_bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16)).astype(np.float64)
    return t.cpu().numpy()


class DeviceRun:
    """The CUDA pipeline on one workload, plus numpy copies of every stage."""

    def __init__(self, w, device="cuda"):
        self.w = w
        self.kv, self.q = upload_workload(w, device)
        self.dec = EntmaxKVDecoder(self.kv, w.num_q_heads, float(w.scale), w.alpha, w.policy,
                                   w.budget_tokens, w.delta)
        self.dec.build_meta()

    def step(self):
        self.dec.step(self.q)
        torch.cuda.synchronize()
        d = self.dec
        r = dict(page_scores=d.page_scores.cpu().numpy().astype(np.float64),
                 sel=d.sel.cpu().numpy(), n_sel=d.n_sel.cpu().numpy(),
                 aux=d.aux.cpu().numpy().astype(np.float64),
                 out=d.out.cpu().numpy().astype(np.float64),
                 tau=d.tau.cpu().numpy().astype(np.float64),
                 support=d.support.cpu().numpy())
        BH = self.w.batch * self.w.num_q_heads
        for k in ("page_scores", "sel", "n_sel", "aux", "out", "tau", "support"):
            r[k] = r[k].reshape((BH,) + r[k].shape[2:])
        return r

    def decode_with(self, sel: np.ndarray, n_sel: np.ndarray):
        """Run only the decode stage on a given selection (e.g. the oracle's)."""
        d = self.dec
        B, Hq = self.w.batch, self.w.num_q_heads
        d.sel.copy_(torch.from_numpy(np.ascontiguousarray(sel, np.int32)).view(B, Hq, -1))
        d.n_sel.copy_(torch.from_numpy(np.ascontiguousarray(n_sel, np.int32)).view(B, Hq))
        d.decode(self.q)
        torch.cuda.synchronize()
        BH = B * Hq
        return (d.out.cpu().numpy().astype(np.float64).reshape(BH, -1),
                d.tau.cpu().numpy().astype(np.float64).reshape(BH),
                d.support.cpu().numpy().reshape(BH))

    def meta(self):
        m = self.dec.meta
        return {k: None if getattr(m, k) is None else to_np(getattr(m, k))
                for k in ("kmin", "kmax", "mean", "var")}


def valid_blocks(w):
    blks = []
    for b in range(w.batch):
        blks.extend(w.page_table[b, :w.pages_of(b)].tolist())
    return np.array(sorted(blks), dtype=np.int64)


def bbox_scale(w, ometa, heads=None):
    """s * sum_j |q_j| max(|kmin_j|, |kmax_j|) per (head, page): the magnitude
    the fp32 bound is accurate relative to."""
    BH = w.batch * w.num_q_heads
    G = w.group
    out = np.ones((BH, w.max_pages))
    amp = np.maximum(np.abs(ometa.kmin), np.abs(ometa.kmax))
    for bh in (range(BH) if heads is None else heads):
        b, h = divmod(bh, w.num_q_heads)
        np_ = w.pages_of(b)
        blk = w.page_table[b, :np_]
        out[bh, :np_] = float(w.scale) * (amp[blk, h // G] @ np.abs(w.q[b, h].astype(np.float64)))
    return out


def gauss_scale(w, ometa, heads=None):
    BH = w.batch * w.num_q_heads
    G = w.group
    out = np.ones((BH, w.max_pages))
    for bh in (range(BH) if heads is None else heads):
        b, h = divmod(bh, w.num_q_heads)
        np_ = w.pages_of(b)
        blk = w.page_table[b, :np_]
        qa = np.abs(w.q[b, h].astype(np.float64))
        m = float(w.scale) * (np.abs(ometa.mean[blk, h // G]) @ qa)
        s = float(w.scale) * np.sqrt(ometa.var[blk, h // G] @ (qa * qa))
        out[bh, :np_] = m + s + 1e-6
    return out


def compare_meta(w, gm, om):
    blk = valid_blocks(w)
    if gm["kmin"] is not None:
        assert np.array_equal(gm["kmin"][blk], om.kmin[blk]), "kmin not bit-exact"
        assert np.array_equal(gm["kmax"][blk], om.kmax[blk]), "kmax not bit-exact"
    if gm["mean"] is not None:
        K = w.k_pool
        scale_m = np.abs(om.mean[blk]) + np.sqrt(om.var[blk]) + 1e-6
        assert np.all(np.abs(gm["mean"][blk] - om.mean[blk]) <= 1e-5 * scale_m)
        assert np.all(np.abs(gm["var"][blk] - om.var[blk]) <= 1e-5 * (om.var[blk] + scale_m ** 2 * 1e-2))


def compare_scores(w, got, ref, mag, heads):
    for bh in heads:
        np_ = w.pages_of(bh // w.num_q_heads)
        g, r, m = got[bh, :np_], ref[bh, :np_], mag[bh, :np_]
        bad = np.abs(g - r) > SCORE_RTOL * m
        assert not bad.any(), (bh, np.nonzero(bad)[0][:5], g[bad][:5], r[bad][:5])


def compare_selection(w, g_sel, g_n, o_sel, o_n, score, mag, boundary, heads):
    """Sets must agree except on pages within TIE_RTOL of the boundary score."""
    ties = 0
    for bh in heads:
        gs = set(g_sel[bh, :g_n[bh]].tolist())
        os_ = set(o_sel[bh, :o_n[bh]].tolist())
        assert list(g_sel[bh, :g_n[bh]]) == sorted(gs), "selection not ascending/distinct"
        diff = gs ^ os_
        for p in diff:
            assert abs(score[bh, p] - boundary[bh]) <= TIE_RTOL * max(mag[bh, p], 1e-30), \
                (bh, p, score[bh, p], boundary[bh])
        ties += len(diff) > 0
    return ties


# Heads whose GPU page selection differs from the oracle's only by pages tied at
# the decision boundary, per test (printed at the end of the session).
TIES: list[tuple[str, int, int]] = []


def record_ties(name: str, heads: int, ties: int) -> None:
    TIES.append((name, heads, ties))


def selected_scores(w, sel, n_sel, bh):
    """fp64 z' = (alpha - 1) s q.k of every valid token of head bh's selected
    pages (K widened exactly)."""
    b, h = divmod(bh, w.num_q_heads)
    pages = sel[bh, :n_sel[bh]]
    K = w.k_pool[w.page_table[b, pages], h // w.group]          # [n, P, d]
    K = bf16_bits_to_f32(K) if w.dtype == "bf16" else K
    q = w.q[b, h].astype(np.float64)
    z = [K[j, :min(w.page_size, int(w.seq_lens[b]) - int(p) * w.page_size)].astype(np.float64) @ q
         for j, p in enumerate(pages)]
    z = np.concatenate(z) if z else np.zeros(0)
    return (w.alpha - 1.0) * float(w.scale) * z


def compare_support(w, sel, n_sel, g_sup, o_sup, o_tau, heads):
    """Support sizes (#{p > 0}) agree, except by tokens whose fp64 score lies
    within the tau tolerance band of the oracle's tau: only such a token can
    change sides between the fp32 and the fp64 threshold."""
    for bh in heads:
        if int(g_sup[bh]) == int(o_sup[bh]):
            continue
        assert np.isfinite(o_tau[bh]), (bh, g_sup[bh], o_sup[bh])
        zp = selected_scores(w, sel, n_sel, bh)
        band = TAU_RTOL * max(abs(o_tau[bh]), 1.0)
        near = int(np.sum(np.abs(zp - o_tau[bh]) <= band))
        assert abs(int(g_sup[bh]) - int(o_sup[bh])) <= near, (bh, g_sup[bh], o_sup[bh], near)


def compare_decode(g_out, g_tau, o_out, o_tau, heads, g_sup=None, o_sup=None):
    for bh in heads:
        if np.isinf(o_tau[bh]):
            assert np.isinf(g_tau[bh]) and np.all(g_out[bh] == 0)
            continue
        assert abs(g_tau[bh] - o_tau[bh]) <= TAU_RTOL * max(abs(o_tau[bh]), 1.0), \
            (bh, g_tau[bh], o_tau[bh])
        err = np.abs(g_out[bh] - o_out[bh])
        ok = err <= OUT_ATOL + OUT_RTOL * np.abs(o_out[bh])
        assert ok.all(), (bh, err.max(), np.nonzero(~ok)[0][:5])
    if g_sup is not None:
        hs = list(heads)
        same = np.mean([g_sup[bh] == o_sup[bh] for bh in hs])
        assert same >= 0.95, same
        assert all(abs(int(g_sup[bh]) - int(o_sup[bh])) <= 2 for bh in hs)
