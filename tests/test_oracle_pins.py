"""Pins for the fp64 CPU oracle, against what the pages and the mathematics fix.

Each test ties one oracle function to something other than itself: hand-derived
values (tests/golden), the variational definition of alpha-entmax, brute force
over supports, library routines (numpy reductions, scipy root finding,
quadrature and constrained optimisation), closed forms, and the identities of
the EntmaxKV page (§2.A upper bound; §3 error bound and support recovery).
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import pytest
from scipy import integrate, optimize

import oracle
from sparse_long_context_08_b300.workloads import bf16_bits_to_f32, make_workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [c.strip() for c in line.split("|")]


# --------------------------------------------------------------------------
# independent helpers (no oracle code): brute force and library routines
# --------------------------------------------------------------------------

def brute_tau(zp, alpha):
    """tau by enumerating every support S and keeping the one whose closed-form
    threshold is consistent (members above it, the rest at or below)."""
    x = np.asarray(zp, dtype=np.float64)
    n = len(x)
    e = 1.0 / (alpha - 1.0)
    found = []
    for r in range(1, n + 1):
        for S in itertools.combinations(range(n), r):
            xs = x[list(S)]
            if e == 1.0:
                t = (xs.sum() - 1.0) / r
            elif e == 2.0:
                a, b, c = r, -2.0 * xs.sum(), (xs ** 2).sum() - 1.0
                disc = b * b - 4 * a * c
                if disc < 0:
                    continue
                t = (-b - math.sqrt(disc)) / (2 * a)
            else:
                g = lambda t: ((xs - t) ** e).sum() - 1.0
                lo_ = xs.max() - 1.0
                if xs.min() <= lo_ or g(xs.min()) > 0:
                    continue  # such a support cannot be consistent
                if g(lo_) <= 0.0:
                    t = lo_  # the top score alone carries all the mass
                else:
                    t = optimize.brentq(g, lo_, xs.min(), xtol=1e-15, rtol=1e-15)
            rest = np.delete(x, list(S))
            if xs.min() > t and (rest.size == 0 or rest.max() <= t + 1e-13):
                found.append(t)
    assert found, "no consistent support"
    assert max(found) - min(found) < 1e-9
    return found[0]


def root_tau(zp, alpha):
    """tau as the root of sum (x - tau)_+^e = 1 by scipy's brentq."""
    x = np.asarray(zp, dtype=np.float64)
    e = 1.0 / (alpha - 1.0)
    f = lambda t: (np.clip(x - t, 0.0, None) ** e).sum() - 1.0
    return optimize.brentq(f, x.max() - 1.0 - 1e-9, x.max(), xtol=1e-15, rtol=1e-15, maxiter=500)


def tsallis_objective(p, z, alpha):
    return p @ z + (1.0 - (p ** alpha).sum()) / (alpha * (alpha - 1.0))


def widen(pool, dtype):
    return bf16_bits_to_f32(pool).astype(np.float64) if dtype == "bf16" else pool.astype(np.float64)


# --------------------------------------------------------------------------
# bf16 widening and metadata  [EntmaxKV §2.A]
# --------------------------------------------------------------------------

def test_bf16_widening_golden(oracle_lib):
    import ctypes as C
    rows = list(_rows("bf16_bits.txt"))
    bits = np.array([int(r[0], 16) for r in rows], dtype=np.uint16)
    want = [float(r[1]) for r in rows]
    for i, w in enumerate(want):
        got = oracle_lib.lib().oracle_widen(bits.ctypes.data_as(C.c_void_p), 1, C.c_int64(i))
        assert got == w and math.copysign(1, got) == math.copysign(1, w), (hex(bits[i]), got, w)
    # the workload module's widening agrees with the same table
    assert np.array_equal(bf16_bits_to_f32(bits).astype(np.float64), np.array(want))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_meta_min_max_mean_var_match_numpy(oracle_lib, dtype):
    w = make_workload("gqa32k", num_q_heads=4, num_kv_heads=2, head_dim=8, page_size=4,
                      batch=2, seq_lens=[37, 20], dtype=dtype, seed=11)
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    K = widen(w.k_pool, dtype)
    for b in range(w.batch):
        for p in range(w.pages_of(b)):
            blk = w.page_table[b, p]
            n = min(w.page_size, int(w.seq_lens[b]) - p * w.page_size)
            for h in range(w.num_kv_heads):
                tile = K[blk, h, :n]
                assert np.array_equal(meta.kmin[blk, h], tile.min(axis=0))
                assert np.array_equal(meta.kmax[blk, h], tile.max(axis=0))
                np.testing.assert_allclose(meta.mean[blk, h], tile.mean(axis=0), rtol=1e-14, atol=1e-15)
                np.testing.assert_allclose(meta.var[blk, h], tile.var(axis=0), rtol=1e-12, atol=1e-15)


def test_meta_arithmetic_progression_closed_form(oracle_lib):
    # keys k_t = a + t c: mean a + c (n-1)/2, population variance c^2 (n^2-1)/12
    w = make_workload("tiny", head_dim=4, page_size=16, seq_lens=[16 + 5], context=21)
    a = np.array([1.0, -2.0, 0.5, 0.0], dtype=np.float32)
    c = np.array([0.25, 1.0, -0.5, 2.0], dtype=np.float32)
    for blk in range(w.num_blocks):
        for t in range(w.page_size):
            w.k_pool[blk, 0, t] = a + t * c
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    for p, n in [(0, 16), (1, 5)]:
        blk = w.page_table[0, p]
        np.testing.assert_allclose(meta.mean[blk, 0], a + c * (n - 1) / 2.0, rtol=0, atol=1e-15)
        np.testing.assert_allclose(meta.var[blk, 0], c.astype(np.float64) ** 2 * (n * n - 1) / 12.0,
                                   rtol=1e-14, atol=1e-15)
        np.testing.assert_array_equal(meta.kmin[blk, 0], np.minimum(a, a + (n - 1) * c))
        np.testing.assert_array_equal(meta.kmax[blk, 0], np.maximum(a, a + (n - 1) * c))


# --------------------------------------------------------------------------
# bounding-box bound  [EntmaxKV §2.A: deterministic upper bound]
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_bbox_bound_dominates_every_token(oracle_lib, dtype):
    w = make_workload("long128k", batch=2, seq_lens=[1000, 769], head_dim=16,
                      num_q_heads=8, num_kv_heads=2, page_size=16, dtype=dtype, seed=5)
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    s = float(w.scale)
    bound = oracle.score_bbox(kv, meta, s)
    K = widen(w.k_pool, dtype)
    G = w.group
    tight = 0
    for b in range(w.batch):
        for h in range(w.num_q_heads):
            q = w.q[b, h].astype(np.float64)
            for p in range(w.pages_of(b)):
                n = min(w.page_size, int(w.seq_lens[b]) - p * w.page_size)
                z = s * (K[w.page_table[b, p], h // G, :n] @ q)
                U = bound[b * w.num_q_heads + h, p]
                assert z.max() <= U + 1e-12 * max(1.0, abs(U))
                tight += n == 1
    assert tight > 0  # the 1-token last page (seq 769) is among them


def test_bbox_bound_is_exact_for_single_token_and_constant_pages(oracle_lib):
    w = make_workload("tiny", head_dim=8, page_size=4, seq_lens=[4 * 6 + 1], context=25, seed=3)
    blk_const = w.page_table[0, 2]
    w.k_pool[blk_const, 0, :] = w.k_pool[blk_const, 0, 0]   # all tokens equal
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    s = float(w.scale)
    bound = oracle.score_bbox(kv, meta, s)
    q = w.q[0, 0].astype(np.float64)
    for p in (2, 6):  # constant page; 1-token last page
        z = s * (w.k_pool[w.page_table[0, p], 0, 0].astype(np.float64) @ q)
        assert abs(bound[0, p] - z) <= 1e-13 * max(1.0, abs(z))


# --------------------------------------------------------------------------
# top-k  [EntmaxKV §2.B.1]
# --------------------------------------------------------------------------

def test_topk_matches_full_sort_with_ties(oracle_lib):
    rng = np.random.default_rng(7)
    w = make_workload("gqa32k", num_q_heads=4, num_kv_heads=1, head_dim=8, page_size=4,
                      batch=3, seq_lens=[4 * 50, 4 * 9 + 2, 4 * 3], seed=2)
    kv = oracle.KV(w)
    bound = np.round(rng.standard_normal((kv.BH, w.max_pages)) * 2) / 2  # many ties
    kp = 10
    sel, n_sel, kth, nxt = oracle.select_topk(kv, bound, kp)
    for bh in range(kv.BH):
        np_ = w.pages_of(bh // w.num_q_heads)
        order = sorted(range(np_), key=lambda p: (-bound[bh, p], p))
        want = sorted(order[:kp])
        assert n_sel[bh] == min(kp, np_)
        assert list(sel[bh, :n_sel[bh]]) == want
        assert kth[bh] == bound[bh, order[min(kp, np_) - 1]]
        assert nxt[bh] == (bound[bh, order[kp]] if kp < np_ else -np.inf)


def test_topk_tie_storm_keeps_lowest_pages(oracle_lib):
    w = make_workload("tiny", head_dim=8, page_size=4, context=4 * 40)
    kv = oracle.KV(w)
    sel, n_sel, _, _ = oracle.select_topk(kv, np.zeros((1, w.max_pages)), 7)
    assert list(sel[0]) == list(range(7))


def test_shared_topk_brute_force_and_group_rows(oracle_lib):
    """GQA-shared selection: brute force over the pages with the group's
    largest bound as the score; every head of a group gets the same rows."""
    rng = np.random.default_rng(11)
    w = make_workload("gqa32k", num_q_heads=8, num_kv_heads=2, head_dim=8, page_size=4,
                      batch=2, seq_lens=[4 * 37, 4 * 6 + 1], seed=3)
    kv = oracle.KV(w)
    bound = np.round(rng.standard_normal((kv.BH, w.max_pages)) * 2) / 2   # many ties
    kp, G = 9, 4
    sel, n_sel, kth, nxt, shared = oracle.select_topk_shared(kv, bound, kp)
    for bh in range(kv.BH):
        b, h = divmod(bh, w.num_q_heads)
        np_ = w.pages_of(b)
        g0 = b * w.num_q_heads + (h // G) * G
        score = [max(bound[g0 + g, p] for g in range(G)) for p in range(np_)]   # by hand
        order = sorted(range(np_), key=lambda p: (-score[p], p))
        k = min(kp, np_)
        assert n_sel[bh] == k
        assert list(sel[bh, :k]) == sorted(order[:k])
        assert kth[bh] == score[order[k - 1]]
        assert nxt[bh] == (score[order[kp]] if kp < np_ else -np.inf)
        assert list(sel[bh, :k]) == list(sel[g0, :k])          # the group's one page set
    # a planted mistake -- the mean instead of the max over the group -- changes a set
    wrong = bound.reshape(-1, G, w.max_pages).mean(axis=1).repeat(G, axis=0)
    s2, n2, _, _ = oracle.select_topk(kv, wrong, kp)
    assert any(list(s2[bh, :n2[bh]]) != list(sel[bh, :n_sel[bh]]) for bh in range(kv.BH))


def test_shared_topk_reduces_to_per_head_topk(oracle_lib):
    """With one query head per kv head (G = 1), or with every head of a group
    holding the same bounds, the shared selection is the per-head top-k."""
    rng = np.random.default_rng(5)
    w1 = make_workload("gqa32k", num_q_heads=4, num_kv_heads=4, head_dim=8, page_size=4,
                       batch=2, seq_lens=[4 * 20, 4 * 7], seed=4)
    kv1 = oracle.KV(w1)
    b1 = rng.standard_normal((kv1.BH, w1.max_pages))
    assert np.array_equal(oracle.select_topk_shared(kv1, b1, 6)[0], oracle.select_topk(kv1, b1, 6)[0])
    w4 = make_workload("gqa32k", num_q_heads=8, num_kv_heads=2, head_dim=8, page_size=4,
                       batch=2, seq_lens=[4 * 20, 4 * 7], seed=4)
    kv4 = oracle.KV(w4)
    b4 = np.repeat(rng.standard_normal((kv4.BH // 4, w4.max_pages)), 4, axis=0)
    assert np.array_equal(oracle.select_topk_shared(kv4, b4, 6)[0], oracle.select_topk(kv4, b4, 6)[0])


# --------------------------------------------------------------------------
# softmax attention (the comparison method)
# --------------------------------------------------------------------------

def _gather(w, b, kvh, pages):
    """Keys and values of the valid tokens of `pages` of sequence b, by hand."""
    K = w.k_pool.astype(np.float64) if w.dtype != "bf16" else bf16_bits_to_f32(w.k_pool).astype(np.float64)
    V = w.v_pool.astype(np.float64) if w.dtype != "bf16" else bf16_bits_to_f32(w.v_pool).astype(np.float64)
    ks, vs = [], []
    for p in pages:
        blk = w.page_table[b, p]
        nt = min(w.page_size, w.seq_lens[b] - p * w.page_size)
        ks.append(K[blk, kvh, :nt]); vs.append(V[blk, kvh, :nt])
    return np.concatenate(ks), np.concatenate(vs)


def test_softmax_decode_brute_force_sparse_and_full(oracle_lib):
    w = make_workload("gqa32k", num_q_heads=4, num_kv_heads=2, head_dim=16, page_size=4,
                      batch=2, seq_lens=[4 * 11 + 3, 4 * 5], seed=9)
    kv = oracle.KV(w)
    rng = np.random.default_rng(2)
    cap = 4
    sel = np.full((kv.BH, cap), -1, np.int32)
    n_sel = np.zeros(kv.BH, np.int32)
    for bh in range(kv.BH):
        np_ = w.pages_of(bh // w.num_q_heads)
        k = min(cap, np_ - 1)
        sel[bh, :k] = np.sort(rng.choice(np_, size=k, replace=False))
        n_sel[bh] = k
    s = float(w.scale)
    out, lse, _ = oracle.decode_softmax(kv, s, sel, n_sel)
    fout, flse, outside = oracle.decode_softmax(kv, s, sel, n_sel, full=True)
    for bh in range(kv.BH):
        b, h = divmod(bh, w.num_q_heads)
        kvh = h // (w.num_q_heads // w.num_kv_heads)
        qv = w.q[b, h].astype(np.float64)
        for pages, o, l in [(sel[bh, :n_sel[bh]], out[bh], lse[bh]),
                            (range(w.pages_of(b)), fout[bh], flse[bh])]:
            Kt, Vt = _gather(w, b, kvh, pages)
            z = s * (Kt @ qv)
            e = np.exp(z - z.max())
            np.testing.assert_allclose(o, (e @ Vt) / e.sum(), rtol=1e-12, atol=1e-12)
            assert abs(l - (z.max() + np.log(e.sum()))) < 1e-12
        # the full softmax's mass outside the kept pages, from the two partition functions
        assert abs(outside[bh] - (1.0 - np.exp(lse[bh] - flse[bh]))) < 1e-12


def test_softmax_decode_constant_keys_is_the_mean_value(oracle_lib):
    w = make_workload("gqa32k", num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=4,
                      batch=1, seq_lens=[4 * 6 - 1], seed=1)
    w.k_pool[:] = w.k_pool[0, 0, 0]
    kv = oracle.KV(w)
    out, lse, _ = oracle.decode_softmax(kv, float(w.scale), full=True)
    _, Vt = _gather(w, 0, 0, range(6))
    for h in range(2):
        np.testing.assert_allclose(out[h], Vt.mean(axis=0), rtol=1e-12, atol=1e-12)
    Kt, _ = _gather(w, 0, 0, [0])
    z0 = float(w.scale) * Kt[0] @ w.q[0, 0].astype(np.float64)
    assert abs(lse[0] - (z0 + np.log(23))) < 1e-10


def test_entmax_decode_tends_to_softmax_decode(oracle_lib):
    """alpha -> 1: the (independently pinned) entmax attention approaches the
    softmax attention over the same kept pages."""
    w = make_workload("gqa32k", num_q_heads=2, num_kv_heads=1, head_dim=16, page_size=4,
                      batch=1, seq_lens=[4 * 8], seed=5)
    kv = oracle.KV(w)
    sel = np.array([[0, 2, 3, 6]] * 2, np.int32)
    n_sel = np.array([4, 4], np.int32)
    so, _, _ = oracle.decode_softmax(kv, float(w.scale), sel, n_sel)
    errs = []
    for a in (1.05, 1.01, 1.002):
        eo, _, _, _ = oracle.decode_sparse(kv, float(w.scale), a, sel, n_sel)
        errs.append(np.abs(eo - so).max())
    assert errs[0] > errs[1] > errs[2] and errs[2] < 5e-3, errs


def test_softmax_decode_ignores_the_physical_layout(oracle_lib):
    w = make_workload("gqa32k", num_q_heads=2, num_kv_heads=1, head_dim=8, page_size=4,
                      batch=1, seq_lens=[4 * 9 - 2], seed=6)
    kv = oracle.KV(w)
    a, la, _ = oracle.decode_softmax(kv, float(w.scale), full=True)
    perm = np.random.default_rng(0).permutation(w.num_blocks)
    k2, v2 = w.k_pool.copy(), w.v_pool.copy()
    w.k_pool[perm] = k2
    w.v_pool[perm] = v2
    w.page_table[:] = perm[w.page_table]
    b, lb, _ = oracle.decode_softmax(oracle.KV(w), float(w.scale), full=True)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(la, lb, rtol=1e-13)


# --------------------------------------------------------------------------
# alpha-entmax threshold
# --------------------------------------------------------------------------

def test_entmax_hand_derived_golden(oracle_lib):
    for alpha, z, p, _ in _rows("entmax_hand.txt"):
        alpha = float(alpha)
        z = np.array([float(v) for v in z.split(",")])
        p = np.array([float(v) for v in p.split(",")])
        got = oracle.entmax(z, alpha)
        np.testing.assert_allclose(got, p, rtol=0, atol=1e-12)
        assert np.all(got[p == 0.0] == 0.0)


@pytest.mark.parametrize("alpha", [2.0, 1.5, 1.25, 3.0])
def test_entmax_tau_brute_force_supports(oracle_lib, alpha):
    rng = np.random.default_rng(int(alpha * 100))
    for n in range(1, 10):
        for _ in range(6):
            zp = rng.standard_normal(n) * rng.choice([0.1, 0.5, 2.0])
            t, k = oracle.entmax_tau(zp, alpha)
            tb = brute_tau(zp, alpha)
            tol = 1e-12 if alpha in (1.5, 2.0) else 1e-11
            assert abs(t - tb) <= tol * max(1.0, abs(tb)), (n, zp, t, tb)
            assert k == int((zp > tb).sum())


@pytest.mark.parametrize("alpha", [1.2, 1.5, 2.0, 2.5])
def test_entmax_is_the_tsallis_maximiser(oracle_lib, alpha):
    rng = np.random.default_rng(3)
    for _ in range(5):
        z = rng.standard_normal(7)
        p = oracle.entmax(z, alpha)
        assert abs(p.sum() - 1.0) < 1e-12 and p.min() >= 0.0
        res = optimize.minimize(lambda x: -tsallis_objective(np.clip(x, 0, None), z, alpha),
                                np.full(7, 1 / 7), method="SLSQP", bounds=[(0, 1)] * 7,
                                constraints={"type": "eq", "fun": lambda x: x.sum() - 1.0},
                                options={"ftol": 1e-14, "maxiter": 500})
        assert tsallis_objective(p, z, alpha) >= -res.fun - 1e-10
        np.testing.assert_allclose(p, np.clip(res.x, 0, None), atol=2e-4)


def test_entmax_approaches_softmax_as_alpha_to_one(oracle_lib):
    z = np.random.default_rng(5).standard_normal(8)
    soft = np.exp(z - z.max())
    soft /= soft.sum()
    errs = [np.abs(oracle.entmax(z, a) - soft).max() for a in (1.1, 1.01, 1.001)]
    assert errs[0] > errs[1] > errs[2]
    assert errs[2] < 2e-3


def test_entmax_sums_to_one_with_exact_zeros(oracle_lib):
    z = np.random.default_rng(9).standard_normal(4096) * 3
    for alpha in (1.5, 2.0, 1.7):
        p = oracle.entmax(z, alpha)
        assert abs(p.sum() - 1.0) < 1e-12
        assert (p == 0.0).sum() > 3000


def test_entmax_large_n_agrees_with_root_finder(oracle_lib):
    rng = np.random.default_rng(21)
    for alpha in (1.5, 2.0, 1.3):
        zp = rng.standard_normal(5000) * 0.3
        t, _ = oracle.entmax_tau(zp, alpha)
        assert abs(t - root_tau(zp, alpha)) < 1e-12


# --------------------------------------------------------------------------
# sparse and full-cache attention  [EntmaxKV §2.C, §3]
# --------------------------------------------------------------------------

def _brute_attention(w, b, h, pages):
    G = w.group
    K = widen(w.k_pool, w.dtype)
    V = widen(w.v_pool, w.dtype)
    q = w.q[b, h].astype(np.float64)
    ks, vs = [], []
    for p in pages:
        n = min(w.page_size, int(w.seq_lens[b]) - p * w.page_size)
        ks.append(K[w.page_table[b, p], h // G, :n])
        vs.append(V[w.page_table[b, p], h // G, :n])
    Kt, Vt = np.concatenate(ks), np.concatenate(vs)
    zp = (w.alpha - 1.0) * (float(w.scale) * (Kt @ q))
    t = root_tau(zp, w.alpha)
    pr = np.clip(zp - t, 0, None) ** (1.0 / (w.alpha - 1.0))
    return pr @ Vt, t


@pytest.mark.parametrize("alpha", [1.5, 2.0, 1.8])
def test_decode_sparse_and_full_match_brute_force(oracle_lib, alpha):
    w = make_workload("long128k", batch=2, seq_lens=[300, 203], num_q_heads=4,
                      num_kv_heads=2, head_dim=16, page_size=8, alpha=alpha, seed=13)
    kv = oracle.KV(w)
    rng = np.random.default_rng(1)
    cap = 6
    sel = np.full((kv.BH, cap), -1, np.int32)
    n_sel = np.zeros(kv.BH, np.int32)
    for bh in range(kv.BH):
        np_ = w.pages_of(bh // w.num_q_heads)
        pick = np.sort(rng.choice(np_, size=cap - bh % 2, replace=False))
        if bh == 1:
            pick = np.array([np_ - 1])  # only the ragged last page
        sel[bh, :len(pick)] = pick
        n_sel[bh] = len(pick)
    out, tau, sup, psum = oracle.decode_sparse(kv, float(w.scale), alpha, sel, n_sel)
    full = oracle.decode_full(kv, float(w.scale), alpha)
    for bh in range(kv.BH):
        b, h = divmod(bh, w.num_q_heads)
        o_ref, t_ref = _brute_attention(w, b, h, sel[bh, :n_sel[bh]])
        np.testing.assert_allclose(out[bh], o_ref, rtol=1e-10, atol=1e-12)
        assert abs(tau[bh] - t_ref) < 1e-11
        assert abs(psum[bh] - 1.0) < 1e-11
        o_full, t_full = _brute_attention(w, b, h, range(w.pages_of(b)))
        np.testing.assert_allclose(full.out[bh], o_full, rtol=1e-10, atol=1e-12)
        assert abs(full.tau[bh] - t_full) < 1e-11


def test_decode_empty_selection(oracle_lib):
    w = make_workload("tiny", head_dim=8, page_size=4, context=64)
    kv = oracle.KV(w)
    out, tau, sup, psum = oracle.decode_sparse(kv, float(w.scale), 1.5,
                                               np.zeros((1, 4), np.int32), np.zeros(1, np.int32))
    assert np.all(out == 0) and tau[0] == np.inf and sup[0] == 0 and psum[0] == 0


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_support_recovery_and_error_bound(oracle_lib, alpha):
    """[EntmaxKV §3]: tau over a kept set is at most the full tau; the output is
    exact when the kept set holds the support; always ||o - o~|| <= 2 B delta;
    and a kept set whose best unkept bound is below tau~ certifies exactness."""
    w = make_workload("long128k", batch=2, context=4096, alpha=alpha, seed=17)
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    bound = oracle.score_bbox(kv, meta, float(w.scale))
    for kp in (8, 32, 128):
        sel, n_sel, kth, nxt = oracle.select_topk(kv, bound, kp)
        out, tau, _, _ = oracle.decode_sparse(kv, float(w.scale), alpha, sel, n_sel)
        full = oracle.decode_full(kv, float(w.scale), alpha, sel, n_sel)
        assert np.all(tau <= full.tau + 1e-12)
        err = np.linalg.norm(full.out - out, axis=1)
        assert np.all(err <= 2 * full.vnorm * full.delta + 1e-12)
        cov = full.covered.astype(bool)
        assert np.all(np.abs(full.out[cov] - out[cov]) <= 1e-12)
        assert np.all(np.abs(full.tau[cov] - tau[cov]) <= 1e-12)
        assert np.all(full.delta[cov] == 0.0)
        assert np.all(full.delta[~cov] > 0.0)
        cert = (alpha - 1.0) * nxt <= tau
        assert np.all(cov[cert])
        if kp == w.cap_pages:
            assert cov.mean() > 0.9  # planted pages make the support recoverable


# --------------------------------------------------------------------------
# Gaussian statistics and tau-hat  [EntmaxKV §2.A, §2.B.2]
# --------------------------------------------------------------------------

@pytest.mark.parametrize("alpha,e", [(1.5, 2), (2.0, 1)])
def test_gaussian_partial_moments_match_quadrature(oracle_lib, alpha, e):
    c = alpha - 1.0
    for m, s, tau in [(0.0, 1.0, 0.0), (0.3, 0.2, 0.1), (-1.0, 0.5, 0.4), (2.0, 0.05, 0.9),
                      (0.5, 3.0, -2.0), (0.7, 0.0, 0.2), (0.1, 0.0, 0.3)]:
        mu, sig = c * m, c * s
        got = oracle.gauss_F([m], [s], [1], alpha, tau) + 1.0
        if sig == 0.0:
            want = max(mu - tau, 0.0) ** e
        else:
            f = lambda y: (y - tau) ** e * math.exp(-0.5 * ((y - mu) / sig) ** 2) / (sig * math.sqrt(2 * math.pi))
            want = integrate.quad(f, tau, max(tau, mu) + 40 * sig, epsabs=1e-14, epsrel=1e-12, limit=200)[0]
        assert abs(got - want) <= 1e-11 * max(1.0, want), (m, s, tau, got, want)
    # textbook values: Y ~ N(0,1), tau = 0
    if e == 2:
        assert abs(oracle.gauss_F([0.0], [2.0], [1], 1.5, 0.0) + 1.0 - 0.5) < 1e-15
    else:
        assert abs(oracle.gauss_F([0.0], [1.0], [1], 2.0, 0.0) + 1.0 - 1 / math.sqrt(2 * math.pi)) < 1e-15


def _gauss_case(seed, n_pages=60):
    rng = np.random.default_rng(seed)
    m = rng.standard_normal(n_pages) * 0.5
    s = np.abs(rng.standard_normal(n_pages)) * 0.3
    n = rng.integers(1, 17, n_pages).astype(np.int32)
    return m, s, n


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_gauss_F_is_decreasing(oracle_lib, alpha):
    m, s, n = _gauss_case(1)
    taus = np.linspace(-3, 3, 301)
    F = np.array([oracle.gauss_F(m, s, n, alpha, t) for t in taus])
    assert np.all(np.diff(F) <= 1e-15)
    assert F[0] > 0 > F[-1]


def _one_head_workload(n_pages, P=16):
    return make_workload("gauss64k", batch=1, num_q_heads=1, num_kv_heads=1, head_dim=8,
                         page_size=P, context=n_pages * P, flat_heads=(), planted_pages=0)


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_tau_hat_is_the_root_of_F(oracle_lib, alpha):
    w = _one_head_workload(60)
    kv = oracle.KV(w)
    m, s, _ = _gauss_case(4)
    n = np.full(60, 16, np.int32)
    sel, n_sel, th, zmax = oracle.select_gauss(kv, m[None], s[None], alpha, 0.1, 60)
    root = optimize.brentq(lambda t: oracle.gauss_F(m, s, n, alpha, t), -10, 10, xtol=1e-15, rtol=1e-15)
    assert abs(th[0] - root) < 1e-12
    # estimated max: m + sqrt(2 ln n) s for n = 16 tokens
    np.testing.assert_allclose(zmax[0], m + math.sqrt(2 * math.log(16)) * s, rtol=1e-15)


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_tau_hat_with_zero_variance_is_exact_tau(oracle_lib, alpha):
    """With constant pages every token of page p scores m_p, so the Gaussian
    normalisation is exact and tau-hat equals the exact threshold of the
    multiset {(alpha-1) m_p repeated n_p}."""
    w = _one_head_workload(12, P=4)
    kv = oracle.KV(w)
    m = np.random.default_rng(8).standard_normal(12) * 0.4
    sel, n_sel, th, _ = oracle.select_gauss(kv, m[None], np.zeros((1, 12)), alpha, 0.0, 12)
    zp = np.repeat((alpha - 1.0) * m, 4)
    assert abs(th[0] - root_tau(zp, alpha)) < 1e-12
    # delta = 0 keeps exactly the pages carrying support (plus the ones at tau)
    keep = set(sel[0, :n_sel[0]])
    assert keep == {p for p in range(12) if (alpha - 1.0) * m[p] >= th[0]}


def test_gauss_select_margin_cap_and_fallback(oracle_lib):
    w = _one_head_workload(60)
    kv = oracle.KV(w)
    m, s, _ = _gauss_case(6)
    alpha = 1.5
    _, n_all, _, zmax = oracle.select_gauss(kv, m[None], s[None], alpha, 1e6, 25)
    assert n_all[0] == 25
    sel, n1, _, _ = oracle.select_gauss(kv, m[None], s[None], alpha, -1e6, 25)
    assert n1[0] == 1 and sel[0, 0] == int(np.argmax(zmax[0]))
    sel, n_cap, _, _ = oracle.select_gauss(kv, m[None], s[None], alpha, 1e6, 5)
    want = sorted(sorted(range(60), key=lambda p: (-zmax[0, p], p))[:5])
    assert list(sel[0, :5]) == want
    # a larger margin never keeps fewer pages
    counts = [oracle.select_gauss(kv, m[None], s[None], alpha, d, 60)[1][0] for d in (0.0, 0.1, 0.3, 1.0)]
    assert counts == sorted(counts)


def test_gauss_meta_statistics_match_token_scores(oracle_lib):
    """m_p and s_p are the mean and standard deviation of the page's token scores
    under the diagonal (independent-coordinate) model: with one coordinate the
    model is exact, so they equal numpy's mean/std of s q k_t."""
    w = make_workload("gauss64k", batch=1, num_q_heads=2, num_kv_heads=1, head_dim=1,
                      page_size=8, seq_lens=[8 * 5 + 3], context=43, flat_heads=(), planted_pages=0)
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    m, s = oracle.score_gauss(kv, meta, float(w.scale))
    K = widen(w.k_pool, w.dtype)
    for h in range(2):
        for p in range(w.pages_of(0)):
            n = min(8, 43 - 8 * p)
            z = float(w.scale) * K[w.page_table[0, p], 0, :n, 0] * float(w.q[0, h, 0])
            assert abs(m[h, p] - z.mean()) < 1e-12
            assert abs(s[h, p] - z.std()) < 1e-12


def _uncorrelated_pages(w, seed=5):
    """Overwrite every page of a one-kv-head fp32 workload with keys whose
    coordinates are exactly uncorrelated over the page's tokens: coordinate j
    of token t is c_j + a_j H[t, j + 1], with H a Sylvester-Hadamard matrix of
    the page's order (rows shuffled per page).  Its columns other than the
    first are +-1 vectors with zero mean and mutually orthogonal, so each
    coordinate has mean c_j and population variance a_j^2, and the sample
    covariance of two coordinates is exactly 0.  c and a are dyadic, so every
    key is exact in fp32.  Returns the per-block (c, a)."""
    from scipy.linalg import hadamard
    P, d = w.page_size, w.head_dim
    H = hadamard(P).astype(np.float64)
    rng = np.random.default_rng(seed)
    ca = {}
    for blk in range(w.num_blocks):
        c = np.array([0.125 * ((3 * j + blk) % 7 - 3) for j in range(d)])
        a = np.array([0.25 * (1 + (j + 2 * blk) % 5) for j in range(d)])
        rows = H[rng.permutation(P)]
        w.k_pool[blk, 0] = (c[None, :] + a[None, :] * rows[:, 1:d + 1]).astype(np.float32)
        ca[blk] = (c, a)
    return ca


def test_gauss_meta_statistics_match_token_scores_multidim(oracle_lib):
    """[EntmaxKV] §2.A, Gaussian page statistics at d = 12: on pages whose
    coordinates are exactly uncorrelated, the diagonal model is exact, so m_p
    and s_p must equal numpy's mean and population std of the token scores
    s q.k_t.  The same check rejects the two plausible slips of the spread: the
    sum of per-coordinate standard deviations s sum_j |q_j| sd_j, and q_j not
    squared."""
    w = make_workload("gauss64k", batch=1, num_q_heads=3, num_kv_heads=1, head_dim=12,
                      page_size=16, seq_lens=[16 * 6], context=96, dtype="f32", flat_heads=(),
                      planted_pages=0, seed=21)
    ca = _uncorrelated_pages(w)
    kv = oracle.KV(w)
    meta = oracle.build_meta(kv)
    m, s = oracle.score_gauss(kv, meta, float(w.scale))
    K = w.k_pool.astype(np.float64)
    sc = float(w.scale)
    for blk, (c, a) in ca.items():          # the metadata itself is exact here
        np.testing.assert_allclose(meta.mean[blk, 0], c, rtol=0, atol=1e-15)
        np.testing.assert_allclose(meta.var[blk, 0], a * a, rtol=0, atol=1e-15)
    checked = 0
    for h in range(w.num_q_heads):
        qh = w.q[0, h].astype(np.float64)
        for p in range(w.pages_of(0)):
            blk = w.page_table[0, p]
            z = sc * (K[blk, 0] @ qh)
            scale_z = sc * (np.abs(qh) @ (np.abs(ca[blk][0]) + ca[blk][1]))
            assert abs(m[h, p] - z.mean()) <= 1e-12 * scale_z
            assert abs(s[h, p] - z.std()) <= 1e-12 * scale_z
            # the slips this pins: each misses numpy's std by far more than 1e-12
            sd = np.sqrt(meta.var[blk, 0])
            sum_of_sd = sc * (np.abs(qh) @ sd)
            unsquared_q = sc * np.sqrt(np.abs(qh) @ meta.var[blk, 0])
            assert abs(sum_of_sd - z.std()) > 1e-3 * z.std()
            assert abs(unsquared_q - z.std()) > 1e-3 * z.std()
            checked += 1
    assert checked == w.num_q_heads * 6
