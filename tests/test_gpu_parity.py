"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, stage by
stage, on seeded workloads that span several tiles and ragged tails, plus the
edge cases the method has.  Tolerances: tests/gpu_util.py."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from sparse_long_context_08_b300 import entmaxkv as E
from sparse_long_context_08_b300.workloads import make_workload

from gpu_util import (DeviceRun, bbox_scale, compare_decode, compare_meta, compare_scores,
                      compare_selection, compare_support, gauss_scale, record_ties)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from sparse_long_context_08_b300 import build
    build.build()
    oracle.lib()


def full_parity(w, heads=None, check_e2e=True):
    """Every stage of one decode step against the oracle; returns report dict."""
    g = DeviceRun(w)
    r = g.step()
    kv = oracle.KV(w)
    om = oracle.build_meta(kv)
    compare_meta(w, g.meta(), om)
    BH = w.batch * w.num_q_heads
    hs = list(range(BH)) if heads is None else list(heads)
    s = float(w.scale)
    rep = {}
    if w.policy in ("topk", "topk_shared"):
        G = w.group
        # the shared score needs the bounds of every head of each sampled group
        hb = hs if w.policy == "topk" else sorted({bh // G * G + g for bh in hs for g in range(G)})
        ob = oracle.score_bbox(kv, om, s, heads=hb)
        mag = bbox_scale(w, om, hb)
        compare_scores(w, r["page_scores"], ob, mag, hb)
        if w.policy == "topk":
            osel, on, okth, onext = oracle.select_topk(kv, ob, w.cap_pages, heads=hs)
            score = ob
        else:
            osel, on, okth, onext, score = oracle.select_topk_shared(kv, ob, w.cap_pages, heads=hs)
            mag = mag.reshape(-1, G, mag.shape[1]).max(axis=1).repeat(G, axis=0)
            for bh in hs:                       # one page set per kv head
                g0 = bh // G * G
                assert np.array_equal(r["sel"][bh, :r["n_sel"][bh]], r["sel"][g0, :r["n_sel"][g0]])
        rep["ties"] = compare_selection(w, r["sel"], r["n_sel"], osel, on, score, mag, okth, hs)
        for bh in hs:
            assert r["n_sel"][bh] == on[bh]
            if on[bh] < w.pages_of(bh // w.num_q_heads):
                assert abs(r["aux"][bh, 0] - okth[bh]) <= 1e-5 * mag[bh].max()
    else:
        om_, os_ = oracle.score_gauss(kv, om, s, heads=hs)
        mag = gauss_scale(w, om, hs)
        compare_scores(w, r["page_scores"][..., 0], om_, mag, hs)
        compare_scores(w, r["page_scores"][..., 1], os_, mag, hs)
        osel, on, oth, ozmax = oracle.select_gauss(kv, om_, os_, w.alpha, w.delta, w.cap_pages,
                                                   heads=hs)
        for bh in hs:
            assert abs(r["aux"][bh, 0] - oth[bh]) <= 1e-5 * max(1.0, abs(oth[bh])), \
                (bh, r["aux"][bh, 0], oth[bh])
        # the decision score is (alpha-1) zmax against tau-hat - delta, or the
        # cap's k-th zmax; report either kind of boundary tie
        c = w.alpha - 1.0
        zs = c * ozmax
        bnd = np.full(BH, np.nan)
        for bh in hs:
            np_ = w.pages_of(bh // w.num_q_heads)
            passing = np.sort(zs[bh, :np_][zs[bh, :np_] >= oth[bh] - w.delta])[::-1]
            bnd[bh] = passing[w.cap_pages - 1] if len(passing) > w.cap_pages else oth[bh] - w.delta
        rep["ties"] = compare_selection(w, r["sel"], r["n_sel"], osel, on, zs, c * mag, bnd, hs)
    # decode on the oracle's own selection
    g_out, g_tau, g_sup = g.decode_with(osel, on)
    o_out, o_tau, o_sup, o_psum = oracle.decode_sparse(kv, s, w.alpha, osel, on, heads=hs)
    compare_decode(g_out, g_tau, o_out, o_tau, hs)
    compare_support(w, osel, on, g_sup, o_sup, o_tau, hs)
    # end to end: where the two selections agree, the outputs agree
    if check_e2e:
        same = [bh for bh in hs if r["n_sel"][bh] == on[bh]
                and np.array_equal(r["sel"][bh, :on[bh]], osel[bh, :on[bh]])]
        assert len(same) >= 0.9 * len(hs)
        compare_decode(r["out"], r["tau"], o_out, o_tau, same)
    assert E.entmaxkv_read_device_status() == E.EKV_OK
    rep["support"] = o_sup
    record_ties(w.name, len(hs), rep["ties"])
    return rep


# ---------------------------------------------------------------------------
# the five workloads at oracle-friendly sizes (ragged tails included)
# ---------------------------------------------------------------------------

def test_tiny_full_size():
    full_parity(make_workload("tiny"))


def test_tiny_ragged_tail():
    full_parity(make_workload("tiny", seq_lens=[4096 - 7], context=4089))


def test_gqa_reduced_context_ragged():
    full_parity(make_workload("gqa32k", batch=2, seq_lens=[8192, 5000]))


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_long128k_reduced(alpha):
    full_parity(make_workload("long128k", batch=2, seq_lens=[16384, 12345], alpha=alpha))


@pytest.mark.parametrize("over", [
    {"batch": 2, "seq_lens": [16384, 12345]},
    {"batch": 2, "seq_lens": [16384, 12345], "alpha": 2.0, "num_q_heads": 16, "num_kv_heads": 2},
    {"batch": 3, "seq_lens": [5 * 32, 20, 1], "budget_tokens": 4096, "planted_pages": 0},
])
def test_shared_selection_reduced(over):
    """GQA-shared selection: one page set per kv head, ranked by the group's
    largest bound; decode unchanged."""
    full_parity(make_workload("long128k", policy="topk_shared", **over))


def test_ctx1m_reduced():
    full_parity(make_workload("ctx1m", context=65536))


@pytest.mark.parametrize("alpha", [1.5, 2.0])
def test_gauss_reduced(alpha):
    full_parity(make_workload("gauss64k", batch=2, seq_lens=[16384, 9999], alpha=alpha))


# ---------------------------------------------------------------------------
# the five workloads at their full sizes, through the same decoder and launch
# shapes the benchmark uses; the oracle checks a seeded sample of query heads
# (every stage of those heads: bounds, selection, tau, output) and the page
# metadata of every block
# ---------------------------------------------------------------------------

def sampled_heads(w, n, seed=11):
    BH = w.batch * w.num_q_heads
    rng = np.random.default_rng(seed)
    return sorted(rng.choice(BH, size=min(n, BH), replace=False).tolist())


@pytest.mark.parametrize("name,alpha,policy", [
    ("tiny", 1.5, None), ("gqa32k", 1.5, None), ("long128k", 1.5, None), ("long128k", 2.0, None),
    ("ctx1m", 1.5, None), ("gauss64k", 1.5, None), ("long128k", 1.5, "topk_shared")])
def test_full_size_sampled_heads(name, alpha, policy):
    w = make_workload(name, alpha=alpha, **({"policy": policy} if policy else {}))
    full_parity(w, heads=sampled_heads(w, 64))
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# full-cache decode (every valid token) against the oracle's full attention
# ---------------------------------------------------------------------------

def full_cache_parity(w, heads=None):
    from sparse_long_context_08_b300.api import EntmaxKVFullDecoder, upload_workload
    kv_d, q = upload_workload(w)
    dec = EntmaxKVFullDecoder(kv_d, w.num_q_heads, float(w.scale), w.alpha)
    dec.decode(q)
    torch.cuda.synchronize()
    BH = w.batch * w.num_q_heads
    out = dec.out.cpu().numpy().astype(np.float64).reshape(BH, -1)
    tau = dec.tau.cpu().numpy().astype(np.float64).reshape(BH)
    sup = dec.support.cpu().numpy().reshape(BH)
    hs = list(range(BH)) if heads is None else list(heads)
    kv = oracle.KV(w)
    f = oracle.decode_full(kv, float(w.scale), w.alpha, heads=hs)
    compare_decode(out, tau, f.out, f.tau, hs, sup, f.support)
    assert E.entmaxkv_read_device_status() == E.EKV_OK
    return sup[hs]


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("tiny", {"seq_lens": [4096 - 7], "context": 4089}),
    ("gqa32k", {"batch": 2, "seq_lens": [8192, 5000]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345], "alpha": 2.0}),
    ("long128k", {"batch": 1, "context": 8192, "alpha": 1.3, "seed": 7}),
    ("gauss64k", {"batch": 2, "seq_lens": [16384, 9999]}),
])
def test_full_cache_reduced(name, over):
    full_cache_parity(make_workload(name, **over))


@pytest.mark.parametrize("name", ["gqa32k", "long128k", "ctx1m"])
def test_full_cache_full_size_sampled_heads(name):
    w = make_workload(name)
    full_cache_parity(w, heads=sampled_heads(w, 48))
    torch.cuda.empty_cache()


def test_large_selection_uses_global_candidates():
    """A budget larger than the shared-memory candidate buffer (cap * P >
    16384 tokens) goes through the global-buffer threshold kernel: same
    parity with the oracle on the same selection."""
    w = make_workload("long128k", batch=2, seq_lens=[32768 * 2, 40000], budget_tokens=32768,
                      planted_pages=4)
    assert w.cap_pages * w.page_size > 16384
    full_parity(w)


# ---------------------------------------------------------------------------
# softmax attention (the comparison method) against the oracle's softmax
# ---------------------------------------------------------------------------

LSE_TOL = 1e-5


def softmax_parity(w, heads=None, full=False):
    from sparse_long_context_08_b300.api import EntmaxKVSoftmaxDecoder, upload_workload
    kv_d, q = upload_workload(w)
    dec = EntmaxKVSoftmaxDecoder(kv_d, w.num_q_heads, float(w.scale), w.policy, w.budget_tokens,
                                 w.delta, w.alpha, full=full)
    dec.build_meta()
    BH = w.batch * w.num_q_heads
    hs = list(range(BH)) if heads is None else list(heads)
    kv = oracle.KV(w)
    if full:
        dec.decode(q)
        o_out, o_lse, _ = oracle.decode_softmax(kv, float(w.scale), full=True, heads=hs)
    else:
        dec.step(q)            # the GPU's own selection feeds the GPU decode ...
        torch.cuda.synchronize()
        sel = dec.sparse.sel.cpu().numpy().reshape(BH, -1)
        n_sel = dec.sparse.n_sel.cpu().numpy().reshape(BH)
        # ... and the oracle attends to the same pages
        o_out, o_lse, _ = oracle.decode_softmax(kv, float(w.scale), sel, n_sel, heads=hs)
    torch.cuda.synchronize()
    out = dec.out.cpu().numpy().astype(np.float64).reshape(BH, -1)
    lse = dec.lse.cpu().numpy().astype(np.float64).reshape(BH)
    for bh in hs:
        if np.isinf(o_lse[bh]):
            assert np.isinf(lse[bh]) and np.all(out[bh] == 0)
            continue
        assert abs(lse[bh] - o_lse[bh]) <= LSE_TOL * max(1.0, abs(o_lse[bh])), (bh, lse[bh], o_lse[bh])
        err = np.abs(out[bh] - o_out[bh])
        ok = err <= 1e-4 + 2e-3 * np.abs(o_out[bh])
        assert ok.all(), (bh, err.max())
    assert E.entmaxkv_read_device_status() == E.EKV_OK


@pytest.mark.parametrize("name,over", [
    ("tiny", {}),
    ("gqa32k", {"batch": 2, "seq_lens": [8192, 5000]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345]}),
    ("long128k", {"batch": 2, "seq_lens": [3000, 2049], "num_q_heads": 8, "num_kv_heads": 1,
                  "page_size": 16, "budget_tokens": 512, "head_dim": 64}),
    ("long128k", {"batch": 2, "seq_lens": [3000, 2049], "num_q_heads": 8, "num_kv_heads": 8,
                  "dtype": "f32", "budget_tokens": 512}),
    ("gauss64k", {"batch": 2, "seq_lens": [16384, 9999]}),
])
@pytest.mark.parametrize("full", [False, True])
def test_softmax_decode(name, over, full):
    softmax_parity(make_workload(name, **over), full=full)


@pytest.mark.parametrize("full", [False, True])
def test_softmax_decode_full_size_sampled_heads(full):
    w = make_workload("long128k")
    softmax_parity(w, heads=sampled_heads(w, 48), full=full)
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# discarded mass of the kept pages: entmax delta and the softmax mass outside
# ---------------------------------------------------------------------------

def mass_parity(w, heads=None):
    from sparse_long_context_08_b300.mass import RECOVERED_TOL, measure
    m = measure(w)
    BH = w.batch * w.num_q_heads
    hs = list(range(BH)) if heads is None else list(heads)
    kv = oracle.KV(w)
    s = float(w.scale)
    f = oracle.decode_full(kv, s, w.alpha, m["sel"], m["n_sel"], heads=hs)
    _, _, outside = oracle.decode_softmax(kv, s, m["sel"], m["n_sel"], full=True, heads=hs)
    for bh in hs:
        assert abs(m["delta"][bh] - f.delta[bh]) <= 1e-4, (bh, m["delta"][bh], f.delta[bh])
        assert abs(m["softmax_outside"][bh] - outside[bh]) <= 5e-4, \
            (bh, m["softmax_outside"][bh], outside[bh])
        if f.covered[bh]:
            assert m["recovered"][bh], (bh, m["delta"][bh])
        elif f.delta[bh] > 10 * RECOVERED_TOL:
            assert not m["recovered"][bh], (bh, m["delta"][bh], f.delta[bh])
    return m


@pytest.mark.parametrize("name,over", [
    ("gqa32k", {"batch": 2, "seq_lens": [8192, 5000]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345], "alpha": 2.0}),
    ("long128k", {"batch": 1, "context": 8192, "alpha": 1.3, "seed": 7}),
    ("gauss64k", {"batch": 2, "seq_lens": [16384, 9999]}),
])
def test_discarded_mass(name, over):
    m = mass_parity(make_workload(name, **over))
    assert np.all(m["softmax_outside"] > 0)       # softmax keeps weight on every token


def test_discarded_mass_full_size_sampled_heads():
    w = make_workload("long128k")
    mass_parity(w, heads=sampled_heads(w, 32))
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# shapes: head_dim, dtype, group size, page size, general alpha
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (16, 4), (32, 4), (16, 8),
                                     (64, 8)])
def test_shapes(d, dtype, hq, hkv):
    w = make_workload("long128k", batch=2, seq_lens=[3000, 2049], head_dim=d, dtype=dtype,
                      num_q_heads=hq, num_kv_heads=hkv, page_size=16, budget_tokens=512,
                      planted_pages=4, seed=100 + d + hq * hkv)
    full_parity(w)


@pytest.mark.parametrize("alpha", [1.3, 2.5])
def test_general_alpha_bisection(alpha):
    full_parity(make_workload("long128k", batch=1, context=8192, alpha=alpha, seed=7))


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def test_budget_covers_every_page_and_single_page_sequences():
    w = make_workload("long128k", batch=3, seq_lens=[5 * 32, 20, 1], budget_tokens=4096,
                      planted_pages=0)
    rep = full_parity(w)
    g = DeviceRun(w)
    r = g.step()
    for bh in range(w.batch * w.num_q_heads):
        np_ = w.pages_of(bh // w.num_q_heads)
        assert list(r["sel"][bh, :r["n_sel"][bh]]) == list(range(np_))
        assert r["aux"][bh, 1] == -np.inf


def test_zero_length_sequence_in_a_batch():
    """A sequence with no tokens: no pages scored or selected, out = 0, tau =
    +inf, support 0, on every path; the other sequences match the oracle."""
    w = make_workload("long128k", batch=3, seq_lens=[5000, 0, 3000], planted_pages=2)
    rep = full_parity(w, heads=[h for h in range(3 * w.num_q_heads) if h // w.num_q_heads != 1])
    g = DeviceRun(w)
    r = g.step()
    Hq = w.num_q_heads
    assert np.all(r["n_sel"][Hq:2 * Hq] == 0)
    assert np.all(r["out"][Hq:2 * Hq] == 0) and np.all(np.isinf(r["tau"][Hq:2 * Hq]))
    assert np.all(r["support"][Hq:2 * Hq] == 0)
    from sparse_long_context_08_b300.api import EntmaxKVFullDecoder, EntmaxKVSoftmaxDecoder
    full = EntmaxKVFullDecoder(g.kv, Hq, float(w.scale), w.alpha)
    full.decode(g.q)
    sm = EntmaxKVSoftmaxDecoder(g.kv, Hq, float(w.scale), w.policy, w.budget_tokens, full=True)
    sm.decode(g.q)
    torch.cuda.synchronize()
    assert torch.all(full.out[1] == 0) and torch.all(torch.isinf(full.tau[1]))
    assert torch.all(sm.out[1] == 0) and torch.all(torch.isinf(sm.lse[1]))
    assert E.entmaxkv_read_device_status() == E.EKV_OK


def test_empty_selection_gives_zero_output():
    w = make_workload("long128k", batch=1, context=2048)
    g = DeviceRun(w)
    g.step()
    BH = w.num_q_heads
    sel = np.zeros((BH, w.cap_pages), np.int32)
    n = np.zeros(BH, np.int32)
    n[::2] = 3
    sel[:, :3] = [0, 5, 9]
    out, tau, sup = g.decode_with(sel, n)
    kv = oracle.KV(w)
    o_out, o_tau, o_sup, _ = oracle.decode_sparse(kv, float(w.scale), w.alpha, sel, n)
    compare_decode(out, tau, o_out, o_tau, range(BH))
    assert np.all(out[1::2] == 0) and np.all(np.isinf(tau[1::2])) and np.all(sup[1::2] == 0)


def test_tie_storm_constant_keys():
    """All keys equal: every bound ties (lowest pages win) and every kept token
    gets the same weight, so out is the mean of the kept values."""
    w = make_workload("long128k", batch=1, context=32 * 40, planted_pages=0, budget_tokens=32 * 7)
    w.k_pool[:] = w.k_pool[0, 0, 0]
    g = DeviceRun(w)
    r = g.step()
    kv = oracle.KV(w)
    for bh in range(w.num_q_heads):
        assert list(r["sel"][bh, :r["n_sel"][bh]]) == list(range(7))
    o_out, o_tau, o_sup, _ = oracle.decode_sparse(kv, float(w.scale), w.alpha, r["sel"], r["n_sel"])
    compare_decode(r["out"], r["tau"], o_out, o_tau, range(w.num_q_heads))
    assert np.all(r["support"] == 7 * 32)


def test_sparsemax_single_token_support():
    """alpha = 2 with one dominant key per head: the support is that token and
    out equals its value row."""
    w = make_workload("long128k", batch=1, context=4096, alpha=2.0, planted_pages=0,
                      num_q_heads=8, num_kv_heads=8, head_dim=64, dtype="f32", seed=9)
    # plant one key per head: 20 q/|q| at page 3, token 5
    blk = w.page_table[0, 3]
    for h in range(8):
        qn = w.q[0, h] / np.linalg.norm(w.q[0, h])
        w.k_pool[blk, h, 5] = 40.0 * qn
    g = DeviceRun(w)
    r = g.step()
    assert np.all(r["support"] == 1)
    for h in range(8):
        np.testing.assert_allclose(r["out"][h], w.v_pool[blk, h, 5], rtol=1e-6, atol=1e-6)
    full_parity(w)


def test_bad_page_table_entry_is_flagged_not_faulted():
    w = make_workload("long128k", batch=1, context=2048, planted_pages=0)
    w.page_table[0, 10] = w.num_blocks + 5     # out of range
    g = DeviceRun(w)
    g.step()
    assert E.entmaxkv_read_device_status() == E.EKV_DEVICE_CHECK_FAILED
    assert E.entmaxkv_read_device_status() == E.EKV_OK     # read clears it


@pytest.mark.parametrize("name,over", [
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345]}),
    ("long128k", {"batch": 2, "seq_lens": [16384, 12345], "policy": "topk_shared"}),
    ("long128k", {"batch": 3, "seq_lens": [3000, 0, 77], "num_q_heads": 16, "num_kv_heads": 2,
                  "planted_pages": 2}),
    ("long128k", {"batch": 2, "seq_lens": [3000, 2049], "num_q_heads": 8, "num_kv_heads": 8,
                  "dtype": "f32", "budget_tokens": 512, "planted_pages": 2}),
    ("gauss64k", {"batch": 2, "seq_lens": [16384, 9999]}),
    ("ctx1m", {"context": 262144}),
])
def test_select_decode_matches_the_separate_calls(name, over):
    """entmaxkv_select_decode (the selection builds the decode's page union:
    per-head clusters, shared selections, groups of 1 to 8, empty sequences;
    Gaussian selection and long contexts keep the decode's own plan) returns,
    bit for bit, what entmaxkv_select followed by entmaxkv_decode returns."""
    w = make_workload(name, **over)
    g = DeviceRun(w)
    d = g.dec
    d.score(g.q)
    d.select()
    d.decode(g.q)
    torch.cuda.synchronize()
    names = ("n_sel", "aux", "out", "tau", "support")
    ref = {k: getattr(d, k).clone() for k in names + ("sel",)}
    for k in names + ("sel",):
        getattr(d, k).fill_(-7)
    d.select_decode(g.q)
    torch.cuda.synchronize()
    for k in names:
        assert torch.equal(getattr(d, k), ref[k]), k
    n = ref["n_sel"].cpu().numpy().reshape(-1)
    a = d.sel.cpu().numpy().reshape(n.size, -1)
    b = ref["sel"].cpu().numpy().reshape(n.size, -1)
    for i in range(n.size):
        assert np.array_equal(a[i, :n[i]], b[i, :n[i]]), i
    assert E.entmaxkv_read_device_status() == E.EKV_OK


def test_bounded_wait_timeout_is_reported_and_the_context_survives():
    """The give-up path of the kernels' bounded waits: a wait on an mbarrier
    that never completes runs out (1 ms limit), the kernel records a timeout
    and returns; the status reads EKV_DEVICE_TIMEOUT once (the read clears it)
    and a decode step afterwards still matches the oracle."""
    import time
    assert E.entmaxkv_read_device_status() == E.EKV_OK
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    E.entmaxkv_check_wait_timeout(1000)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 >= 1e-3
    assert E.entmaxkv_read_device_status() == E.EKV_DEVICE_TIMEOUT
    assert E.entmaxkv_read_device_status() == E.EKV_OK
    full_parity(make_workload("long128k", batch=1, context=4096))


def test_deterministic_across_runs():
    w = make_workload("long128k", batch=2, context=8192)
    g = DeviceRun(w)
    a = g.step()
    b = g.step()
    for k in ("page_scores", "sel", "n_sel", "out", "tau", "support"):
        assert np.array_equal(a[k], b[k]), k


def test_step_host_graph_matches_the_device_step():
    """step_host replays its step (H2D of q, kernels, D2H of out) as one CUDA
    graph; every call returns what the device step returns, bit for bit, and
    follows new host inputs."""
    w = make_workload("long128k", batch=2, context=8192)
    g = DeviceRun(w)
    q_host = g.q.cpu().pin_memory()
    out_host = torch.empty(g.dec.out.shape, dtype=torch.float32).pin_memory()
    q_dev = torch.empty_like(g.q)
    for it in range(3):
        if it == 2:
            q_host.copy_(q_host * 0.5)            # new input through the same buffers
        g.dec.step_host(q_host, out_host, q_dev)
        torch.cuda.synchronize()
        got = out_host.clone()
        g.dec.step(q_host.cuda())
        torch.cuda.synchronize()
        assert torch.equal(got, g.dec.out.cpu()), it


def test_graph_capture_replays_the_step():
    w = make_workload("long128k", batch=2, context=8192)
    g = DeviceRun(w)
    ref = g.step()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g.dec.step(g.q)          # warm-up on the capture stream
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.dec.step(g.q)
    g.dec.out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    out = g.dec.out.cpu().numpy().astype(np.float64).reshape(ref["out"].shape)
    assert np.array_equal(out, ref["out"])



def test_copy_in_from_pinned_host_memory():
    """The input-staging kernel copies pinned host memory (16-byte path and
    byte path, misaligned views included) exactly; pageable host memory is
    rejected on the host, before any launch."""
    gen = torch.Generator().manual_seed(5)
    for n in (1, 15, 16, 1000, 4099, 1 << 17):
        src = torch.randint(0, 256, (n + 1,), dtype=torch.uint8, generator=gen).pin_memory()
        for view in (src[:n], src[1:]):
            dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
            E.entmaxkv_copy_in(dst, view)
            torch.cuda.synchronize()
            assert torch.equal(dst.cpu(), view), n
    pageable = torch.zeros(64, dtype=torch.uint8)
    with pytest.raises(E.EntmaxKVError):
        E.entmaxkv_copy_in(torch.zeros(64, dtype=torch.uint8, device="cuda"), pageable)


def test_select_decode_writes_pinned_host_output():
    """out in pinned host memory is written by the decode kernel directly and
    equals the device-memory result bit for bit."""
    w = make_workload("long128k", batch=2, context=8192)
    g = DeviceRun(w)
    g.dec.score(g.q)
    g.dec.select_decode(g.q)
    torch.cuda.synchronize()
    ref = g.dec.out.cpu().clone()
    host = torch.full(g.dec.out.shape, float("nan"), dtype=torch.float32).pin_memory()
    g.dec.select_decode(g.q, out=host)
    torch.cuda.synchronize()
    assert torch.equal(host, ref)
