"""Python access to the fp64 CPU oracle of the EntmaxKV decode pipeline.

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  The arithmetic lives in
oracle.c (plain C, fp64); this module only marshals numpy arrays.

Method source: the web page "Riepilogo Tecnico: EntmaxKV - Decodifica
Consapevole del Supporto per l'Attention Entmax", §2.A-§2.C and §3; the
alpha-entmax mapping of Peters, Niculae and Martins (ACL 2019).
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None


class _KV(C.Structure):
    _fields_ = [("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("dtype", C.c_int),
                ("num_blocks", C.c_int), ("num_kv_heads", C.c_int),
                ("page_size", C.c_int), ("head_dim", C.c_int),
                ("page_table", C.c_void_p), ("max_pages", C.c_int),
                ("seq_lens", C.c_void_p), ("batch", C.c_int)]


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        _lib = C.CDLL(path)
        dp = C.POINTER(C.c_double)
        _lib.oracle_gauss_F.restype = C.c_double
        _lib.oracle_widen.restype = C.c_double
        _lib.oracle_entmax_tau.argtypes = [dp, C.c_int, C.c_double, dp]
        _lib.oracle_entmax_probs.argtypes = [dp, C.c_int, C.c_double, dp]
        _lib.oracle_gauss_F.argtypes = [dp, dp, C.c_void_p, C.c_int, C.c_double, C.c_double]
    return _lib


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(lib().oracle_get_threads())


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


class KV:
    """Holds the ctypes view of a paged cache (the arrays must stay alive)."""

    def __init__(self, w):
        self.w = w
        self.k = np.ascontiguousarray(w.k_pool)
        self.v = np.ascontiguousarray(w.v_pool)
        self.pt = np.ascontiguousarray(w.page_table, dtype=np.int32)
        self.sl = np.ascontiguousarray(w.seq_lens, dtype=np.int32)
        self.q = np.ascontiguousarray(w.q, dtype=np.float32)
        nb, hkv, P, d = self.k.shape
        self.s = _KV(_ptr(self.k), _ptr(self.v), 1 if w.dtype == "bf16" else 0,
                     nb, hkv, P, d, _ptr(self.pt), self.pt.shape[1], _ptr(self.sl),
                     self.sl.shape[0])
        self.Hq = w.num_q_heads
        self.meta_shape = (nb, hkv, d)
        self.BH = self.sl.shape[0] * w.num_q_heads

    @property
    def ref(self):
        return C.byref(self.s)


def _heads(heads):
    if heads is None:
        return None, 0
    h = np.ascontiguousarray(heads, dtype=np.int32)
    return h, len(h)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


@dataclass
class Meta:
    kmin: np.ndarray
    kmax: np.ndarray
    mean: np.ndarray
    var: np.ndarray


def build_meta(kv: KV) -> Meta:
    shp = kv.meta_shape
    arrs = [np.full(shp, np.nan) for _ in range(4)]
    _check(lib().oracle_build_meta(kv.ref, *[_ptr(a) for a in arrs]), "build_meta")
    return Meta(*arrs)


def score_bbox(kv: KV, meta: Meta, scale: float, heads=None) -> np.ndarray:
    h, nh = _heads(heads)
    out = np.full((kv.BH, kv.pt.shape[1]), np.nan)
    _check(lib().oracle_score_bbox(kv.ref, _ptr(kv.q), C.c_int(kv.Hq), C.c_double(scale),
                                   _ptr(meta.kmin), _ptr(meta.kmax), _ptr(h), C.c_int(nh),
                                   _ptr(out)), "score_bbox")
    return out


def select_topk(kv: KV, bound: np.ndarray, kp: int, heads=None):
    h, nh = _heads(heads)
    bound = _f64(bound)
    sel = np.full((kv.BH, kp), -1, dtype=np.int32)
    n_sel = np.zeros(kv.BH, dtype=np.int32)
    kth = np.full(kv.BH, np.nan)
    nxt = np.full(kv.BH, np.nan)
    _check(lib().oracle_select_topk(kv.ref, C.c_int(kv.Hq), _ptr(bound), C.c_int(kp),
                                    _ptr(h), C.c_int(nh), _ptr(sel), _ptr(n_sel),
                                    _ptr(kth), _ptr(nxt)), "select_topk")
    return sel, n_sel, kth, nxt


def select_topk_shared(kv: KV, bound: np.ndarray, kp: int, heads=None):
    """Top-k shared by a kv head's query group (one page set per kv head): a
    page's score for the group is the largest of its G query heads' bounds
    ([EntmaxKV §2.A] bound, [EntmaxKV §2.B.1] top-k on that score), and every
    head of the group receives the group's top-kp pages, ties to the lower
    page.  `bound` must hold every head of the groups named in `heads`.
    Returns (sel, n_sel, kth, next, shared score) per head."""
    bound = _f64(bound)
    G = kv.Hq // kv.meta_shape[1]
    BH, M = bound.shape
    h = np.arange(BH) if heads is None else np.asarray(heads)
    groups = np.unique(h // G)
    shared = np.full_like(bound, np.nan)
    for grp in groups:
        shared[grp * G:(grp + 1) * G] = bound[grp * G:(grp + 1) * G].max(axis=0)
    sel, n_sel, kth, nxt = select_topk(kv, shared, kp, heads)
    return sel, n_sel, kth, nxt, shared


def score_gauss(kv: KV, meta: Meta, scale: float, heads=None):
    h, nh = _heads(heads)
    m = np.full((kv.BH, kv.pt.shape[1]), np.nan)
    s = np.full((kv.BH, kv.pt.shape[1]), np.nan)
    _check(lib().oracle_score_gauss(kv.ref, _ptr(kv.q), C.c_int(kv.Hq), C.c_double(scale),
                                    _ptr(meta.mean), _ptr(meta.var), _ptr(h), C.c_int(nh),
                                    _ptr(m), _ptr(s)), "score_gauss")
    return m, s


def gauss_F(m, s, n, alpha: float, tau: float) -> float:
    m = _f64(m)
    s = _f64(s)
    n = np.ascontiguousarray(n, dtype=np.int32)
    dp = C.POINTER(C.c_double)
    return float(lib().oracle_gauss_F(m.ctypes.data_as(dp), s.ctypes.data_as(dp),
                                      _ptr(n), len(m), alpha, tau))


def select_gauss(kv: KV, m, s, alpha: float, delta: float, cap: int, heads=None):
    h, nh = _heads(heads)
    m = _f64(m)
    s = _f64(s)
    sel = np.full((kv.BH, cap), -1, dtype=np.int32)
    n_sel = np.zeros(kv.BH, dtype=np.int32)
    tau_hat = np.full(kv.BH, np.nan)
    zmax = np.full((kv.BH, kv.pt.shape[1]), np.nan)
    _check(lib().oracle_select_gauss(kv.ref, C.c_int(kv.Hq), _ptr(m), _ptr(s),
                                     C.c_double(alpha), C.c_double(delta), C.c_int(cap),
                                     _ptr(h), C.c_int(nh), _ptr(sel), _ptr(n_sel),
                                     _ptr(tau_hat), _ptr(zmax)), "select_gauss")
    return sel, n_sel, tau_hat, zmax


def entmax_tau(zp, alpha: float):
    zp = _f64(zp)
    t = C.c_double()
    dp = C.POINTER(C.c_double)
    k = lib().oracle_entmax_tau(zp.ctypes.data_as(dp), len(zp), alpha, C.byref(t))
    return t.value, int(k)


def entmax_probs(zp, alpha: float) -> np.ndarray:
    zp = _f64(zp)
    p = np.empty_like(zp)
    dp = C.POINTER(C.c_double)
    lib().oracle_entmax_probs(zp.ctypes.data_as(dp), len(zp), alpha, p.ctypes.data_as(dp))
    return p


def entmax(z, alpha: float) -> np.ndarray:
    """alpha-entmax of raw scores z (the mapping works on z' = (alpha-1) z)."""
    return entmax_probs((alpha - 1.0) * _f64(z), alpha)


def decode_sparse(kv: KV, scale: float, alpha: float, sel, n_sel, heads=None):
    h, nh = _heads(heads)
    sel = np.ascontiguousarray(sel, dtype=np.int32)
    n_sel = np.ascontiguousarray(n_sel, dtype=np.int32)
    d = kv.meta_shape[2]
    out = np.full((kv.BH, d), np.nan)
    tau = np.full(kv.BH, np.nan)
    sup = np.full(kv.BH, -1, dtype=np.int32)
    psum = np.full(kv.BH, np.nan)
    _check(lib().oracle_decode_sparse(kv.ref, _ptr(kv.q), C.c_int(kv.Hq), C.c_double(scale),
                                      C.c_double(alpha), _ptr(sel), _ptr(n_sel),
                                      C.c_int(sel.shape[1]), _ptr(h), C.c_int(nh),
                                      _ptr(out), _ptr(tau), _ptr(sup), _ptr(psum)),
           "decode_sparse")
    return out, tau, sup, psum


def decode_softmax(kv: KV, scale: float, sel=None, n_sel=None, full: bool = False, heads=None):
    """Softmax attention over the selected pages (every page when full).
    Returns (out, lse, outside): outside = the full softmax's mass outside the
    kept pages when both full and sel are given (NaN otherwise)."""
    h, nh = _heads(heads)
    cap = 0
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        n_sel = np.ascontiguousarray(n_sel, dtype=np.int32)
        cap = sel.shape[1]
    d = kv.meta_shape[2]
    out = np.full((kv.BH, d), np.nan)
    lse = np.full(kv.BH, np.nan)
    outside = np.full(kv.BH, np.nan)
    _check(lib().oracle_decode_softmax(kv.ref, _ptr(kv.q), C.c_int(kv.Hq), C.c_double(scale),
                                       _ptr(sel), _ptr(n_sel), C.c_int(cap), C.c_int(int(full)),
                                       _ptr(h), C.c_int(nh), _ptr(out), _ptr(lse),
                                       _ptr(outside)), "decode_softmax")
    return out, lse, outside


@dataclass
class Full:
    out: np.ndarray
    tau: np.ndarray
    support: np.ndarray
    delta: np.ndarray
    vnorm: np.ndarray
    covered: np.ndarray
    support_pages: np.ndarray


def decode_full(kv: KV, scale: float, alpha: float, sel=None, n_sel=None, heads=None) -> Full:
    h, nh = _heads(heads)
    cap = 0
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32)
        n_sel = np.ascontiguousarray(n_sel, dtype=np.int32)
        cap = sel.shape[1]
    d = kv.meta_shape[2]
    f = Full(np.full((kv.BH, d), np.nan), np.full(kv.BH, np.nan),
             np.full(kv.BH, -1, dtype=np.int32), np.full(kv.BH, np.nan),
             np.full(kv.BH, np.nan), np.full(kv.BH, -1, dtype=np.int32),
             np.full(kv.BH, -1, dtype=np.int32))
    _check(lib().oracle_decode_full(kv.ref, _ptr(kv.q), C.c_int(kv.Hq), C.c_double(scale),
                                    C.c_double(alpha), _ptr(sel), _ptr(n_sel), C.c_int(cap),
                                    _ptr(h), C.c_int(nh), _ptr(f.out), _ptr(f.tau),
                                    _ptr(f.support), _ptr(f.delta), _ptr(f.vnorm),
                                    _ptr(f.covered), _ptr(f.support_pages)), "decode_full")
    return f


def sparse_step(kv: KV, w, heads=None, meta: Meta | None = None):
    """One decode step of the pipeline for the workload's policy: score, select,
    then sparse attention.  Returns a dict of every intermediate."""
    meta = meta if meta is not None else build_meta(kv)
    scale = float(w.scale)
    res = {"meta": meta}
    if w.policy == "topk":
        bound = score_bbox(kv, meta, scale, heads)
        sel, n_sel, kth, nxt = select_topk(kv, bound, w.cap_pages, heads)
        res.update(bound=bound, kth=kth, next=nxt)
    elif w.policy == "topk_shared":
        G = w.group
        hh = None if heads is None else np.unique(
            (np.asarray(heads)[:, None] // G * G + np.arange(G)[None, :]).ravel()).astype(np.int32)
        bound = score_bbox(kv, meta, scale, hh)
        sel, n_sel, kth, nxt, shared = select_topk_shared(kv, bound, w.cap_pages, heads)
        res.update(bound=bound, kth=kth, next=nxt, shared=shared)
    else:
        m, s = score_gauss(kv, meta, scale, heads)
        sel, n_sel, tau_hat, zmax = select_gauss(kv, m, s, w.alpha, w.delta, w.cap_pages, heads)
        res.update(m=m, s=s, tau_hat=tau_hat, zmax=zmax)
    out, tau, sup, psum = decode_sparse(kv, scale, w.alpha, sel, n_sel, heads)
    res.update(sel=sel, n_sel=n_sel, out=out, tau=tau, support=sup, psum=psum)
    return res
