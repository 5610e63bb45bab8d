"""entmaxkv_decode_noalloc against entmaxkv_decode.

The no-allocation decode exists for callers that cannot allocate device memory
at the moment they decode (an allocator callback, a plugin given only its input
and output buffers, a server whose memory is fixed up front); it uses a scratch
array built into the library instead of a caller workspace.  This file is named
to be collected last so that a run stopping at the first failure has already run
every other test.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

from sparse_long_context_08_b300 import entmaxkv as E
from sparse_long_context_08_b300.api import EntmaxKVDecoder, upload_workload
from sparse_long_context_08_b300.workloads import make_workload

from gpu_util import compare_decode

pytestmark = pytest.mark.gpu


def _noalloc(lib):
    f = lib.entmaxkv_decode_noalloc
    vp, i32, f32 = C.c_void_p, C.c_int32, C.c_float
    f.argtypes = [vp, i32, f32, vp, vp, vp, i32, f32, vp, vp, vp, vp]
    f.restype = C.c_int
    return f


def _call(f, dec, q, out, tau, sup):
    st = f(C.c_void_p(q.data_ptr()), dec.Hq, dec.scale, dec.kv.ref,
           C.c_void_p(dec.sel.data_ptr()), C.c_void_p(dec.n_sel.data_ptr()), dec.cap, dec.alpha,
           C.c_void_p(out.data_ptr()), C.c_void_p(tau.data_ptr()), C.c_void_p(sup.data_ptr()),
           C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == E.EKV_OK, E.entmaxkv_status_string(st)


def _np(t):
    return t.cpu().numpy().astype(np.float64).reshape(-1, *t.shape[2:]) if t.dim() > 2 \
        else t.cpu().numpy().astype(np.float64).reshape(-1)


def test_noalloc_decode_matches_workspace_decode_on_two_calls():
    assert torch.cuda.is_available(), "GPU test"
    from sparse_long_context_08_b300 import build
    build.build()
    f = _noalloc(E.lib())
    w = make_workload("long128k", batch=2, seq_lens=[8192, 5000])
    kv, q = upload_workload(w)
    dec = EntmaxKVDecoder(kv, w.num_q_heads, float(w.scale), w.alpha, w.policy, w.budget_tokens)
    dec.build_meta()
    out = torch.empty_like(dec.out)
    tau = torch.empty_like(dec.tau)
    sup = torch.empty_like(dec.support)
    heads = range(w.batch * w.num_q_heads)
    # two calls in a row with different queries (and so different selections):
    # the second must not see anything the first left in the shared scratch
    for qq in (q, torch.flip(q, dims=[1]).contiguous() * 1.3):
        dec.step(qq)                       # workspace path (entmaxkv_decode)
        torch.cuda.synchronize()
        ref_out, ref_tau, ref_sup = _np(dec.out), _np(dec.tau), dec.support.cpu().numpy().reshape(-1)
        out.fill_(float("nan"))
        tau.fill_(float("nan"))
        _call(f, dec, qq, out, tau, sup)
        torch.cuda.synchronize()
        compare_decode(_np(out), _np(tau), ref_out, ref_tau, heads,
                       sup.cpu().numpy().reshape(-1), ref_sup)
    assert E.entmaxkv_read_device_status() == E.EKV_OK


def test_noalloc_rejects_sizes_beyond_its_scratch():
    assert torch.cuda.is_available(), "GPU test"
    f = _noalloc(E.lib())
    big = E._PagedKV(16, 16, 1, 65536 * 64, 8, 16, 128, 16, 4096, 16, 64)
    # batch 64 x 64 heads with a 1024-page cap needs far more than the built-in
    # scratch; the call must refuse before touching any (here dummy) pointer
    need = E.entmaxkv_workspace_size(64, 64, 8, 128, 16, 4096, 1024)
    assert need > 16 * 1024 * 1024
    st = f(C.c_void_p(16), 64, 1.0, C.byref(big), C.c_void_p(16), C.c_void_p(16), 1024, 1.5,
           C.c_void_p(16), None, None, None)
    assert st == E.EKV_WORKSPACE_TOO_SMALL
