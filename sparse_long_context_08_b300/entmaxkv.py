"""Thin Python binding of the EntmaxKV C ABI (include/entmaxkv.h).

Argument marshalling only: torch tensors on the GPU are checked for dtype,
shape, device and contiguity and passed as raw device pointers together with
the current CUDA stream.  Every computation runs in libentmaxkv.so; if the
library is missing this module raises instead of computing anything itself.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libentmaxkv.so")

EKV_OK = 0
EKV_INVALID_ARG = 1
EKV_UNSUPPORTED = 2
EKV_WORKSPACE_TOO_SMALL = 3
EKV_CUDA_ERROR = 4
EKV_DEVICE_CHECK_FAILED = 5
EKV_DEVICE_TIMEOUT = 6
EKV_F32 = 0
EKV_BF16 = 1
EKV_SELECT_TOPK = 0
EKV_SELECT_GAUSS = 1
EKV_SELECT_TOPK_SHARED = 2

SYMBOLS = ("entmaxkv_build_page_meta", "entmaxkv_score_pages", "entmaxkv_select",
           "entmaxkv_decode", "entmaxkv_workspace_size", "entmaxkv_status_string",
           "entmaxkv_read_device_status", "entmaxkv_version", "entmaxkv_set_stage_events",
           "entmaxkv_decode_counts", "entmaxkv_decode_noalloc", "entmaxkv_decode_full",
           "entmaxkv_full_workspace_size", "entmaxkv_decode_softmax",
           "entmaxkv_decode_softmax_full", "entmaxkv_softmax_workspace_size",
           "entmaxkv_kept_mass", "entmaxkv_check_wait_timeout", "entmaxkv_select_decode",
           "entmaxkv_copy_in")


class EntmaxKVError(RuntimeError):
    def __init__(self, call: str, status: int):
        super().__init__(f"{call} failed: {entmaxkv_status_string(status)} (status {status})")
        self.status = status


class _PagedKV(C.Structure):
    _fields_ = [("k_pool", C.c_void_p), ("v_pool", C.c_void_p), ("dtype", C.c_int32),
                ("num_blocks", C.c_int32), ("num_kv_heads", C.c_int32),
                ("page_size", C.c_int32), ("head_dim", C.c_int32),
                ("page_table", C.c_void_p), ("max_pages", C.c_int32),
                ("seq_lens", C.c_void_p), ("batch", C.c_int32)]


class _PageMeta(C.Structure):
    _fields_ = [("kmin", C.c_void_p), ("kmax", C.c_void_p), ("mean", C.c_void_p),
                ("var", C.c_void_p)]


_lib = None


def lib() -> C.CDLL:
    """Load libentmaxkv.so (built in-tree by sparse_long_context_08_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m sparse_long_context_08_b300.build`")
        L = C.CDLL(LIB_PATH)
        vp, i32, f32, sz = C.c_void_p, C.c_int32, C.c_float, C.c_size_t
        L.entmaxkv_build_page_meta.argtypes = [vp, i32, i32, vp, i32, i32, vp]
        L.entmaxkv_score_pages.argtypes = [vp, i32, f32, vp, vp, i32, vp, vp]
        L.entmaxkv_select.argtypes = [vp, vp, i32, i32, i32, f32, f32, vp, vp, vp, vp, sz, vp]
        L.entmaxkv_decode.argtypes = [vp, i32, f32, vp, vp, vp, i32, f32, vp, vp, vp, vp, sz, vp]
        L.entmaxkv_workspace_size.argtypes = [i32] * 7
        L.entmaxkv_workspace_size.restype = sz
        L.entmaxkv_status_string.argtypes = [i32]
        L.entmaxkv_status_string.restype = C.c_char_p
        L.entmaxkv_read_device_status.argtypes = [vp, vp]
        L.entmaxkv_version.restype = i32
        L.entmaxkv_set_stage_events.argtypes = [vp, i32]
        L.entmaxkv_decode_counts.argtypes = [vp] + [i32] * 7 + [vp, vp, vp]
        L.entmaxkv_decode_full.argtypes = [vp, i32, f32, vp, f32, vp, vp, vp, vp, sz, vp]
        L.entmaxkv_full_workspace_size.argtypes = [i32] * 6
        L.entmaxkv_full_workspace_size.restype = sz
        L.entmaxkv_decode_softmax.argtypes = [vp, i32, f32, vp, vp, vp, i32, vp, vp, vp, sz, vp]
        L.entmaxkv_decode_softmax_full.argtypes = [vp, i32, f32, vp, vp, vp, vp, sz, vp]
        L.entmaxkv_kept_mass.argtypes = [vp] + [i32] * 7 + [f32, vp, vp, vp]
        L.entmaxkv_softmax_workspace_size.argtypes = [i32] * 7
        L.entmaxkv_softmax_workspace_size.restype = sz
        L.entmaxkv_check_wait_timeout.argtypes = [C.c_uint32, vp]
        L.entmaxkv_select_decode.argtypes = [vp, vp, i32, f32, vp, i32, i32, f32, f32, vp, vp,
                                             vp, vp, vp, vp, vp, sz, vp]
        L.entmaxkv_copy_in.argtypes = [vp, vp, sz, vp]
        for name in ("entmaxkv_build_page_meta", "entmaxkv_score_pages", "entmaxkv_select",
                     "entmaxkv_decode", "entmaxkv_read_device_status",
                     "entmaxkv_set_stage_events", "entmaxkv_decode_counts", "entmaxkv_decode_noalloc",
                     "entmaxkv_decode_full", "entmaxkv_decode_softmax",
                     "entmaxkv_decode_softmax_full", "entmaxkv_kept_mass",
                     "entmaxkv_check_wait_timeout", "entmaxkv_select_decode", "entmaxkv_copy_in"):
            getattr(L, name).restype = C.c_int
        _lib = L
    return _lib


# ---------------------------------------------------------------------------
# tensor checks
# ---------------------------------------------------------------------------

def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _need(t: torch.Tensor, name: str, dtype: torch.dtype | tuple, shape: tuple | None = None,
          pinned_ok: bool = False):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    dts = dtype if isinstance(dtype, tuple) else (dtype,)
    if t.dtype not in dts:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dts}")
    if not t.is_cuda and not (pinned_ok and t.is_pinned()):
        raise ValueError(f"{name} must be on a CUDA device" + (" or in pinned host memory"
                                                               if pinned_ok else ""))
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(int(stream))


def _check(call: str, status: int) -> None:
    if status != EKV_OK:
        raise EntmaxKVError(call, status)


@dataclass
class PagedKV:
    """A paged cache on the GPU: k_pool/v_pool [num_blocks, Hkv, P, d] (float32 or
    bfloat16), page_table int32 [B, max_pages], seq_lens int32 [B]."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor

    def __post_init__(self):
        _need(self.k_pool, "k_pool", (torch.float32, torch.bfloat16))
        _need(self.v_pool, "v_pool", self.k_pool.dtype, tuple(self.k_pool.shape))
        if self.k_pool.dim() != 4:
            raise ValueError("k_pool must be [num_blocks, num_kv_heads, page_size, head_dim]")
        _need(self.page_table, "page_table", torch.int32)
        _need(self.seq_lens, "seq_lens", torch.int32, (self.page_table.shape[0],))
        nb, hkv, P, d = self.k_pool.shape
        self._s = _PagedKV(self.k_pool.data_ptr(), self.v_pool.data_ptr(),
                           EKV_BF16 if self.k_pool.dtype == torch.bfloat16 else EKV_F32,
                           nb, hkv, P, d, self.page_table.data_ptr(), self.page_table.shape[1],
                           self.seq_lens.data_ptr(), self.page_table.shape[0])

    @property
    def ref(self):
        return C.byref(self._s)

    @property
    def batch(self) -> int:
        return self.page_table.shape[0]

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pool.shape[1]

    @property
    def page_size(self) -> int:
        return self.k_pool.shape[2]

    @property
    def head_dim(self) -> int:
        return self.k_pool.shape[3]

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]


@dataclass
class PageMeta:
    """Per-page key metadata, each [num_blocks, Hkv, d]: kmin/kmax in the K dtype,
    mean/var float32; unused entries may be None."""
    kmin: torch.Tensor | None = None
    kmax: torch.Tensor | None = None
    mean: torch.Tensor | None = None
    var: torch.Tensor | None = None

    @staticmethod
    def empty_like(kv: PagedKV, bbox: bool = True, gauss: bool = False) -> "PageMeta":
        shp = (kv.num_blocks, kv.num_kv_heads, kv.head_dim)
        dev = kv.k_pool.device
        m = PageMeta()
        if bbox:
            m.kmin = torch.empty(shp, dtype=kv.k_pool.dtype, device=dev)
            m.kmax = torch.empty(shp, dtype=kv.k_pool.dtype, device=dev)
        if gauss:
            m.mean = torch.empty(shp, dtype=torch.float32, device=dev)
            m.var = torch.empty(shp, dtype=torch.float32, device=dev)
        return m

    def _struct(self, kv: PagedKV) -> _PageMeta:
        shp = (kv.num_blocks, kv.num_kv_heads, kv.head_dim)
        for name in ("kmin", "kmax"):
            t = getattr(self, name)
            if t is not None:
                _need(t, name, kv.k_pool.dtype, shp)
        for name in ("mean", "var"):
            t = getattr(self, name)
            if t is not None:
                _need(t, name, torch.float32, shp)
        return _PageMeta(*(None if t is None else t.data_ptr()
                           for t in (self.kmin, self.kmax, self.mean, self.var)))


# ---------------------------------------------------------------------------
# the C ABI, same names
# ---------------------------------------------------------------------------

def entmaxkv_status_string(status: int) -> str:
    return lib().entmaxkv_status_string(int(status)).decode()


def entmaxkv_version() -> int:
    return int(lib().entmaxkv_version())


def entmaxkv_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, page_size, max_pages,
                            cap_pages) -> int:
    return int(lib().entmaxkv_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                             page_size, max_pages, cap_pages))


def entmaxkv_build_page_meta(kv: PagedKV, first_page: int, num_pages: int, meta: PageMeta,
                             want_bbox: bool = True, want_gauss: bool = False, stream=None) -> None:
    m = meta._struct(kv)
    _check("entmaxkv_build_page_meta",
           lib().entmaxkv_build_page_meta(kv.ref, first_page, num_pages, C.byref(m),
                                          int(want_bbox), int(want_gauss), _stream(stream)))


def entmaxkv_score_pages(q: torch.Tensor, num_q_heads: int, scale: float, kv: PagedKV,
                         meta: PageMeta, policy: int, page_scores: torch.Tensor,
                         stream=None) -> None:
    _need(q, "q", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    nout = 2 if policy == EKV_SELECT_GAUSS else 1
    shape = (kv.batch, num_q_heads, kv.max_pages) + ((2,) if nout == 2 else ())
    _need(page_scores, "page_scores", torch.float32, shape)
    m = meta._struct(kv)
    _check("entmaxkv_score_pages",
           lib().entmaxkv_score_pages(_ptr(q), num_q_heads, float(scale), kv.ref, C.byref(m),
                                      policy, _ptr(page_scores), _stream(stream)))


def entmaxkv_select(page_scores: torch.Tensor, kv: PagedKV, num_q_heads: int, policy: int,
                    budget_tokens: int, alpha: float, delta: float, sel: torch.Tensor,
                    n_sel: torch.Tensor, aux: torch.Tensor | None = None, stream=None) -> None:
    cap = budget_tokens // kv.page_size
    _need(page_scores, "page_scores", torch.float32)
    _need(sel, "sel", torch.int32, (kv.batch, num_q_heads, cap))
    _need(n_sel, "n_sel", torch.int32, (kv.batch, num_q_heads))
    if aux is not None:
        _need(aux, "aux", torch.float32, (kv.batch, num_q_heads, 2))
    _check("entmaxkv_select",
           lib().entmaxkv_select(_ptr(page_scores), kv.ref, num_q_heads, policy, budget_tokens,
                                 float(alpha), float(delta), _ptr(sel), _ptr(n_sel), _ptr(aux),
                                 None, 0, _stream(stream)))


def entmaxkv_decode(q: torch.Tensor, num_q_heads: int, scale: float, kv: PagedKV,
                    sel: torch.Tensor, n_sel: torch.Tensor, cap_pages: int, alpha: float,
                    out: torch.Tensor, tau_out: torch.Tensor | None, support_out: torch.Tensor | None,
                    workspace: torch.Tensor, stream=None) -> None:
    _need(q, "q", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    _need(sel, "sel", torch.int32, (kv.batch, num_q_heads, cap_pages))
    _need(n_sel, "n_sel", torch.int32, (kv.batch, num_q_heads))
    _need(out, "out", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    if tau_out is not None:
        _need(tau_out, "tau_out", torch.float32, (kv.batch, num_q_heads))
    if support_out is not None:
        _need(support_out, "support_out", torch.int32, (kv.batch, num_q_heads))
    _need(workspace, "workspace", torch.uint8)
    _check("entmaxkv_decode",
           lib().entmaxkv_decode(_ptr(q), num_q_heads, float(scale), kv.ref, _ptr(sel),
                                 _ptr(n_sel), cap_pages, float(alpha), _ptr(out), _ptr(tau_out),
                                 _ptr(support_out), _ptr(workspace), workspace.numel(),
                                 _stream(stream)))


def entmaxkv_select_decode(page_scores: torch.Tensor, q: torch.Tensor, num_q_heads: int,
                           scale: float, kv: PagedKV, policy: int, budget_tokens: int,
                           alpha: float, delta: float, sel: torch.Tensor, n_sel: torch.Tensor,
                           aux: torch.Tensor | None, out: torch.Tensor,
                           tau_out: torch.Tensor | None, support_out: torch.Tensor | None,
                           workspace: torch.Tensor, stream=None) -> None:
    """entmaxkv_select then entmaxkv_decode in one call (the selection also
    builds the decode's page union for the top-k policies)."""
    cap = budget_tokens // kv.page_size
    _need(page_scores, "page_scores", torch.float32)
    _need(q, "q", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    _need(sel, "sel", torch.int32, (kv.batch, num_q_heads, cap))
    _need(n_sel, "n_sel", torch.int32, (kv.batch, num_q_heads))
    if aux is not None:
        _need(aux, "aux", torch.float32, (kv.batch, num_q_heads, 2))
    _need(out, "out", torch.float32, (kv.batch, num_q_heads, kv.head_dim), pinned_ok=True)
    if tau_out is not None:
        _need(tau_out, "tau_out", torch.float32, (kv.batch, num_q_heads))
    if support_out is not None:
        _need(support_out, "support_out", torch.int32, (kv.batch, num_q_heads))
    _need(workspace, "workspace", torch.uint8)
    _check("entmaxkv_select_decode",
           lib().entmaxkv_select_decode(_ptr(page_scores), _ptr(q), num_q_heads, float(scale),
                                        kv.ref, policy, budget_tokens, float(alpha),
                                        float(delta), _ptr(sel), _ptr(n_sel), _ptr(aux),
                                        _ptr(out), _ptr(tau_out), _ptr(support_out),
                                        _ptr(workspace), workspace.numel(), _stream(stream)))


def entmaxkv_full_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, page_size,
                                 max_pages) -> int:
    return int(lib().entmaxkv_full_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                  page_size, max_pages))


def entmaxkv_decode_full(q: torch.Tensor, num_q_heads: int, scale: float, kv: PagedKV,
                         alpha: float, out: torch.Tensor, tau_out: torch.Tensor | None,
                         support_out: torch.Tensor | None, workspace: torch.Tensor,
                         stream=None) -> None:
    """Full-cache alpha-entmax decode: every valid token of every sequence."""
    _need(q, "q", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    _need(out, "out", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    if tau_out is not None:
        _need(tau_out, "tau_out", torch.float32, (kv.batch, num_q_heads))
    if support_out is not None:
        _need(support_out, "support_out", torch.int32, (kv.batch, num_q_heads))
    _need(workspace, "workspace", torch.uint8)
    _check("entmaxkv_decode_full",
           lib().entmaxkv_decode_full(_ptr(q), num_q_heads, float(scale), kv.ref, float(alpha),
                                      _ptr(out), _ptr(tau_out), _ptr(support_out),
                                      _ptr(workspace), workspace.numel(), _stream(stream)))


def entmaxkv_softmax_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, page_size,
                                    max_pages, cap_pages) -> int:
    return int(lib().entmaxkv_softmax_workspace_size(batch, num_q_heads, num_kv_heads, head_dim,
                                                     page_size, max_pages, cap_pages))


def entmaxkv_decode_softmax(q: torch.Tensor, num_q_heads: int, scale: float, kv: PagedKV,
                            sel: torch.Tensor | None, n_sel: torch.Tensor | None, cap_pages: int,
                            out: torch.Tensor, lse_out: torch.Tensor | None,
                            workspace: torch.Tensor, stream=None) -> None:
    """Softmax attention over the selected pages (sel None: every page)."""
    _need(q, "q", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    _need(out, "out", torch.float32, (kv.batch, num_q_heads, kv.head_dim))
    if lse_out is not None:
        _need(lse_out, "lse_out", torch.float32, (kv.batch, num_q_heads))
    _need(workspace, "workspace", torch.uint8)
    if sel is None:
        _check("entmaxkv_decode_softmax_full",
               lib().entmaxkv_decode_softmax_full(_ptr(q), num_q_heads, float(scale), kv.ref,
                                                  _ptr(out), _ptr(lse_out), _ptr(workspace),
                                                  workspace.numel(), _stream(stream)))
        return
    _need(sel, "sel", torch.int32, (kv.batch, num_q_heads, cap_pages))
    _need(n_sel, "n_sel", torch.int32, (kv.batch, num_q_heads))
    _check("entmaxkv_decode_softmax",
           lib().entmaxkv_decode_softmax(_ptr(q), num_q_heads, float(scale), kv.ref, _ptr(sel),
                                         _ptr(n_sel), cap_pages, _ptr(out), _ptr(lse_out),
                                         _ptr(workspace), workspace.numel(), _stream(stream)))


def entmaxkv_kept_mass(workspace: torch.Tensor, batch, num_q_heads, num_kv_heads, head_dim,
                       page_size, max_pages, cap_pages, alpha: float, tau: torch.Tensor,
                       mass_out: torch.Tensor, stream=None) -> None:
    """Mass the alpha-entmax with threshold tau puts on each head's kept tokens
    (after an entmaxkv_decode on `workspace`)."""
    _need(tau, "tau", torch.float32, (batch, num_q_heads))
    _need(mass_out, "mass_out", torch.float32, (batch, num_q_heads))
    _check("entmaxkv_kept_mass",
           lib().entmaxkv_kept_mass(_ptr(workspace), batch, num_q_heads, num_kv_heads, head_dim,
                                    page_size, max_pages, cap_pages, float(alpha), _ptr(tau),
                                    _ptr(mass_out), _stream(stream)))


def entmaxkv_read_device_status(stream=None) -> int:
    st = C.c_int32(0)
    _check("entmaxkv_read_device_status",
           lib().entmaxkv_read_device_status(C.byref(st), _stream(stream)))
    return int(st.value)


def entmaxkv_copy_in(dst: torch.Tensor, src: torch.Tensor, stream=None) -> None:
    """Copy src (device memory or pinned host memory) into dst (same size)
    with a kernel instead of a copy engine: a step captured after it has no
    copy-engine hand-off, and the score kernel sets up while it runs."""
    if src.numel() * src.element_size() != dst.numel() * dst.element_size():
        raise ValueError("entmaxkv_copy_in: src and dst differ in size")
    if not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("entmaxkv_copy_in: src and dst must be contiguous")
    _check("entmaxkv_copy_in", lib().entmaxkv_copy_in(_ptr(dst), _ptr(src),
                                                      dst.numel() * dst.element_size(),
                                                      _stream(stream)))


def entmaxkv_check_wait_timeout(limit_us: int, stream=None) -> None:
    """Launch the library's self-check whose bounded wait runs out after
    limit_us microseconds; entmaxkv_read_device_status then reports
    EKV_DEVICE_TIMEOUT."""
    _check("entmaxkv_check_wait_timeout",
           lib().entmaxkv_check_wait_timeout(int(limit_us), _stream(stream)))


def entmaxkv_set_stage_events(events: list | None) -> None:
    """events: four torch.cuda.Event(enable_timing=True), or None to disable."""
    if not events:
        _check("entmaxkv_set_stage_events", lib().entmaxkv_set_stage_events(None, 0))
        return
    for e in events:
        if not e.cuda_event:
            e.record()  # materialise the underlying cudaEvent_t
    arr = (C.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check("entmaxkv_set_stage_events", lib().entmaxkv_set_stage_events(arr, len(events)))


def entmaxkv_decode_counts(workspace: torch.Tensor, batch, num_q_heads, num_kv_heads, head_dim,
                           page_size, max_pages, cap_pages, stream=None):
    """Per-unit (union pages read for K, distinct tokens whose V row was read)
    of the last decode."""
    import numpy as np
    U = batch * num_kv_heads
    up = np.zeros(U, np.int32)
    vp = np.zeros(U, np.int32)
    _check("entmaxkv_decode_counts",
           lib().entmaxkv_decode_counts(_ptr(workspace), batch, num_q_heads, num_kv_heads,
                                        head_dim, page_size, max_pages, cap_pages,
                                        up.ctypes.data_as(C.c_void_p),
                                        vp.ctypes.data_as(C.c_void_p), _stream(stream)))
    return up, vp
