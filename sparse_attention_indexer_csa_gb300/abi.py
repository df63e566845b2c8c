"""ctypes binding of ``libcsa_index.so`` (the C ABI of ``include/csa_index.h``).

Argument marshalling only: tensors are passed as raw pointers with the
caller's CUDA stream, every step of the indexer runs in the library's
kernels.  There is no fallback: if the library is missing or a call fails,
an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcsa_index.so")

CSA_OK, CSA_ERR_INVALID_ARG, CSA_ERR_UNSUPPORTED, CSA_ERR_CUDA, CSA_ERR_TIMEOUT, CSA_ERR_DEVICE = range(6)
CSA_BF16, CSA_F32 = 0, 1
CSA_Q_HEAD_MAJOR, CSA_Q_SEQ_MAJOR = 0, 1

EXPORTED = (
    "csa_index_score",
    "csa_index_topk",
    "csa_index_fused",
    "csa_index_fused_noalloc",
    "csa_index_fused_host",
    "csa_index_fused_host_bytes",
    "csa_index_gather",
    "csa_index_backward",
    "csa_index_workspace_size",
    "csa_index_device_status",
    "csa_index_selftest_timeout",
    "csa_status_string",
    "csa_index_abi_version",
)


class CsaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} failed: status {status} ({msg})")
        self.status = status


class Problem(ctypes.Structure):
    """Mirror of ``csa_problem`` (strides in elements; 0 = contiguous)."""

    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("S", ctypes.c_int32),
        ("D", ctypes.c_int32), ("W", ctypes.c_int32), ("compress_rate", ctypes.c_int32),
        ("scale", ctypes.c_float), ("top_k", ctypes.c_int32), ("w_dtype", ctypes.c_int32),
        ("q_layout", ctypes.c_int32),
        ("q_stride_b", ctypes.c_int64), ("q_stride_h", ctypes.c_int64), ("q_stride_s", ctypes.c_int64),
        ("k_stride_b", ctypes.c_int64), ("k_stride_w", ctypes.c_int64),
        ("w_stride_b", ctypes.c_int64), ("w_stride_s", ctypes.c_int64),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with sparse_attention_indexer_csa_gb300.build.build()")
    lib = ctypes.CDLL(p)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    P = ctypes.POINTER(Problem)
    lib.csa_index_score.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_index_topk.argtypes = [P, vp, vp, vp, sz, vp]
    lib.csa_index_fused.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.csa_index_fused_noalloc.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.csa_index_fused_host.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.csa_index_fused_host_bytes.argtypes = [P, vp, i32, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    lib.csa_index_gather.argtypes = [P, vp, vp, vp, vp]
    lib.csa_index_backward.argtypes = [P, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.csa_index_workspace_size.argtypes = [P, i32]
    lib.csa_index_workspace_size.restype = sz
    lib.csa_index_device_status.argtypes = [vp]
    lib.csa_index_selftest_timeout.argtypes = [ctypes.c_uint32, vp]
    lib.csa_status_string.argtypes = [i32]
    lib.csa_status_string.restype = ctypes.c_char_p
    lib.csa_index_abi_version.restype = i32
    for name in ("csa_index_score", "csa_index_topk", "csa_index_fused", "csa_index_fused_noalloc",
                 "csa_index_fused_host", "csa_index_fused_host_bytes", "csa_index_gather",
                 "csa_index_backward",
                 "csa_index_device_status",
                 "csa_index_selftest_timeout"):
        getattr(lib, name).restype = i32
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().csa_status_string(status).decode()


def _check(fn: str, status: int):
    if status != CSA_OK:
        raise CsaError(fn, status, status_string(status))


def _ptr(t: Optional[torch.Tensor], strided: bool = False):
    """Device pointer of `t`.  Inputs whose strides the problem carries (q, k,
    w) may be views with a contiguous innermost dimension; every other
    tensor must be contiguous."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to the library must live on the GPU")
    if strided:
        if t.dim() > 0 and t.stride(-1) != 1 and t.shape[-1] != 1:
            raise ValueError("the innermost dimension of q, k and w must be contiguous")
    elif not t.is_contiguous():
        raise ValueError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def make_problem(q: torch.Tensor, k: torch.Tensor, w: torch.Tensor, scale: float, compress_rate: int,
                 top_k: int = 1, q_layout: int = CSA_Q_HEAD_MAJOR) -> Problem:
    """Problem of q [B,H,S,D] (head-major) or q [B,S,H,D] (q_layout=CSA_Q_SEQ_MAJOR),
    k [B,W,D], w [B,S,H]; the tensors' own strides are passed on, so views
    (e.g. q sliced out of a wider projection output) need no copy."""
    if q_layout == CSA_Q_SEQ_MAJOR:
        B, S, H, D = q.shape
        qb, qs, qh = q.stride(0), q.stride(1), q.stride(2)
    else:
        B, H, S, D = q.shape
        qb, qh, qs = q.stride(0), q.stride(1), q.stride(2)
    W = k.shape[1]
    wd = {torch.bfloat16: CSA_BF16, torch.float32: CSA_F32}.get(w.dtype)
    if wd is None:
        raise ValueError("weights must be bf16 or fp32")
    # a dimension of extent 1 has no meaningful stride: leave the default
    one = lambda n, st: 0 if n == 1 else int(st)  # noqa: E731
    return Problem(B, H, S, D, W, int(compress_rate), float(scale), int(top_k), wd, int(q_layout),
                   one(B, qb), one(H, qh), one(S, qs), one(B, k.stride(0)), one(W, k.stride(1)),
                   one(B, w.stride(0)), one(S, w.stride(1)))


# ----------------------------------------------------------------------------- raw C-ABI calls
def index_score_raw(p: Problem, q, k, w, q_seg, kv_seg, q_start, scores, stream=None) -> int:
    return load().csa_index_score(ctypes.byref(p), _ptr(q, True), _ptr(k, True), _ptr(w, True), _ptr(q_seg),
                                  _ptr(kv_seg),
                                  _ptr(q_start), _ptr(scores), _stream(stream))


def index_topk_raw(p: Problem, scores, idx, workspace=None, stream=None) -> int:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return load().csa_index_topk(ctypes.byref(p), _ptr(scores), _ptr(idx), _ptr(workspace), nbytes,
                                 _stream(stream))


def index_fused_raw(p: Problem, q, k, w, q_seg, kv_seg, q_start, idx, scores_dbg=None, workspace=None,
                    stream=None) -> int:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return load().csa_index_fused(ctypes.byref(p), _ptr(q, True), _ptr(k, True), _ptr(w, True), _ptr(q_seg),
                                  _ptr(kv_seg),
                                  _ptr(q_start), _ptr(idx), _ptr(scores_dbg), _ptr(workspace), nbytes,
                                  _stream(stream))


def index_fused_noalloc_raw(p: Problem, q, k, w, q_seg, kv_seg, q_start, idx, stream=None) -> int:
    """csa_index_fused_noalloc: no workspace, scores in the library's static scratch."""
    return load().csa_index_fused_noalloc(ctypes.byref(p), _ptr(q, True), _ptr(k, True), _ptr(w, True),
                                          _ptr(q_seg), _ptr(kv_seg),
                                          _ptr(q_start), _ptr(idx), _stream(stream))


def _host_ptr(t: Optional[torch.Tensor]):
    """Host pointer of a contiguous CPU tensor (csa_index_fused_host)."""
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("csa_index_fused_host takes host (CPU) tensors")
    if not t.is_contiguous():
        raise ValueError("host tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def index_fused_host_raw(p: Problem, q, k, w, q_seg, kv_seg, q_start, idx, workspace, stream=None) -> int:
    """csa_index_fused_host: host inputs and idx, device `workspace`."""
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return load().csa_index_fused_host(ctypes.byref(p), _host_ptr(q), _host_ptr(k), _host_ptr(w), _host_ptr(q_seg),
                                       _host_ptr(kv_seg), _host_ptr(q_start), _host_ptr(idx), _ptr(workspace),
                                       nbytes, _stream(stream))


def fused_host_bytes(p: Problem, q_start=None, with_segments: bool = False):
    """(host->device, device->host) bytes of one csa_index_fused_host call."""
    h2d, d2h = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("csa_index_fused_host_bytes",
           load().csa_index_fused_host_bytes(ctypes.byref(p), _host_ptr(q_start), 1 if with_segments else 0,
                                             ctypes.byref(h2d), ctypes.byref(d2h)))
    return int(h2d.value), int(d2h.value)


def index_backward_raw(p: Problem, q, k, w, q_seg, kv_seg, q_start, g, dq, dk, dw, workspace=None,
                       stream=None) -> int:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return load().csa_index_backward(ctypes.byref(p), _ptr(q, True), _ptr(k, True), _ptr(w, True), _ptr(q_seg),
                                     _ptr(kv_seg),
                                     _ptr(q_start), _ptr(g), _ptr(dq), _ptr(dk), _ptr(dw), _ptr(workspace), nbytes,
                                     _stream(stream))


def workspace_size(p: Problem, which: int) -> int:
    return int(load().csa_index_workspace_size(ctypes.byref(p), which))


def device_status(stream=None) -> int:
    return int(load().csa_index_device_status(_stream(stream)))


def selftest_timeout(timeout_us: int, stream=None) -> int:
    return int(load().csa_index_selftest_timeout(timeout_us, _stream(stream)))


# ----------------------------------------------------------------------------- tensor-level helpers
def index_score(q, k, w, scale, compress_rate, q_seg=None, kv_seg=None, q_start=None, out=None, stream=None,
                q_layout=CSA_Q_HEAD_MAJOR):
    """Scores [B,S,W] fp32 (-inf where masked) on the GPU."""
    p = make_problem(q, k, w, scale, compress_rate, 1, q_layout)
    if out is None:
        out = torch.empty(p.B, p.S, p.W, dtype=torch.float32, device=q.device)
    _check("csa_index_score", index_score_raw(p, q, k, w, q_seg, kv_seg, q_start, out, stream))
    return out


def index_topk(scores, top_k, out=None, stream=None):
    """Per-row selection from scores [B,S,W] fp32 -> idx [B,S,top_k] int32."""
    B, S, W = scores.shape
    p = Problem(B, 1, S, 1, W, 1, 1.0, int(top_k), CSA_F32, CSA_Q_HEAD_MAJOR)
    if out is None:
        out = torch.empty(B, S, top_k, dtype=torch.int32, device=scores.device)
    _check("csa_index_topk", index_topk_raw(p, scores, out, None, stream))
    return out


def index_fused(q, k, w, scale, compress_rate, top_k, q_seg=None, kv_seg=None, q_start=None, out=None,
                scores_dbg=None, workspace=None, stream=None, q_layout=CSA_Q_HEAD_MAJOR):
    """Scores and selection in one call -> idx [B,S,top_k] int32."""
    p = make_problem(q, k, w, scale, compress_rate, top_k, q_layout)
    if out is None:
        out = torch.empty(p.B, p.S, p.top_k, dtype=torch.int32, device=q.device)
    need = workspace_size(p, 1)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check("csa_index_fused", index_fused_raw(p, q, k, w, q_seg, kv_seg, q_start, out, scores_dbg,
                                              workspace, stream))
    return out


def index_fused_host(q, k, w, scale, compress_rate, top_k, q_seg=None, kv_seg=None, q_start=None, out=None,
                     workspace=None, stream=None, q_layout=CSA_Q_HEAD_MAJOR, device=None):
    """csa_index_fused on host tensors (pinned for asynchronous copies) ->
    idx [B,S,top_k] int32 on the host, valid once `stream` has been
    synchronised (this helper does not wait)."""
    p = make_problem(q, k, w, scale, compress_rate, top_k, q_layout)
    if out is None:
        out = torch.empty(p.B, p.S, p.top_k, dtype=torch.int32, pin_memory=True)
    if workspace is None:
        workspace = torch.empty(workspace_size(p, 3), dtype=torch.uint8,
                                device=device if device is not None else torch.cuda.current_device())
    _check("csa_index_fused_host", index_fused_host_raw(p, q, k, w, q_seg, kv_seg, q_start, out, workspace, stream))
    return out


def index_backward(q, k, w, scale, compress_rate, g, q_seg=None, kv_seg=None, q_start=None, workspace=None,
                   stream=None, q_layout=CSA_Q_HEAD_MAJOR):
    """Gradients of sum(g * score) over the visible scores -> (dq in q's
    layout, dk [B,W,D], dw [B,S,H]), fp32, for g [B,S,W] fp32."""
    p = make_problem(q, k, w, scale, compress_rate, 1, q_layout)
    dq = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    dk = torch.empty(p.B, p.W, p.D, dtype=torch.float32, device=q.device)
    dw = torch.empty(p.B, p.S, p.H, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(workspace_size(p, 2), dtype=torch.uint8, device=q.device)
    _check("csa_index_backward", index_backward_raw(p, q, k, w, q_seg, kv_seg, q_start, g, dq, dk, dw,
                                                    workspace, stream))
    return dq, dk, dw


def index_gather(k, idx, out=None, stream=None):
    """Selected compressed rows: out[b,s,i,:] = k[b, idx[b,s,i], :] (zeros for -1)."""
    B, W, D = k.shape
    _, S, K = idx.shape
    p = Problem(B, 1, S, D, W, 1, 1.0, int(K), CSA_BF16, CSA_Q_HEAD_MAJOR)
    p.k_stride_b = 0 if B == 1 else k.stride(0)
    p.k_stride_w = 0 if W == 1 else k.stride(1)
    if out is None:
        out = torch.empty(B, S, K, D, dtype=k.dtype, device=k.device)
    _check("csa_index_gather", load().csa_index_gather(ctypes.byref(p), _ptr(k, True), _ptr(idx), _ptr(out),
                                                       _stream(stream)))
    return out


def index_decode(q, k, w, scale, compress_rate, top_k, q_start, q_seg=None, kv_seg=None, **kw):
    """Autoregressive selection: one query row per sequence.

    The segment mask is not applied in autoregressive mode ("DSV4: Add
    indexer_save_selection and indexer_sharded_topk", review of the decode
    mask), so segment ids given here are ignored.
    """
    del q_seg, kv_seg
    return index_fused(q, k, w, scale, compress_rate, top_k, None, None, q_start, **kw)
