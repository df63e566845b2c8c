"""Host-side checks of the C-ABI library (no GPU, no compute calls).

The library must load, export every entry point declared in
include/csa_index.h, and reject bad arguments on the host before any CUDA
call is made.
"""
import ctypes
import os
import re

import pytest

import sparse_attention_indexer_csa_gb300 as csa
from sparse_attention_indexer_csa_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(abi.LIB_PATH):
        from sparse_attention_indexer_csa_gb300 import build
        build.build()
    return abi.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "csa_index.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert "csa_index_score" in names and "csa_index_fused" in names and "csa_index_topk" in names
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(abi.EXPORTED)


def test_abi_version_and_strings(lib):
    assert lib.csa_index_abi_version() == 106
    for s in range(6):
        assert abi.status_string(s)
    assert abi.status_string(99) == "unknown status"


def _p(**kw):
    d = dict(B=1, H=64, S=16, D=128, W=4, compress_rate=4, scale=0.1, top_k=2, w_dtype=abi.CSA_BF16, q_layout=0)
    d.update(kw)
    return abi.Problem(**d)


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced by the checks
ODD = ctypes.c_void_p(0x10002)


def _score(lib, p, q=FAKE, k=FAKE, w=FAKE, qs=None, kvs=None, st=None, out=FAKE):
    return lib.csa_index_score(ctypes.byref(p) if p is not None else None, q, k, w, qs, kvs, st, out, None)


@pytest.mark.parametrize("bad", [dict(B=0), dict(H=0), dict(S=-1), dict(D=0), dict(W=0),
                                 dict(compress_rate=0), dict(top_k=0), dict(scale=0.0),
                                 dict(scale=-1.0), dict(scale=float("inf")), dict(scale=float("nan")),
                                 dict(w_dtype=7), dict(q_layout=2), dict(q_layout=-1)])
def test_bad_problem_rejected(lib, bad):
    assert _score(lib, _p(**bad)) == abi.CSA_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(q_stride_s=100), dict(q_stride_h=-8), dict(q_stride_b=4), dict(k_stride_w=130),
                                 dict(k_stride_b=-128), dict(w_stride_s=-1), dict(w_stride_b=-64),
                                 dict(q_stride_s=1 << 40)])
def test_bad_strides_rejected(lib, bad):
    # q and k strides feed TMA maps (multiples of 8 bf16 = 16 bytes); none may be negative
    assert _score(lib, _p(**bad)) == abi.CSA_ERR_INVALID_ARG


def test_good_strides_accepted_by_the_checks(lib):
    # valid strides pass the argument checks and reach the device query, which
    # fails only for lack of a device (not an argument error); never run where
    # a device exists, since the pointers here are fake
    import torch
    if torch.cuda.is_available():
        pytest.skip("uses fake pointers; only meaningful without a device")
    ok = _p(q_stride_s=192 * 128, q_stride_h=128, q_stride_b=192 * 128 * 16, k_stride_w=136, w_stride_s=72)
    assert _score(lib, ok) != abi.CSA_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_rejected(lib):
    assert _score(lib, None) == abi.CSA_ERR_INVALID_ARG
    assert _score(lib, _p(), q=None) == abi.CSA_ERR_INVALID_ARG
    assert _score(lib, _p(), out=None) == abi.CSA_ERR_INVALID_ARG
    assert _score(lib, _p(), q=ODD) == abi.CSA_ERR_INVALID_ARG   # TMA needs 16-byte bases
    assert _score(lib, _p(), k=ODD) == abi.CSA_ERR_INVALID_ARG
    # segment ids must come in pairs
    assert _score(lib, _p(), qs=FAKE) == abi.CSA_ERR_INVALID_ARG
    assert _score(lib, _p(), kvs=FAKE) == abi.CSA_ERR_INVALID_ARG


def test_unsupported_shapes_rejected_not_fallen_back(lib):
    assert _score(lib, _p(H=32)) == abi.CSA_ERR_UNSUPPORTED
    assert _score(lib, _p(D=64)) == abi.CSA_ERR_UNSUPPORTED
    p = _p(W=60000)
    assert lib.csa_index_topk(ctypes.byref(p), FAKE, FAKE, None, 0, None) == abi.CSA_ERR_UNSUPPORTED
    p = _p(S=1, W=60000)
    assert lib.csa_index_fused(ctypes.byref(p), FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, 0,
                               None) == abi.CSA_ERR_UNSUPPORTED


def test_fused_large_w_needs_workspace(lib):
    p = _p(S=1, W=32768, B=64)
    need = abi.workspace_size(p, 1)
    assert need == 64 * 1 * 32768 * 4
    assert lib.csa_index_fused(ctypes.byref(p), FAKE, FAKE, FAKE, None, None, None, FAKE, None, None, 0,
                               None) == abi.CSA_ERR_INVALID_ARG
    # one-kernel path: a two-item staging ring per CTA (at most 256 CTAs),
    # then (256-byte aligned) a 64-byte segment summary per item of four rows
    assert abi.workspace_size(_p(W=4096, S=16384), 1) == 256 * 2 * 4 * 4096 * 4 + 1 * 4096 * 64
    ring = 2 * 2 * 4 * 128 * 4
    assert abi.workspace_size(_p(W=100, S=8), 1) == (ring + 255) // 256 * 256 + 2 * 64
    assert abi.workspace_size(_p(), 0) == 0
    assert abi.workspace_size(_p(B=0), 1) == 0


def test_selftest_argument_checks(lib):
    assert lib.csa_index_selftest_timeout(0, None) == abi.CSA_ERR_INVALID_ARG
    assert lib.csa_index_selftest_timeout(20_000_000, None) == abi.CSA_ERR_INVALID_ARG


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError):
        abi.load(str(tmp_path / "missing.so"))


def _bwd(lib, p, g=FAKE, dq=FAKE, dk=FAKE, dw=FAKE, ws=FAKE, nbytes=1 << 40, q=FAKE):
    return lib.csa_index_backward(ctypes.byref(p), q, FAKE, FAKE, None, None, None, g, dq, dk, dw, ws, nbytes, None)


def test_backward_workspace_size():
    # the dk kernel's work counter, then a 64-byte segment summary per item of
    # four rows: P never leaves the SM
    for kw in (dict(S=16, W=4), dict(S=16384, W=4096), dict(S=5, W=300), dict(S=16384, W=32768, B=3)):
        pp = _p(**kw)
        assert abi.workspace_size(pp, 2) == 256 + pp.B * ((pp.S + 3) // 4) * 64
    assert abi.workspace_size(_p(B=0), 2) == 0


def test_backward_argument_checks(lib):
    assert _bwd(lib, _p(B=0)) == abi.CSA_ERR_INVALID_ARG
    for kw in (dict(g=None), dict(dq=None), dict(dk=None), dict(dw=None), dict(q=None), dict(dq=ODD)):
        assert _bwd(lib, _p(), **kw) == abi.CSA_ERR_INVALID_ARG, kw
    # workspace missing, short or misaligned
    need = abi.workspace_size(_p(), 2)
    assert _bwd(lib, _p(), ws=None) == abi.CSA_ERR_INVALID_ARG
    assert _bwd(lib, _p(), nbytes=need - 1) == abi.CSA_ERR_INVALID_ARG
    assert _bwd(lib, _p(), ws=ctypes.c_void_p(0x10004)) == abi.CSA_ERR_INVALID_ARG
    # dq and dk take 16-byte vector stores and atomics
    assert _bwd(lib, _p(), dq=ctypes.c_void_p(0x10008)) == abi.CSA_ERR_INVALID_ARG
    assert _bwd(lib, _p(), dk=ctypes.c_void_p(0x10008)) == abi.CSA_ERR_INVALID_ARG
    # only H=64, D=128
    assert _bwd(lib, _p(H=4, D=32)) == abi.CSA_ERR_UNSUPPORTED


# ----------------------------------------------------------------------------- host-buffer entry point
def _up(x):
    return (x + 255) // 256 * 256


def _host_ws(p):
    """csa_index_workspace_size(p, 3) restated: q, k, w, both id arrays,
    q_start, idx and csa_index_fused's workspace, each 256-byte aligned."""
    wsz = 2 if p.w_dtype == abi.CSA_BF16 else 4
    parts = [p.B * p.H * p.S * p.D * 2, p.B * p.W * p.D * 2, p.B * p.S * p.H * wsz, p.B * p.S * 4, p.B * p.W * 4,
             p.B * 8, p.B * p.S * p.top_k * 4, abi.workspace_size(p, 1)]
    return sum(_up(x) for x in parts)


@pytest.mark.parametrize("kw", [dict(), dict(B=2, S=16384, W=4096, top_k=2048), dict(W=9000, S=300),
                                dict(S=1, W=32768, top_k=2048), dict(w_dtype=abi.CSA_F32, q_layout=1)])
def test_host_workspace_size(lib, kw):
    p = _p(**kw)
    assert abi.workspace_size(p, 3) == _host_ws(p)


def _host_bytes(p, q_start=None, segs=False):
    import torch
    st = None if q_start is None else torch.tensor(q_start, dtype=torch.int64)
    return abi.fused_host_bytes(p, st, segs)


def test_host_bytes_prefill_16k(lib):
    """prefill B=2 S=16384 W=4096 top_k=2048: rows s < 8195 see at most 2048
    entries; the item of rows 8192..8195 is the first that can be scored, so
    rows 8192.. of each batch are sent (half of q)."""
    p = _p(B=2, S=16384, W=4096, top_k=2048)
    h2d, d2h = _host_bytes(p)
    q_rows = 2 * (16384 - 8192) * 64 * 128 * 2
    assert h2d == q_rows + 2 * 4096 * 128 * 2 + 2 * 16384 * 64 * 2
    assert d2h == 2 * 16384 * 2048 * 4
    # sequence-major q: the same rows
    assert _host_bytes(_p(B=2, S=16384, W=4096, top_k=2048, q_layout=1)) == (h2d, d2h)


def test_host_bytes_follow_offsets_ids_and_paths(lib):
    row = 64 * 128 * 2
    base = 2 * 4096 * 128 * 2 + 2 * 16384 * 64 * 2
    p = _p(B=2, S=16384, W=4096, top_k=2048)
    # a sequence starting at position 8000 sees more than top_k entries from
    # row 196 ((2048 + 1) * 4 - 8000 - 1 = 195 -> item of rows 192..195);
    # one starting at 100000 from its first row
    h2d, _ = _host_bytes(p, q_start=[8000, 100000])
    assert h2d == (16384 - 192) * row + 16384 * row + base + 2 * 8
    # segment ids are sent when given
    h2d_s, _ = _host_bytes(p, segs=True)
    assert h2d_s == 2 * 8192 * row + base + 2 * 16384 * 4 + 2 * 4096 * 4
    # W <= top_k: every row keeps its visible set, no q row is sent
    p = _p(B=1, S=4096, W=1024, top_k=1024)
    assert _host_bytes(p)[0] == 1024 * 128 * 2 + 4096 * 64 * 2
    # single-row problems and rows past 16384 entries take two passes: all of q
    for kw in (dict(B=3, S=1, W=32768, top_k=2048), dict(B=1, S=64, W=20000, top_k=2048)):
        p = _p(**kw)
        h2d, _ = _host_bytes(p)
        assert h2d == p.B * p.S * row + p.B * p.W * 128 * 2 + p.B * p.S * 64 * 2


def _host_call(lib, p, q=FAKE, k=FAKE, w=FAKE, qs=None, kvs=None, st=None, out=FAKE, ws=FAKE, nbytes=None):
    nbytes = abi.workspace_size(p, 3) if nbytes is None else nbytes
    return lib.csa_index_fused_host(ctypes.byref(p), q, k, w, qs, kvs, st, out, ws, nbytes, None)


def test_host_entry_argument_checks(lib):
    """Every check returns before a copy is enqueued (no GPU here)."""
    p = _p(S=64, W=16, top_k=4)
    assert _host_call(lib, p, q=None) == abi.CSA_ERR_INVALID_ARG
    assert _host_call(lib, p, out=None) == abi.CSA_ERR_INVALID_ARG
    assert _host_call(lib, p, qs=FAKE) == abi.CSA_ERR_INVALID_ARG  # ids of one side only
    assert _host_call(lib, p, ws=None) == abi.CSA_ERR_INVALID_ARG
    assert _host_call(lib, p, ws=ctypes.c_void_p(0x10010)) == abi.CSA_ERR_INVALID_ARG  # not 256-byte aligned
    assert _host_call(lib, p, nbytes=abi.workspace_size(p, 3) - 1) == abi.CSA_ERR_INVALID_ARG
    strided = _p(S=64, W=16, top_k=4, q_stride_s=256)  # rows further apart than D
    assert _host_call(lib, strided) == abi.CSA_ERR_INVALID_ARG
    dense = _p(S=64, W=16, top_k=4, q_stride_b=64 * 64 * 128, q_stride_h=64 * 128, q_stride_s=128)
    assert _host_call(lib, dense, ws=None) == abi.CSA_ERR_INVALID_ARG  # the strides pass; the workspace does not
    assert _host_call(lib, _p(S=64, W=16, top_k=4, H=8)) == abi.CSA_ERR_UNSUPPORTED
    assert _host_call(lib, _p(S=1, W=60000, top_k=4)) == abi.CSA_ERR_UNSUPPORTED
