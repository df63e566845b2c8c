"""GPU parity of csa_index_fused_host: host inputs and indices, the copies
enqueued by the library.  Its result must equal csa_index_fused's on the
same inputs, bit for bit, while it transfers only the q rows that can need
scores; the q rows it skips are filled with NaN in the device workspace
first, so a read of any of them would change the selection."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_csa_gb300 as csa
from csa_inputs import WORKLOADS, make_inputs
from parity import assert_status_ok, check_select_vs_oracle, oracle_scores, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    csa.load()


def _pinned(t):
    return None if t is None else t.contiguous().pin_memory()


def _run_host(inp, q_layout=csa.CSA_Q_HEAD_MAJOR, poison=True):
    wl = inp.wl
    q = inp.q if q_layout == csa.CSA_Q_HEAD_MAJOR else inp.q.permute(0, 2, 1, 3).contiguous()
    hq, hk, hw = _pinned(q), _pinned(inp.k), _pinned(inp.w)
    hqs, hks, hst = _pinned(inp.q_seg), _pinned(inp.kv_seg), _pinned(inp.q_start)
    p = csa.make_problem(hq, hk, hw, wl.scale, wl.compress_rate, wl.top_k, q_layout)
    ws = torch.empty(csa.workspace_size(p, 3), dtype=torch.uint8, device="cuda")
    if poison:
        ws.fill_(0xFF)  # bf16 0xFFFF is a NaN: every q row left uncopied reads as NaN
    out = torch.full((wl.B, wl.S, wl.top_k), -7, dtype=torch.int32).pin_memory()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    st = csa.index_fused_host_raw(p, hq, hk, hw, hqs, hks, hst, out, ws, stream)
    assert st == csa.CSA_OK, csa.abi.status_string(st)
    stream.synchronize()
    h2d, d2h = csa.fused_host_bytes(p, hst, hqs is not None)
    return out, h2d, d2h


def _device_fused(inp, q_layout=csa.CSA_Q_HEAD_MAJOR):
    wl = inp.wl
    d = to_dev(inp)
    q = d["q"] if q_layout == csa.CSA_Q_HEAD_MAJOR else d["q"].permute(0, 2, 1, 3).contiguous()
    return csa.index_fused(q, d["k"], d["w"], wl.scale, wl.compress_rate, wl.top_k, d["q_seg"], d["kv_seg"],
                           d["q_start"], q_layout=q_layout).cpu()


def _q_rows_sent(wl, q_start):
    """Rows of q per batch the host call transfers (one-kernel path): from
    the item of four rows holding the first row whose future-mask bound
    exceeds top_k."""
    rows = []
    for b in range(wl.B):
        qs = 0 if q_start is None else int(q_start[b])
        if wl.W <= wl.top_k:
            rows.append(0)
            continue
        s = (wl.top_k + 1) * wl.compress_rate - qs - 1
        s0 = wl.S if s >= wl.S else (0 if s <= 0 else s // 4 * 4)
        rows.append(wl.S - s0)
    return rows


CASES = [
    # prefill: the first ~half of the rows keep their visible sets (not sent)
    ("prefill_4k", dict(S=2048, W=512, top_k=200), None, csa.CSA_Q_HEAD_MAJOR),
    # two sequences at different offsets, sequence-major q
    ("prefill_4k", dict(B=2, S=1030, W=700, top_k=150), [0, 333], csa.CSA_Q_SEQ_MAJOR),
    # a row block straddling the bound (top_k + 1) * r - 1 that is not a multiple of 4
    ("prefill_4k", dict(S=777, W=300, top_k=61, compress_rate=3), [5], csa.CSA_Q_HEAD_MAJOR),
    # packed documents: segment ids copied too, the document-mode kernel
    ("packed_8k", dict(B=2, S=2048, W=512, top_k=60, seed=1), None, csa.CSA_Q_HEAD_MAJOR),
    # every row at or below top_k: no q row is sent
    ("prefill_4k", dict(S=512, W=128, top_k=128), None, csa.CSA_Q_HEAD_MAJOR),
]


@pytest.mark.parametrize("ci", range(len(CASES)))
def test_host_entry_equals_device_entry(ci):
    name, over, q_start, layout = CASES[ci]
    wl = WORKLOADS[name].with_(**over)
    inp = make_inputs(wl)
    if q_start is not None:
        inp.q_start = torch.tensor(q_start, dtype=torch.int64)
    got, h2d, d2h = _run_host(inp, layout)
    want = _device_fused(inp, layout)
    assert_status_ok()
    assert torch.equal(got, want)
    # bytes: the q rows of _q_rows_sent, plus k, w, ids and offsets; idx back
    q_row = wl.H * wl.D * 2
    other = inp.k.numel() * 2 + inp.w.numel() * inp.w.element_size()
    if inp.q_seg is not None:
        other += (inp.q_seg.numel() + inp.kv_seg.numel()) * 4
    if inp.q_start is not None:
        other += wl.B * 8
    sent = _q_rows_sent(wl, inp.q_start)
    assert h2d == sum(sent) * q_row + other
    assert d2h == got.numel() * 4
    if ci == 0:
        assert sent == [wl.S - 800]  # rows 800.. of 2048 ((200 + 1) * 4 - 1 = 803 -> item 200)
    if ci == len(CASES) - 1:
        assert sent == [0]


def test_host_entry_against_the_oracle():
    """Sampled rows of a host call, selection compared with the oracle."""
    wl = WORKLOADS["prefill_4k"].with_(S=1536, W=384, top_k=100, seed=5)
    inp = make_inputs(wl)
    got, _, _ = _run_host(inp)
    rows = np.array([0, 1, 402, 403, 404, 405, 900, 1535])
    ref = oracle_scores(inp, rows=rows)
    check_select_vs_oracle(ref, got.numpy()[:, rows], wl.top_k)


def test_host_entry_two_pass_path_copies_all_of_q():
    """Single-row (decode) problems take the two-pass path, which reads
    every q row: all of q is sent and the result equals the device call."""
    wl = WORKLOADS["decode_32k"].with_(B=4, W=4096, q_start=16383)
    inp = make_inputs(wl)
    got, h2d, _ = _run_host(inp)
    want = _device_fused(inp)
    assert torch.equal(got, want)
    assert h2d >= inp.q.numel() * 2 + inp.k.numel() * 2


def test_host_calls_in_flight_on_two_streams():
    """Two calls with separate workspaces overlapping on two streams: each
    result equals its own device call."""
    wls = [WORKLOADS["prefill_4k"].with_(S=1024, W=256, top_k=64, seed=s) for s in (7, 8)]
    inps = [make_inputs(wl) for wl in wls]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for inp, stream in zip(inps, streams):
        wl = inp.wl
        hq, hk, hw = _pinned(inp.q), _pinned(inp.k), _pinned(inp.w)
        p = csa.make_problem(hq, hk, hw, wl.scale, wl.compress_rate, wl.top_k)
        ws = torch.empty(csa.workspace_size(p, 3), dtype=torch.uint8, device="cuda")
        out = torch.empty(wl.B, wl.S, wl.top_k, dtype=torch.int32).pin_memory()
        stream.wait_stream(torch.cuda.current_stream())
        assert csa.index_fused_host_raw(p, hq, hk, hw, None, None, None, out, ws, stream) == csa.CSA_OK
        outs.append((out, ws, hq, hk, hw))
    torch.cuda.synchronize()
    for (out, *_), inp in zip(outs, inps):
        assert torch.equal(out, _device_fused(inp))
