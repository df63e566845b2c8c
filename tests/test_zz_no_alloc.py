"""The allocation-free fused entry point against the regular one (GPU).

csa_index_fused_noalloc serves callers that cannot allocate device memory
where they call the indexer (their memory pool already holds the free device
memory, or an allocation's implicit device synchronisation is not allowed):
it needs no workspace and keeps the scores in a fixed 8 MiB scratch array
inside the library.  These tests call it through the C ABI twice in a row on
each problem and check that every call returns exactly the indices of
csa_index_fused, the tested entry point, so the reused scratch carries
nothing from one call into the next.  This file is collected last.
"""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_csa_gb300 as csa
from csa_inputs import WORKLOADS, Workload, make_inputs
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu

MAX_SCORES = 2 * 1024 * 1024  # capacity of the library's scratch, in fp32 scores


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    csa.load()


def _dev(inp):
    g = lambda t: None if t is None else t.cuda().contiguous()  # noqa: E731
    return g(inp.q), g(inp.k), g(inp.w), g(inp.q_seg), g(inp.kv_seg), g(inp.q_start)


def _two_calls_match_fused(inp):
    wl = inp.wl
    q, k, w, qs, ks, st = _dev(inp)
    ref = csa.index_fused(q, k, w, wl.scale, wl.compress_rate, wl.top_k, qs, ks, st)
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    for _ in range(2):
        out = torch.full((wl.B, wl.S, wl.top_k), -7, dtype=torch.int32, device="cuda")
        status = csa.abi.index_fused_noalloc_raw(p, q, k, w, qs, ks, st, out)
        assert status == csa.CSA_OK, csa.abi.status_string(status)
        torch.cuda.synchronize()
        assert csa.device_status() == csa.CSA_OK
        assert torch.equal(out, ref)


def test_decode_rows_match_fused():
    # 8 single-row sequences over 32768 entries: the decode-style path
    _two_calls_match_fused(make_inputs(WORKLOADS["decode_32k"].with_(B=8, seed=5)))


def test_selection_equals_oracle_selector_on_gpu_scores():
    # the oracle's selector, run on the scores of csa_index_score (the same
    # score kernel the no-allocation path runs), reproduces its indices
    wl = WORKLOADS["prefill_4k"].with_(S=700, W=175, top_k=50, seed=11)
    inp = make_inputs(wl)
    q, k, w, qs, ks, st = _dev(inp)
    sc = csa.index_score(q, k, w, wl.scale, wl.compress_rate)
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    out = torch.empty(wl.B, wl.S, wl.top_k, dtype=torch.int32, device="cuda")
    assert csa.abi.index_fused_noalloc_raw(p, q, k, w, None, None, None, out) == csa.CSA_OK
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
    ref = O.select_topk(sc.double().cpu().numpy(), wl.top_k)
    assert np.array_equal(out.cpu().numpy(), ref)


def test_calls_ordered_on_a_non_default_stream():
    # two calls enqueued on one side stream, the second right behind the
    # first (the scratch is reused in stream order), read after that stream
    wl = WORKLOADS["decode_32k"].with_(B=4, W=8192, q_start=32767, seed=12)
    inp = make_inputs(wl)
    q, k, w, qs, ks, st = _dev(inp)
    ref = csa.index_fused(q, k, w, wl.scale, wl.compress_rate, wl.top_k, q_start=st)
    torch.cuda.synchronize()
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    side = torch.cuda.Stream()
    outs = [torch.full((wl.B, wl.S, wl.top_k), -7, dtype=torch.int32, device="cuda") for _ in range(2)]
    side.wait_stream(torch.cuda.current_stream())
    for o in outs:
        assert csa.abi.index_fused_noalloc_raw(p, q, k, w, None, None, st, o, stream=side) == csa.CSA_OK
    side.synchronize()
    assert csa.device_status(side) == csa.CSA_OK
    for o in outs:
        assert torch.equal(o, ref)


def test_prefill_rows_match_fused():
    _two_calls_match_fused(make_inputs(WORKLOADS["prefill_4k"].with_(S=1200, W=300, top_k=64, seed=6)))


def test_packed_documents_match_fused():
    wl = WORKLOADS["packed_8k"].with_(B=2, S=1024, W=256, top_k=40, seed=7)
    _two_calls_match_fused(make_inputs(wl))


def test_largest_problem_fits_and_one_more_row_is_rejected():
    wl = Workload(name="cap", B=64, S=1, W=32768, H=64, D=128, compress_rate=4, top_k=16,
                  w_dtype="bf16", sigma_w=0.125, scale=128 ** -0.5, q_start=131071, seed=8)
    assert wl.B * wl.S * wl.W == MAX_SCORES
    inp = make_inputs(wl)
    _two_calls_match_fused(inp)
    q, k, w, qs, ks, st = _dev(inp)
    p = csa.make_problem(q, k, w, wl.scale, wl.compress_rate, wl.top_k)
    p.S = 2  # one score beyond the scratch: refused before any launch
    out = torch.empty(1, dtype=torch.int32, device="cuda")
    assert csa.abi.index_fused_noalloc_raw(p, q, k, w, None, None, st, out) == csa.CSA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
