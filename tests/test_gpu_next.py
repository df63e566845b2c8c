"""GPU parity of the widened path: sequence-major q, decode batches of
sequences with different lengths, and the gather of the selected rows."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_csa_gb300 as csa
from csa_inputs import WORKLOADS, make_inputs
from oracle import csa_oracle as O
from parity import (assert_status_ok, check_scores, check_select_exact, check_select_vs_oracle, oracle_scores,
                    to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    csa.load()


@pytest.mark.parametrize("name,over", [("tiny", {}), ("prefill_4k", dict(S=1000, W=250, top_k=100)),
                                       ("packed_8k", dict(B=2, S=1024, W=256, top_k=40))])
def test_sequence_major_q_equals_head_major(name, over):
    """q stored [B,S,H,D] gives the same bits as q stored [B,H,S,D]."""
    wl = WORKLOADS[name].with_(**over)
    inp = make_inputs(wl)
    d = to_dev(inp)
    q_sm = d["q"].permute(0, 2, 1, 3).contiguous()
    args = (wl.scale, wl.compress_rate)
    hm = csa.index_score(d["q"], d["k"], d["w"], *args, d["q_seg"], d["kv_seg"], d["q_start"])
    sm = csa.index_score(q_sm, d["k"], d["w"], *args, d["q_seg"], d["kv_seg"], d["q_start"],
                         q_layout=csa.CSA_Q_SEQ_MAJOR)
    i_hm = csa.index_fused(d["q"], d["k"], d["w"], *args, wl.top_k, d["q_seg"], d["kv_seg"], d["q_start"])
    i_sm = csa.index_fused(q_sm, d["k"], d["w"], *args, wl.top_k, d["q_seg"], d["kv_seg"], d["q_start"],
                           q_layout=csa.CSA_Q_SEQ_MAJOR)
    assert_status_ok()
    assert torch.equal(hm, sm)
    assert torch.equal(i_hm, i_sm)
    check_scores(sm.cpu().numpy(), oracle_scores(inp))


def test_decode_sequences_of_different_lengths():
    """One k buffer sized for the longest sequence; each sequence's position
    bounds what it sees, and entries past its length are never selected."""
    wl = WORKLOADS["decode_32k"].with_(B=12, seed=3)
    inp = make_inputs(wl)
    g = torch.Generator().manual_seed(4)
    lengths = torch.randint(1, 4 * wl.W, (wl.B,), generator=g)  # tokens per sequence
    lengths[0], lengths[1], lengths[2] = 1, 4 * wl.W, 4 * 2048 + 3   # empty, full, near top_k
    inp.q_start = (lengths - 1).to(torch.int64)
    d = to_dev(inp)
    sc = csa.index_score(d["q"], d["k"], d["w"], wl.scale, wl.compress_rate, q_start=d["q_start"])
    idx = csa.index_fused(d["q"], d["k"], d["w"], wl.scale, wl.compress_rate, wl.top_k, q_start=d["q_start"])
    assert_status_ok()
    ref = oracle_scores(inp)
    g_sc = sc.cpu().numpy()
    check_scores(g_sc, ref)
    gi = idx.cpu().numpy()
    check_select_exact(g_sc, gi, wl.top_k)
    check_select_vs_oracle(ref, gi, wl.top_k)
    for b in range(wl.B):
        n_vis = int(lengths[b]) // wl.compress_rate
        assert np.all(gi[b][gi[b] >= 0] < n_vis)


def test_gather_selected_rows_bit_exact():
    wl = WORKLOADS["decode_32k"].with_(B=6, seed=9, top_k=300)
    inp = make_inputs(wl)
    inp.q_start = torch.tensor([131071, 131071, 200, 3, 0, 4000], dtype=torch.int64)  # short rows pad with -1
    d = to_dev(inp)
    idx = csa.index_fused(d["q"], d["k"], d["w"], wl.scale, wl.compress_rate, wl.top_k, q_start=d["q_start"])
    out = csa.index_gather(d["k"], idx)
    assert_status_ok()
    i_np = idx.cpu().numpy()
    assert (i_np == -1).any()
    ref = O.gather_selected(inp.k.view(torch.int16).numpy(), i_np)  # compare the bf16 bit patterns
    assert np.array_equal(out.cpu().view(torch.int16).numpy(), ref)


def test_gather_reports_out_of_range_indices():
    k = torch.randn(1, 10, 128, device="cuda").to(torch.bfloat16)
    idx = torch.tensor([[[0, 9, -1, 10, 3]]], dtype=torch.int32, device="cuda")
    out = csa.index_gather(k, idx)
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_ERR_DEVICE
    assert csa.device_status() == csa.CSA_OK
    o = out[0, 0]
    assert torch.equal(o[0], k[0, 0]) and torch.equal(o[1], k[0, 9]) and torch.equal(o[4], k[0, 3])
    assert bool((o[2] == 0).all()) and bool((o[3] == 0).all())


def test_strided_views_equal_contiguous_inputs():
    """q sliced out of a wider [B,S,H',D] projection output, k rows with a
    padded pitch, w with padded rows: the same scores, selection, gather and
    backward as contiguous copies of the same values, with no copy made."""
    wl = WORKLOADS["prefill_4k"].with_(B=2, S=700, W=300, top_k=60, seed=31)
    inp = make_inputs(wl)
    B, H, S, D, W = wl.B, wl.H, wl.S, wl.D, wl.W
    g = torch.Generator().manual_seed(32)
    big_q = torch.randn(B, S, H + 32, D, generator=g).to(torch.bfloat16)
    big_q[:, :, 16:16 + H] = inp.q.permute(0, 2, 1, 3)
    q_view = big_q.cuda()[:, :, 16:16 + H]                      # [B,S,H,D], row pitch (H+32)*D
    big_k = torch.zeros(B, W + 3, D + 64, dtype=torch.bfloat16)
    big_k[:, 3:, :D] = inp.k
    k_view = big_k.cuda()[:, 3:, :D]                             # row pitch D+64, offset 3 rows
    big_w = torch.zeros(B, S, H + 8, dtype=inp.w.dtype)
    big_w[:, :, 4:4 + H] = inp.w
    w_view = big_w.cuda()[:, :, 4:4 + H]                         # row pitch H+8
    assert not q_view.is_contiguous() and not k_view.is_contiguous() and not w_view.is_contiguous()
    d = to_dev(inp)
    q_sm = d["q"].permute(0, 2, 1, 3).contiguous()
    sm = csa.CSA_Q_SEQ_MAJOR
    args = (wl.scale, wl.compress_rate)
    s_ref = csa.index_score(q_sm, d["k"], d["w"], *args, q_layout=sm)
    s_view = csa.index_score(q_view, k_view, w_view, *args, q_layout=sm)
    i_ref = csa.index_fused(q_sm, d["k"], d["w"], *args, wl.top_k, q_layout=sm)
    i_view = csa.index_fused(q_view, k_view, w_view, *args, wl.top_k, q_layout=sm)
    g_ref = csa.index_gather(d["k"], i_ref)
    g_view = csa.index_gather(k_view, i_view)
    cot = torch.randn(B, S, W, generator=torch.Generator().manual_seed(33)).cuda()
    dq_r, dk_r, dw_r = csa.index_backward(q_sm, d["k"], d["w"], *args, cot, q_layout=sm)
    dq_v, dk_v, dw_v = csa.index_backward(q_view, k_view, w_view, *args, cot, q_layout=sm)
    assert_status_ok()
    assert torch.equal(s_ref, s_view)
    assert torch.equal(i_ref, i_view)
    assert torch.equal(g_ref, g_view)
    assert torch.equal(dq_r, dq_v) and torch.equal(dw_r, dw_v)
    # dk sums its items' partial products with atomics: equal up to the order of fp32 additions
    assert torch.allclose(dk_r, dk_v, rtol=0, atol=1e-5 * float(dk_r.abs().max()))
    check_scores(s_view.cpu().numpy(), oracle_scores(inp))
    # head-major view: q sliced along heads of a [B,H',S,D] buffer
    big_h = torch.zeros(B, H + 8, S, D, dtype=torch.bfloat16)
    big_h[:, 8:] = inp.q
    q_hv = big_h.cuda()[:, 8:]
    assert torch.equal(csa.index_fused(q_hv, k_view, w_view, *args, wl.top_k), i_ref)
