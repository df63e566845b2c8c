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
