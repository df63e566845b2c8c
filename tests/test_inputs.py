"""Host checks of the seeded input generator (no GPU)."""
import torch

from csa_inputs import WORKLOADS, make_inputs


def test_tiny_shapes_and_dtypes():
    inp = make_inputs(WORKLOADS["tiny"])
    assert inp.q.shape == (1, 4, 256, 32) and inp.q.dtype == torch.bfloat16
    assert inp.k.shape == (1, 64, 32) and inp.k.dtype == torch.bfloat16
    assert inp.w.shape == (1, 256, 4) and inp.w.dtype == torch.float32
    assert inp.q_seg is None and inp.q_start is None


def test_deterministic():
    a = make_inputs(WORKLOADS["tiny"])
    b = make_inputs(WORKLOADS["tiny"])
    assert torch.equal(a.q, b.q) and torch.equal(a.k, b.k) and torch.equal(a.w, b.w)
    c = make_inputs(WORKLOADS["tiny"].with_(seed=1))
    assert not torch.equal(a.q, c.q)


def test_packed_segments_structure():
    wl = WORKLOADS["packed_8k"].with_(S=512, W=128)
    inp = make_inputs(wl)
    r = wl.compress_rate
    for b in range(wl.B):
        seg = inp.q_seg[b]
        n = int(seg[-1]) + 1
        assert 3 <= n <= 8
        assert bool((seg[1:] >= seg[:-1]).all())
        cuts = torch.nonzero(seg[1:] != seg[:-1]).flatten() + 1
        assert bool((cuts % r == 0).all())
        last = torch.arange(wl.W) * r + r - 1
        assert torch.equal(inp.kv_seg[b], seg[last])
