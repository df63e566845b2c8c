"""GPU selection kernel on crafted score matrices, checked exactly against the
oracle selector.  The cases drive every branch of the selection, in the
one-CTA kernel and, for rows longer than 16384, the four-CTA cluster kernel:
continuous scores (binned search), heavy ties (threshold bin over capacity: radix
search), all-equal rows, signed zeros, a value range whose width overflows
fp32, denormals, scores far from zero relative to their spread, masked
entries, and rows with fewer visible entries than k."""
import numpy as np
import pytest
import torch

import sparse_attention_indexer_csa_gb300 as csa
from oracle import csa_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    csa.load()


def _case(kind, rows, W, rng):
    if kind == "normal":
        x = rng.standard_normal((rows, W)).astype(np.float32)
    elif kind == "ties":
        x = rng.integers(-3, 4, size=(rows, W)).astype(np.float32)
    elif kind == "few_values":
        x = (rng.integers(0, 2, size=(rows, W)) * 0.5).astype(np.float32)
    elif kind == "equal":
        x = np.full((rows, W), 1.25, dtype=np.float32)
    elif kind == "zeros":
        x = np.where(rng.random((rows, W)) < 0.5, 0.0, -0.0).astype(np.float32)
        x[:, ::7] = rng.standard_normal(x[:, ::7].shape).astype(np.float32)
    elif kind == "huge":
        x = np.clip(rng.standard_normal((rows, W)) * 3e38, -3.4e38, 3.4e38).astype(np.float32)
    elif kind == "denormal":
        x = (rng.standard_normal((rows, W)) * 1e-40).astype(np.float32)
    elif kind == "offset":  # values far from zero relative to their spread
        x = (1000.0 + 1e-3 * rng.standard_normal((rows, W))).astype(np.float32)
    elif kind == "relu_like":  # most entries exactly zero, a few positive
        x = np.maximum(rng.standard_normal((rows, W)) - 1.5, 0).astype(np.float32)
    else:
        raise ValueError(kind)
    mask = rng.random((rows, W)) < 0.25
    x[mask] = -np.inf
    x[0, :] = -np.inf          # an empty row
    if rows > 1:
        x[1, 3:] = -np.inf     # a row with 3 or fewer visible entries
    return x


KINDS = ["normal", "ties", "few_values", "equal", "zeros", "huge", "denormal", "offset", "relu_like"]


# W > 16384 runs on clusters of four CTAs per row: an odd W (scalar staging,
# ragged last segment), the longest row, top_k above one CTA's segment, k = 1
@pytest.mark.parametrize("W,k", [(1000, 300), (4096, 2048), (300, 1), (32768, 2048), (257, 400), (9000, 700),
                                 (20001, 3000), (49152, 4096), (16385, 9000), (32768, 1)])
@pytest.mark.parametrize("kind", KINDS)
def test_topk_kernel_matches_oracle_selector(kind, W, k):
    rng = np.random.default_rng(abs(hash((kind, W, k))) % 2**32)
    rows = 6 if W > 8192 else 24
    x = _case(kind, rows, W, rng)
    g = torch.from_numpy(x).reshape(2, rows // 2, W).cuda()
    idx = csa.index_topk(g, k).cpu().numpy()
    torch.cuda.synchronize()
    assert csa.device_status() == csa.CSA_OK
    ref = O.select_topk(x.astype(np.float64), k).reshape(2, rows // 2, k)
    assert np.array_equal(idx, ref)
