"""GB300 (sm_103a) CSA indexer: per-row top-k selection of compressed KV
entries by the head-reduced score  sum_h w[b,s,h] * ReLU(scale * q.k).

The compute lives in ``libcsa_index.so`` (hand-written CUDA behind the C ABI
of ``include/csa_index.h``); this package is its build script and a thin
ctypes binding.
"""
from .abi import (CSA_BF16, CSA_ERR_CUDA, CSA_Q_HEAD_MAJOR, CSA_Q_SEQ_MAJOR, CSA_ERR_DEVICE, CSA_ERR_INVALID_ARG,  # noqa: F401
                  CSA_ERR_TIMEOUT, CSA_ERR_UNSUPPORTED, CSA_F32, CSA_OK, CsaError, Problem,
                  device_status, fused_host_bytes, index_backward, index_decode, index_gather, index_fused,
                  index_fused_host, index_fused_host_raw, index_fused_raw, index_score,
                  index_score_raw, index_topk, index_topk_raw, load, make_problem,
                  selftest_timeout, workspace_size)
