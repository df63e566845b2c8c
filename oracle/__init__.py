"""CPU oracle (test infrastructure only; see ``oracle/csa_oracle.py``)."""
from .csa_oracle import (brute_force_scores, causal_threshold, index_scores,  # noqa: F401
                         index_topk, scale_value, select_topk, visibility,
                         visible_counts)
