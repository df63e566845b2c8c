"""CPU oracle (test infrastructure only; see ``oracle/csa_oracle.py``)."""
from .csa_oracle import (brute_force_scores, causal_threshold, gather_selected, index_scores,  # noqa: F401
                         index_scores_vjp, index_topk, scale_value, select_topk, visibility,
                         visible_counts)
