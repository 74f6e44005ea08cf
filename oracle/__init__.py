"""CPU oracle of the CSA / HCA path -- test infrastructure only (see csa_oracle)."""
from .csa_oracle import *  # noqa: F401,F403
from .csa_oracle import (bf16_to_f64, round_bf16, compress, n_visible, indexer_scores, topk,
                         window_rows, attend_one, csa_compress, csa_index_scores, csa_index_topk,
                         csa_attend, hca_attend, csa_layer_prefill)
