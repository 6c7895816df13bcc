"""fp64 CPU oracle for BA-Att selection and block-sparse attention.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the library.  Every function
here is pinned by ``tests/test_oracle_pins.py`` (see that file for the pins).
"""

from .ba_oracle import *  # noqa: F401,F403
from .ba_oracle import (SORT_NONE, SORT_K, SORT_Q, SORT_QK,  # noqa: F401
                        select_one, ba_select, sparse_attention, sparse_attention_one,
                        dense_attention, dense_attention_one, merge_lse, topk_blocks,
                        block_moments, block_logits, covariance_compensation,
                        compensated_logits, token_norms, norm_sort_permutation,
                        num_blocks, block_ranges, kappa_for_sparsity,
                        oracle_block_mass, deviation_bound, block_distribution)
