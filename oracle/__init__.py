"""CPU oracle for paged chunk attention -- test infrastructure only.

Importable by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs; never by the library or its binding. See pkv_oracle.py.
"""
from .pkv_oracle import *  # noqa: F401,F403
from .pkv_oracle import (attention_backward, attention_block, attention_forward, chunk_recurrent_step,
                         chunk_local_selection, chunk_selection, full_causal_attention,
                         local_pages, logical_rows,
                         page_allowed_from_lists, page_representatives, query_page_means,
                         scatter_rows, select_pages, softmax_scale)
