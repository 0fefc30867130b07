"""fp64 CPU oracle for the DDTree tree-verify step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. It shares no code with the CUDA
path in ``tree_speculative_decoding_ddtree_gb300``.
"""
from .ddtree_oracle import *  # noqa: F401,F403
from .ddtree_oracle import (Tree, Accept, draft_topk, build_tree, child_lists,
                            visibility_matrix, visibility_words, unpack_vis,
                            tree_verify_attention, attention_row, argmax_lowest,
                            accept_greedy, accept_sample, philox4x32_10,
                            philox4x32_10_np, draw_words, to_uniform, bf16_to_f64,
                            children, gather_context, commit_kv,
                            accept_sample_ratio)
