"""Seeded synthetic inputs for scoring one prefetched subtree batch.

This package is the only code shared by the CPU oracle side and the CUDA
side.  It draws trees, cut indices, logits rows, sampled tokens and acceptance
uniforms; it computes no log-probability, suffix sum, acceptance ratio or walk.
"""

from .trees import (ChainTree, Layout, assemble_layout, bfs_tree, spine_tree,
                    example5_tree)
from .workload import (CONFIGS, Workload, draw_tokens, gen_logits, make_workload,
                       workload_config5)

__all__ = [
    "ChainTree", "Layout", "assemble_layout", "bfs_tree", "spine_tree",
    "example5_tree", "CONFIGS", "Workload", "draw_tokens", "gen_logits",
    "make_workload", "workload_config5",
]
