"""fp64 CPU oracle of the CompKV decode step -- test infrastructure only.

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  It shares no code with the CUDA path.
"""
from .compkv_oracle import *  # noqa: F401,F403
from .compkv_oracle import (BLOCK, HeadState, Scores, StepResult, block_counts,  # noqa: F401
                            block_scores, block_summaries, boundary_gap, compkv_attend,
                            decode_head, dense_attention, forced_blocks, num_blocks,
                            select_blocks)
