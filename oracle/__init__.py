"""fp64 CPU oracle -- test infrastructure only (tests, smoke check, bench CPU baseline)."""
from .oracle import (block_attn, block_loop, build, confidence_unmask, generate_blocks,  # noqa: F401
                     hw_threads, kv_append, load, mamba_state_seed)
