"""fp64 CPU oracle -- test infrastructure only (tests, smoke check, bench CPU baseline)."""
from .oracle import (adaln_single, bf16_decode, block_attn, block_loop, build,  # noqa: F401
                     confidence_unmask, generate_blocks, hw_threads, kv_append, load, lse_combine,
                     mamba_state_seed)
