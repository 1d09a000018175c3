"""fp64 CPU oracle -- test infrastructure only (tests, smoke check, bench CPU baseline)."""
from .oracle import (block_attn, block_loop, build, confidence_unmask, hw_threads, kv_append,  # noqa: F401
                     load)
