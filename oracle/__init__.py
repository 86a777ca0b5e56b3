"""CPU oracle of the DFlash draft cycle — test infrastructure only.

Imported by tests/, the package smoke check and the benchmark's CPU-baseline
leg; never by the product path.  See dflash_oracle.py for what it computes and
which passages of the DFlash pages each function follows.
"""
from .dflash_oracle import *  # noqa: F401,F403
from .dflash_oracle import (RequestCache, attention_block, attention_masked, dflash_mask, draft_cycle,
                            draft_forward, expected_accept_len, fuse_context, inject_context, inject_kv,
                            linear, lm_head_argmax, rms_norm, rope, silu, store, verify_greedy, weights_to_host,
                            weights_to_numpy)
