"""Device-side failure detection without a GPU fault: a bounded wait that
nothing completes gives up after its cycle budget, records DFLASH_ERR_TIMEOUT
in the model's status word and returns.  The status then clears, and the same
context runs a draft cycle that still matches the oracle."""
import time

import pytest
import torch

import oracle
from dflash_inputs import TINY, make_tokens, replace
from parity_util import OracleSide, features_for, gpu_draft, gpu_inject, make_gpu

pytestmark = pytest.mark.gpu

DFLASH_ERR_TIMEOUT = -5


def test_bounded_wait_runs_out_sets_timeout_and_the_context_stays_usable():
    import block_diffusion_drafter_dflash_gb300 as df
    cfg = replace(TINY, name="tiny-bf16", dtype="bf16")
    g = make_gpu(cfg, seed=5, batch=1, capacity=64, block=4, max_rows=32)
    df.dflash_clear_status(g.model)
    assert df.dflash_get_status(g.model) == 0
    t0 = time.perf_counter()
    df.dflash_selftest_wait_timeout(g.model, 2_000_000)   # about a millisecond of SM clock
    assert df.dflash_get_status(g.model) == DFLASH_ERR_TIMEOUT
    assert time.perf_counter() - t0 < 10.0
    df.dflash_clear_status(g.model)
    assert df.dflash_get_status(g.model) == 0

    feats = features_for(cfg, [32], seed=6)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    orc.inject(0, feats[0].cpu())
    anchors = make_tokens(cfg, 1, seed=7, device="cuda")
    drafts, logits = gpu_draft(g, anchors, 4)
    torch.cuda.synchronize()
    orc.check_request(0, int(anchors[0].item()), 4, logits[0].cpu().numpy(), drafts[0].cpu().numpy())
    assert df.dflash_get_status(g.model) == 0


def test_selftest_rejects_budgets_outside_its_range():
    import block_diffusion_drafter_dflash_gb300 as df
    g = make_gpu(TINY, seed=5, batch=1, capacity=16, block=4, max_rows=16)
    for bad in (0, -1, 5_000_000_000):
        with pytest.raises(df.DFlashError):
            df.dflash_selftest_wait_timeout(g.model, bad)
    assert df.dflash_get_status(g.model) == 0
