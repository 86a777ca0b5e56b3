"""Whole draft cycle on the tiny fp32 drafter vs the oracle (1e-4 relative).

Tiny drafter: D=256, 2 layers, 4 q / 2 kv heads of 64, SwiGLU 768, vocab 1024,
block 4, context 64, batch 1, seed 0 — plus ragged batches, other block sizes,
an empty context, incremental injection from device-side counts and the
capacity guard."""
import numpy as np
import pytest
import torch

import oracle
from dflash_inputs import TINY, make_features, make_tokens, replace
from parity_util import (OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, synthetic_target,
                         tol)

pytestmark = pytest.mark.gpu


def _cycle_compare(orc, g, anchors, block):
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    an = anchors.cpu().numpy()
    lg, dr = logits.cpu().numpy(), drafts.cpu().numpy()
    for b in range(len(an)):
        orc.check_request(b, int(an[b]), block, lg[b], dr[b])
    return drafts


@pytest.mark.parametrize("cfg", [TINY, replace(TINY, name="tiny-bf16", dtype="bf16")], ids=["fp32", "bf16"])
def test_tiny_config_one_cycle_then_incremental_injection(cfg):
    block, ctx = 4, 64
    g = make_gpu(cfg, seed=0, batch=1, capacity=128, block=block, max_rows=64)
    orc = OracleSide(cfg, oracle.weights_to_numpy(g.weights), 1)
    feats = features_for(cfg, [ctx], seed=1)
    gpu_inject(g, feats)
    orc.inject(0, feats[0].float().cpu().numpy())
    compare_cache(g, orc.exact, tol(cfg))
    anchors = make_tokens(cfg, 1, seed=2, device="cuda")
    drafts = _cycle_compare(orc, g, anchors, block)

    # verify against a synthetic target, then inject the tau committed tokens
    # using the device-side accepted lengths (no host copy of the counts)
    import block_diffusion_drafter_dflash_gb300 as df
    y = synthetic_target(cfg, drafts.cpu(), [0.9], seed=3).cuda()
    tau = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    df.dflash_verify_greedy(drafts, y, tau, out, nxt)
    t_o, o_o, n_o = oracle.verify_greedy(drafts.cpu().numpy()[0], y.cpu().numpy()[0])
    assert int(tau.item()) == t_o and out.cpu().tolist()[0] == o_o and int(nxt.item()) == n_o
    new = make_features(cfg, block, seed=4, device="cuda")          # features of up to `block` committed tokens
    gpu_inject(g, [new], max_rows=block, host_counts=False, n_new_dev=tau)
    orc.inject(0, new[:t_o].float().cpu().numpy())
    compare_cache(g, orc.exact, tol(cfg))
    _cycle_compare(orc, g, nxt, block)
    import block_diffusion_drafter_dflash_gb300 as df2
    assert df2.dflash_get_status(g.model) == 0


TINY_BF16 = replace(TINY, name="tiny-bf16", dtype="bf16")


@pytest.mark.parametrize("cfg", [TINY, TINY_BF16], ids=["fp32", "bf16"])
@pytest.mark.parametrize("block", [1, 3, 17, 32])
@pytest.mark.parametrize("ctxs", [[0, 1, 65], [130]])
def test_tiny_ragged_batches_and_block_sizes(cfg, block, ctxs):
    B = len(ctxs)
    g = make_gpu(cfg, seed=5, batch=B, capacity=160, block=block, max_rows=max(1, sum(ctxs)))
    orc = OracleSide(cfg, oracle.weights_to_numpy(g.weights), B)
    feats = features_for(cfg, ctxs, seed=6)
    gpu_inject(g, feats)
    for b in range(B):
        if ctxs[b]:
            orc.inject(b, feats[b].float().cpu().numpy())
    compare_cache(g, orc.exact, tol(cfg))
    anchors = make_tokens(cfg, B, seed=7, device="cuda")
    _cycle_compare(orc, g, anchors, block)


def test_capacity_is_guarded_on_host_and_device():
    import block_diffusion_drafter_dflash_gb300 as df
    cfg = TINY
    g = make_gpu(cfg, seed=0, batch=2, capacity=10, block=4, max_rows=16)
    f = features_for(cfg, [8, 8], seed=1)
    with pytest.raises(df.DFlashError):
        gpu_inject(g, [f[0], torch.cat([f[1], f[1]])[:11]])          # 11 > capacity: refused on the host
    gpu_inject(g, f)                                                  # 8 + 8 fit
    n = torch.tensor([4, 1], dtype=torch.int32, device="cuda")
    gpu_inject(g, f, max_rows=16, host_counts=False, n_new_dev=n)     # request 0 would reach 12 > 10
    assert df.dflash_get_status(g.model) == -3
    lens = g.cache.ctx_len().cpu().tolist()
    assert lens == [10, 9]                                            # the rows that fit were kept
    df.dflash_clear_status(g.model)
    assert df.dflash_get_status(g.model) == 0
