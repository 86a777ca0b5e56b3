"""dflash_draft_cycle — injection of the committed tokens' features and the
drafter pass in one call, one persistent launch when both fit it — against
the float64 oracle over consecutive cycles (the injected counts come from the
verification output on the device): logits within 2e-2 and the 1e-3
regression bar, drafts identical wherever the oracle's top-2 margin exceeds
1e-2, the cache within the bars, verification bit-exact.  Also the fallback
(calls that do not fit one launch run the two calls in turn) and a cycle with
nothing to inject."""
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_4B, QWEN3_8B, TINY, make_features, make_tokens, replace
from parity_util import OracleSide, compare_cache, features_for, gpu_inject, make_gpu, synthetic_target, tol

pytestmark = pytest.mark.gpu


def _cycles(cfg, B, ctx, block, seed, cycles=3, p=0.8):
    import block_diffusion_drafter_dflash_gb300 as df
    g = make_gpu(cfg, seed=seed, batch=B, capacity=ctx + (cycles + 2) * block, block=block,
                 max_rows=max(B * ctx, B * block))
    feats = features_for(cfg, [ctx] * B, seed=seed + 1)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in range(B):
        orc.inject(b, feats[b].cpu())
    del feats
    anchors = make_tokens(cfg, B, seed=seed + 2, device="cuda")
    tau = torch.full((B,), 3, dtype=torch.int32, device="cuda")    # the previous cycle kept 3 tokens each
    out = torch.empty((B, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    rows = B * block
    stats = []
    for c in range(cycles):
        new = make_features(cfg, rows, seed=seed + 10 + c, device="cuda")
        th = tau.cpu().tolist()
        drafts = torch.full((B, block - 1), -7, dtype=torch.int32, device="cuda")
        logits = torch.empty((B, block - 1, cfg.vocab), dtype=torch.float32, device="cuda")
        df.dflash_draft_cycle(g.model, g.cache, new, tau, anchors, block, drafts, logits, max_rows=rows, workspace=g.ws)
        torch.cuda.synchronize()
        start = 0
        for b in range(B):
            orc.inject(b, new[start:start + th[b]].cpu())
            start += th[b]
        an = anchors.cpu().numpy()
        for b in range(B):
            stats.append(orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy()))
        compare_cache(g, orc.exact, tol(cfg))
        y = synthetic_target(cfg, drafts.cpu(), [p] * B, seed=seed + 20 + c).cuda()
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        dh, yh = drafts.cpu().numpy(), y.cpu().numpy()
        tl = tau.cpu().tolist()
        for b in range(B):
            assert (tl[b], out[b].cpu().tolist(), int(nxt[b])) == oracle.verify_greedy(dh[b], yh[b])
        anchors = nxt.clone()
    assert df.dflash_get_status(g.model) == 0
    print(cfg.name, B, block, stats)
    return g


def _stage_launches(g, fn):
    import block_diffusion_drafter_dflash_gb300 as df
    df.dflash_profile_start(g.model, 64)
    fn()
    return df.dflash_profile_stop(g.model)


def test_fused_cycle_8b_bs1():
    g = _cycles(QWEN3_8B, B=1, ctx=2048, block=16, seed=600)
    import block_diffusion_drafter_dflash_gb300 as df
    # the cycle is one persistent launch (plus its two prologue kernels)
    new = make_features(QWEN3_8B, 16, seed=690, device="cuda")
    n = torch.tensor([4], dtype=torch.int32, device="cuda")
    a = make_tokens(QWEN3_8B, 1, seed=691, device="cuda")
    d = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    prof = _stage_launches(g, lambda: df.dflash_draft_cycle(g.model, g.cache, new, n, a, 16, d, None, max_rows=16,
                                                            workspace=g.ws))
    assert prof["cycle_persist"][1] == 1 and prof["draft_persist"][1] == 0 and prof["inject_persist"][1] == 0


def test_fused_cycle_4b_two_requests_block_8():
    _cycles(QWEN3_4B, B=2, ctx=512, block=8, seed=610)


def test_fused_cycle_tiny_bf16_head_dim_64():
    _cycles(replace(TINY, name="tiny-bf16", dtype="bf16"), B=2, ctx=64, block=4, seed=620)


def test_cycle_that_does_not_fit_one_launch_runs_both_calls():
    # 2 x 16 rows: the multi-kernel path for both the injection and the drafter
    _cycles(QWEN3_4B, B=2, ctx=256, block=16, seed=630, cycles=2)


def test_cycle_without_injection_drafts_only():
    import block_diffusion_drafter_dflash_gb300 as df
    cfg = QWEN3_4B
    g = make_gpu(cfg, seed=640, batch=1, capacity=256, block=16, max_rows=128)
    feats = features_for(cfg, [128], seed=641)
    gpu_inject(g, feats)
    a = make_tokens(cfg, 1, seed=642, device="cuda")
    d1 = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    d2 = torch.empty((1, 15), dtype=torch.int32, device="cuda")
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    df.dflash_draft_cycle(g.model, g.cache, feats[0][:1].contiguous(), zero, a, 16, d1, None, max_rows=0,
                          workspace=g.ws)
    df.dflash_draft_block(g.model, g.cache, a, 16, d2, None, g.ws)
    torch.cuda.synchronize()
    assert torch.equal(d1, d2)
    assert g.cache.ctx_len().cpu().tolist() == [128]
