"""The one-bf16 LM-head input (dflash_config.head_bf16 = 1: the final normed
hidden state enters the LM head as one bf16 rounded to nearest) against the
oracle over consecutive cycles.

Bars: logits within the 2e-2 contract bar of the exact float64 oracle and
within the 1e-3 regression bar of the oracle with its final hidden state
rounded to bf16 (storage class "h": the computation the GPU performs); drafts
identical to both wherever the oracle's top-2 margin exceeds 1e-2;
verification bit-exact.

Paths: head_bf16 models run the multi-kernel path at every batch: the split-K
tcgen05 GEMM with one operand plane (small batches) and the dense persistent
GEMM with 256-row one-plane token tiles (batch 32)."""
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_4B, QWEN3_8B, TINY, make_features, make_tokens, replace
from parity_util import OracleSide, compare_cache, features_for, gpu_inject, make_gpu, synthetic_target, tol

pytestmark = pytest.mark.gpu


def _head(cfg):
    return replace(cfg, name=cfg.name + "-head-bf16", dtype="bf16", head_bf16=True)


def _cycles(cfg, ctx, block, seed, cycles=2, p=0.8, check=None):
    """Set-up injection, then `cycles` cycles (dflash_draft_cycle); requests in
    `check` (all by default) compared with both oracles every cycle."""
    import block_diffusion_drafter_dflash_gb300 as df
    B = len(ctx)
    check = list(range(B)) if check is None else check
    g = make_gpu(cfg, seed=seed, batch=B, capacity=max(ctx) + (cycles + 2) * block, block=block,
                 max_rows=max(sum(ctx), B * block))
    feats = features_for(cfg, ctx, seed=seed + 1)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in check:
        orc.inject(b, feats[b].cpu())
    del feats
    anchors = make_tokens(cfg, B, seed=seed + 2, device="cuda")
    tau = torch.full((B,), 3, dtype=torch.int32, device="cuda")
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
        starts = [sum(th[:b]) for b in range(B)]
        for b in check:
            orc.inject(b, new[starts[b]:starts[b] + th[b]].cpu())
        an = anchors.cpu().numpy()
        for b in check:
            stats.append(orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy()))
        y = synthetic_target(cfg, drafts.cpu(), [p] * B, seed=seed + 20 + c).cuda()
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        dh, yh = drafts.cpu().numpy(), y.cpu().numpy()
        tl = tau.cpu().tolist()
        for b in range(B):
            assert (tl[b], out[b].cpu().tolist(), int(nxt[b])) == oracle.verify_greedy(dh[b], yh[b])
        anchors = nxt.clone()
    if check == list(range(B)):
        compare_cache(g, orc.exact, tol(cfg))
    assert df.dflash_get_status(g.model) == 0
    print(cfg.name, B, block, stats)
    return stats


def test_head_bf16_tiny_head_dim_64():
    _cycles(_head(TINY), ctx=[64, 40], block=4, seed=800, cycles=3)


def test_head_bf16_4b_batch_1_takes_the_multi_kernel_path():
    _cycles(_head(QWEN3_4B), ctx=[700], block=16, seed=810)


def test_head_bf16_4b_ragged_batch_4():
    _cycles(_head(QWEN3_4B), ctx=[300, 1000, 77, 512], block=10, seed=815)


def test_head_bf16_8b_batch_32_sampled_requests():
    # 480 mask rows: the LM head runs the dense GEMM with 256-row one-plane tiles
    ctx = [160 + 37 * b for b in range(32)]
    _cycles(_head(QWEN3_8B), ctx=ctx, block=16, seed=820, cycles=1, check=[0, 31])


def test_head_bf16_with_the_one_plane_cache_4b_batch_4():
    # both one-bf16 options at once (the oracle rounds the kv and h classes)
    cfg = replace(_head(QWEN3_4B), name="qwen3-4b-shaped-head-kv-bf16", kv_bf16=True)
    _cycles(cfg, ctx=[300, 1000, 77, 512], block=10, seed=830)
