"""The one-plane bf16 context cache (dflash_config.kv_bf16 = 1: every cached
K/V value rounded to one bf16, the storage paper §7.3 counts) against the
oracle over consecutive cycles.

Bars: logits within the 2e-2 contract bar of the exact float64 oracle, and
within a 5e-3 regression bar of the same oracle with its cached K/V rounded
to bf16 (storage class "kv"), which is the computation the GPU performs (the
two round fp32-level and float64 values, so boundary cases land one bf16 step
apart; see parity_util); drafts
identical to both wherever the oracle's top-2 margin exceeds 1e-2; the cache
within the bf16 rounding of the exact values (2^-8 relative) and, element by
element, equal to the rounded oracle cache except where the exact value lies
within fp32 rounding of a bf16 rounding boundary (then one bf16 step apart).

Paths: the persistent cycle launch (one key tile per attention chunk, and
chunks that hold context tiles followed by the block tile), the multi-kernel
split-KV attention, head size 64, the input-fusion ablation."""
import numpy as np
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_4B, QWEN3_8B, TINY, make_features, make_tokens, replace
from parity_util import OracleSide, compare_cache, features_for, gpu_inject, make_gpu, synthetic_target, tol

pytestmark = pytest.mark.gpu


def _kv(cfg):
    return replace(cfg, name=cfg.name + "-kv-bf16", dtype="bf16", kv_bf16=True)


def _check_cache_elements(g, orc):
    """Every cached value is a bf16 equal to the rounded oracle's, or one bf16
    step from it where the operands' fp32-level error decides the last bit
    (rare); values near zero may differ by that error, relative to the slab's
    largest value, instead."""
    K, V = g.cache.k().cpu().numpy(), g.cache.v().cpu().numpy()
    lens = g.cache.ctx_len().cpu().numpy()
    total = off = 0
    for b, oc in enumerate(orc.stored):
        c = int(lens[b])
        for l in range(len(oc.k)):
            for gpu, ref in ((K[b, l, :, :c, :], oc.k[l]), (V[b, l, :, :c, :], oc.v[l])):
                ref = np.transpose(ref, (1, 0, 2))
                gpu = gpu.astype(np.float64)
                np.testing.assert_array_equal(gpu, oracle.store(gpu, "bf16"))      # one bf16 per value
                d = gpu != ref
                total += gpu.size
                off += int(d.sum())
                if d.any():   # one bf16 step at most
                    step = np.maximum(np.abs(ref[d]) * 2.0 ** -7, 1e-4 * np.max(np.abs(ref)))
                    assert np.all(np.abs(gpu[d] - ref[d]) <= step), "cached value more than one bf16 step off"
    assert off <= max(4, total // 50), f"{off} of {total} cached values differ from the rounded oracle"
    return off, total


def _cycles(cfg, ctx, block, seed, cycles=3, p=0.8):
    """Set-up injection of ctx[b] tokens per request, then `cycles` draft
    cycles (dflash_draft_cycle: inject the previous cycle's accepted tokens,
    draft), each checked against both oracles; verification bit-exact."""
    import block_diffusion_drafter_dflash_gb300 as df
    B = len(ctx)
    g = make_gpu(cfg, seed=seed, batch=B, capacity=max(ctx) + (cycles + 2) * block, block=block,
                 max_rows=max(sum(ctx), B * block))
    feats = features_for(cfg, ctx, seed=seed + 1)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in range(B):
        orc.inject(b, feats[b].cpu())
    del feats
    compare_cache(g, orc.exact, tol(cfg))
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
    off, total = _check_cache_elements(g, orc)
    print(cfg.name, B, block, f"cache values one step off: {off}/{total}", stats)
    return g, orc


def test_kv_bf16_tiny_head_dim_64_persistent():
    _cycles(_kv(TINY), ctx=[64, 37], block=4, seed=700)


def test_kv_bf16_tiny_head_dim_64_multi_kernel():
    # 2 x 16 rows: the multi-kernel injection and split-KV attention
    _cycles(_kv(TINY), ctx=[150, 64], block=16, seed=705)


def test_kv_bf16_4b_bs1_chunks_with_context_and_block_tiles():
    # 4096 + injected tokens = 33 key tiles over 19 chunks a kv head: chunks of
    # two tiles, the last of them a context tile followed by the block tile
    _cycles(_kv(QWEN3_4B), ctx=[4096], block=16, seed=710)


def test_kv_bf16_4b_ragged_multi_kernel():
    _cycles(_kv(QWEN3_4B), ctx=[300, 1000, 77], block=8, seed=715, cycles=2)


def test_kv_bf16_8b_bs1():
    _cycles(_kv(QWEN3_8B), ctx=[2048], block=16, seed=720, cycles=2)


def test_kv_bf16_input_fusion_tiny():
    cfg = replace(_kv(TINY), name="tiny-input-fusion-kv-bf16", input_fusion=True)
    _cycles(cfg, ctx=[64, 40], block=4, seed=730, cycles=2)
