"""Qwen3-8B-shaped bf16 drafter (D=4096, 5 layers, 32 q / 8 kv heads of 128,
SwiGLU 12288, W_c 20480->4096, vocab 151936, block 16) vs the oracle at full
size: logits within 2e-2 relative (per row, against the row's largest
magnitude; 1e-3 regression bar), drafts identical wherever the oracle's top-2
margin exceeds 1e-2, injected K/V within 2e-2, verification bit-exact.
Batch 32 (ragged contexts 512..8192) and the 4 x 32768 long-context case are
checked on sampled requests: requests are independent, so the oracle computes
them one by one.  The long-context case runs 16 consecutive cycles, each
appending the accepted tokens' features to every request's cache.  Drafting
without a logits buffer (the call a serving loop makes) must give the same
drafts as drafting with one."""
import numpy as np
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_8B, make_features, make_tokens, workloads
from parity_util import BF16_TOL, OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, \
    synthetic_target

pytestmark = pytest.mark.gpu


def _check_requests(orc, g, anchors, block, which, drafts=None, logits=None):
    if drafts is None:
        drafts, logits = gpu_draft(g, anchors, block)
        torch.cuda.synchronize()
    an = anchors.cpu().numpy()
    stats = [orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy()) for b in which]
    print(stats)
    return drafts, logits, stats


def test_8b_bs1_two_cycles():
    wl = workloads()["8b_bs1"]
    cfg, block, ctx = wl.cfg, wl.block, wl.ctx[0]
    g = make_gpu(cfg, seed=wl.seed, batch=1, capacity=ctx + 4 * block, block=block, max_rows=ctx)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    feats = features_for(cfg, [ctx], seed=wl.seed + 1)
    gpu_inject(g, feats)
    orc.inject(0, feats[0].cpu())
    compare_cache(g, orc.exact, BF16_TOL)
    anchors = make_tokens(cfg, 1, seed=wl.seed + 2, device="cuda")
    drafts, _, _ = _check_requests(orc, g, anchors, block, [0])
    nolog, _ = gpu_draft(g, anchors, block, want_logits=False)     # the persistent launch without logits
    assert torch.equal(nolog, drafts)

    import block_diffusion_drafter_dflash_gb300 as df
    y = synthetic_target(cfg, drafts.cpu(), wl.accept_p, seed=wl.seed + 3).cuda()
    tau = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    df.dflash_verify_greedy(drafts, y, tau, out, nxt)
    t_o, o_o, n_o = oracle.verify_greedy(drafts.cpu().numpy()[0], y.cpu().numpy()[0])
    assert int(tau.item()) == t_o and out.cpu().tolist()[0] == o_o and int(nxt.item()) == n_o
    new = make_features(cfg, block, seed=wl.seed + 4, device="cuda")
    gpu_inject(g, [new], max_rows=block, host_counts=False, n_new_dev=tau)
    orc.inject(0, new[:t_o].cpu())
    compare_cache(g, orc.exact, BF16_TOL)
    _check_requests(orc, g, nxt, block, [0])
    assert df.dflash_get_status(g.model) == 0


def test_8b_bs1_mask_rows_draft_distinct_tokens():
    """With weights N(0, 0.03) (instead of 0.02) the 15 mask rows of a block
    draft mostly different tokens (13 of 15 distinct for the oracle on a
    CPU-drawn instance at context 128), so argmax parity checks a separate
    decision on every row rather than one token repeated."""
    cfg, block, ctx = QWEN3_8B, 16, 128
    g = make_gpu(cfg, seed=1001, batch=1, capacity=ctx + 2 * block, block=block, max_rows=ctx, std=0.03)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    feats = features_for(cfg, [ctx], seed=1002)
    gpu_inject(g, feats)
    orc.inject(0, feats[0].cpu())
    anchors = make_tokens(cfg, 1, seed=1003, device="cuda")
    drafts, _, stats = _check_requests(orc, g, anchors, block, [0])
    assert stats[0]["distinct_drafts"] >= 6, stats
    assert stats[0]["checked"] >= 10, stats
    nolog, _ = gpu_draft(g, anchors, block, want_logits=False)
    assert torch.equal(nolog, drafts)


def test_8b_bs32_ragged_sampled_requests():
    wl = workloads()["8b_bs32"]
    cfg, block, B = wl.cfg, wl.block, wl.batch
    cap = max(wl.ctx) + 2 * block
    g = make_gpu(cfg, seed=wl.seed, batch=B, capacity=cap, block=block, max_rows=sum(wl.ctx))
    feats = features_for(cfg, wl.ctx, seed=wl.seed + 1)
    gpu_inject(g, feats)
    anchors = make_tokens(cfg, B, seed=wl.seed + 2, device="cuda")
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    order = np.argsort(wl.ctx)
    which = [int(order[0]), int(order[len(order) // 2])]          # shortest and a median-length request
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in which:
        orc.inject(b, feats[b].cpu())
    del feats
    lens = g.cache.ctx_len().cpu().numpy()
    assert list(lens) == wl.ctx
    _check_requests(orc, g, anchors, block, which, drafts, logits)
    nolog, _ = gpu_draft(g, anchors, block, want_logits=False)     # the many-row path without logits
    assert torch.equal(nolog, drafts)


def test_8b_long_context_sixteen_cycles():
    """4 requests of 32768 injected context tokens, then 16 whole cycles:
    draft, synthetic target, verify, and inject the tau committed tokens'
    features (counts read by the device from the verification output).
    Verification is checked bit-exact on every cycle for every request; the
    last request's drafts and logits against the oracle on the first and the
    last cycle, and its cache at the end."""
    import block_diffusion_drafter_dflash_gb300 as df
    wl = workloads()["8b_long"]
    cfg, block, B, cycles = wl.cfg, wl.block, wl.batch, wl.cycles
    ctx = wl.ctx[0]
    g = make_gpu(cfg, seed=wl.seed, batch=B, capacity=ctx + (cycles + 2) * block, block=block, max_rows=B * ctx)
    feats = features_for(cfg, wl.ctx, seed=wl.seed + 1)
    gpu_inject(g, feats)
    anchors = make_tokens(cfg, B, seed=wl.seed + 2, device="cuda")
    sb = B - 1
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    f = feats[sb].cpu()
    del feats
    for s0 in range(0, ctx, 4096):          # incremental injection equals one-shot injection (oracle pin)
        orc.inject(sb, f[s0:s0 + 4096])
    del f
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty((B, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    for c in range(cycles):
        check = c in (0, cycles - 1)
        drafts, logits = gpu_draft(g, anchors, block, want_logits=check)
        torch.cuda.synchronize()
        if check:
            _check_requests(orc, g, anchors, block, [sb], drafts, logits)
        y = synthetic_target(cfg, drafts.cpu(), wl.accept_p, seed=wl.seed + 10 + c).cuda()
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        dh, yh = drafts.cpu().numpy(), y.cpu().numpy()
        th, oh, nh = tau.cpu().tolist(), out.cpu().tolist(), nxt.cpu().tolist()
        for b in range(B):
            t_o, o_o, n_o = oracle.verify_greedy(dh[b], yh[b])
            assert (th[b], oh[b], nh[b]) == (t_o, o_o, n_o), (c, b)
        new = make_features(cfg, B * block, seed=wl.seed + 20 + c, device="cuda")
        gpu_inject(g, [new], max_rows=B * block, host_counts=False, n_new_dev=tau)
        first = sum(th[:sb])
        orc.inject(sb, new[first:first + th[sb]].cpu())
        anchors = nxt.clone()
    lens = g.cache.ctx_len().cpu().tolist()
    assert lens[sb] == orc.exact[sb].length and all(v > ctx for v in lens)
    compare_cache(g, [orc.exact[sb]], BF16_TOL, batch_index=sb)
    assert df.dflash_get_status(g.model) == 0
