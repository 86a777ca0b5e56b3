"""Qwen3-8B-shaped bf16 drafter (D=4096, 5 layers, 32 q / 8 kv heads of 128,
SwiGLU 12288, W_c 20480->4096, vocab 151936, block 16) vs the oracle at full
size: logits within 2e-2 relative (per row, against the row's largest
magnitude), drafts identical wherever the oracle's top-2 margin exceeds 1e-2,
injected K/V within 2e-2, verification bit-exact.  Batch 32 (ragged contexts
512..8192) and the 4 x 32768 long-context case are checked on sampled
requests: requests are independent, so the oracle computes them one by one."""
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


def test_8b_long_context_sampled_request():
    wl = workloads()["8b_long"]
    cfg, block, B = wl.cfg, wl.block, wl.batch
    ctx = wl.ctx[0]
    g = make_gpu(cfg, seed=wl.seed, batch=B, capacity=ctx + 2 * block, block=block, max_rows=B * ctx)
    feats = features_for(cfg, wl.ctx, seed=wl.seed + 1)
    gpu_inject(g, feats)
    anchors = make_tokens(cfg, B, seed=wl.seed + 2, device="cuda")
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    which = [B - 1]
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    f = feats[which[0]].cpu()
    del feats
    for s in range(0, ctx, 4096):          # incremental injection equals one-shot injection (oracle pin)
        orc.inject(which[0], f[s:s + 4096])
    _check_requests(orc, g, anchors, block, which, drafts, logits)
