"""Qwen3-4B-shaped bf16 drafter (D=2560, 5 layers, 32 q / 8 kv heads of 128,
SwiGLU 9728, W_c 12800->2560, vocab 151936, context 4096) vs the oracle.

The block-size x batch sweep (blocks 8/10/16 x batch 1/4/16, all nine points)
is checked on sampled requests (requests are independent, so the oracle
computes them one by one): calls of at most 16 token rows run as one
persistent launch, 32-64 rows the multi-kernel path, 128-256 rows the
many-row tensor-core GEMMs.  Consecutive cycles with incremental injection of
the tau committed tokens are checked cycle by cycle, and the workload's 64
cycles are run on the device and checked at the end.  Bars: logits within 2e-2
relative (per row, against the row's largest magnitude), drafts identical
wherever the oracle's top-2 margin exceeds 1e-2, the injected K/V within 2e-2,
verification bit-exact."""
import pytest
import torch

import oracle
from dflash_inputs import make_features, make_tokens, workloads
from parity_util import BF16_TOL, OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, \
    synthetic_target

pytestmark = pytest.mark.gpu


def _check(orc, g, anchors, block, which, drafts, logits):
    an = anchors.cpu().numpy()
    return [orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy()) for b in which]


@pytest.mark.parametrize("name", [f"4b_g{g}_b{b}" for g in (8, 10, 16) for b in (1, 4, 16)])
def test_4b_sweep_sampled_requests(name):
    wl = workloads()[name]
    cfg, block, B = wl.cfg, wl.block, wl.batch
    g = make_gpu(cfg, seed=wl.seed, batch=B, capacity=max(wl.ctx) + 2 * block, block=block, max_rows=sum(wl.ctx))
    feats = features_for(cfg, wl.ctx, seed=wl.seed + 1)
    gpu_inject(g, feats)
    anchors = make_tokens(cfg, B, seed=wl.seed + 2, device="cuda")
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    which = [0] if B == 1 else [0, B - 1]
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in which:
        orc.inject(b, feats[b].cpu())
    del feats
    assert g.cache.ctx_len().cpu().tolist() == wl.ctx
    print(_check(orc, g, anchors, block, which, drafts, logits))

    import block_diffusion_drafter_dflash_gb300 as df
    assert df.dflash_get_status(g.model) == 0


def test_4b_consecutive_cycles_with_incremental_injection():
    """Three whole cycles of one request: draft, synthetic target, verify,
    then inject the tau committed tokens (counts read by the device from the
    verification output) before the next draft."""
    import block_diffusion_drafter_dflash_gb300 as df
    wl = workloads()["4b_g16_b1"]
    cfg, block, ctx = wl.cfg, wl.block, wl.ctx[0]
    cycles = 3
    g = make_gpu(cfg, seed=wl.seed, batch=1, capacity=ctx + (cycles + 2) * block, block=block, max_rows=ctx)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    feats = features_for(cfg, [ctx], seed=wl.seed + 1)
    gpu_inject(g, feats)
    orc.inject(0, feats[0].cpu())
    del feats
    anchor = make_tokens(cfg, 1, seed=wl.seed + 2, device="cuda")
    tau = torch.empty(1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    for c in range(cycles):
        drafts, logits = gpu_draft(g, anchor, block)
        torch.cuda.synchronize()
        print(_check(orc, g, anchor, block, [0], drafts, logits))
        y = synthetic_target(cfg, drafts.cpu(), wl.accept_p, seed=wl.seed + 10 + c).cuda()
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        t_o, o_o, n_o = oracle.verify_greedy(drafts.cpu().numpy()[0], y.cpu().numpy()[0])
        assert int(tau.item()) == t_o and out.cpu().tolist()[0] == o_o and int(nxt.item()) == n_o
        new = make_features(cfg, block, seed=wl.seed + 20 + c, device="cuda")
        gpu_inject(g, [new], max_rows=block, host_counts=False, n_new_dev=tau)
        orc.inject(0, new[:t_o].cpu())
        compare_cache(g, orc.exact, BF16_TOL)
        anchor = nxt.clone()
    assert g.cache.ctx_len().cpu().tolist() == [orc.exact[0].length]
    assert df.dflash_get_status(g.model) == 0


def test_4b_sixty_four_cycles_then_the_oracle():
    """The workload's 64 cycles (one request, block 16): each cycle drafts,
    verifies against the synthetic target and injects the tau committed
    tokens' features (the count read by the device from the verification
    output, dflash_draft_cycle); the host keeps the committed rows.  After the
    64th cycle the cache (4096 + sum of tau positions) and the next draft are
    compared with the oracle given the same committed rows."""
    import block_diffusion_drafter_dflash_gb300 as df
    wl = workloads()["4b_g16_b1"]
    cfg, block, ctx = wl.cfg, wl.block, wl.ctx[0]
    cycles = 64
    g = make_gpu(cfg, seed=wl.seed + 5, batch=1, capacity=ctx + (cycles + 2) * block, block=block,
                 max_rows=ctx)
    feats = features_for(cfg, [ctx], seed=wl.seed + 6)
    gpu_inject(g, feats)
    committed = [feats[0].cpu()]
    del feats
    anchor = make_tokens(cfg, 1, seed=wl.seed + 7, device="cuda")
    tau = torch.full((1,), 1, dtype=torch.int32, device="cuda")
    out = torch.empty((1, block), dtype=torch.int32, device="cuda")
    nxt = torch.empty(1, dtype=torch.int32, device="cuda")
    drafts = torch.empty((1, block - 1), dtype=torch.int32, device="cuda")
    total = 0
    for c in range(cycles):
        new = make_features(cfg, block, seed=wl.seed + 100 + c, device="cuda")
        t_prev = int(tau.item())
        df.dflash_draft_cycle(g.model, g.cache, new, tau, anchor, block, drafts, None, max_rows=block,
                              workspace=g.ws)
        committed.append(new[:t_prev].cpu())
        total += t_prev
        y = synthetic_target(cfg, drafts.cpu(), wl.accept_p, seed=wl.seed + 300 + c).cuda()
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        anchor = nxt.clone()
    torch.cuda.synchronize()
    assert g.cache.ctx_len().cpu().tolist() == [ctx + total]
    assert df.dflash_get_status(g.model) == 0
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    orc.inject(0, torch.cat(committed, 0))
    compare_cache(g, orc.exact, BF16_TOL)
    d, lg = gpu_draft(g, anchor, block)
    torch.cuda.synchronize()
    print(total, _check(orc, g, anchor, block, [0], d, lg))

