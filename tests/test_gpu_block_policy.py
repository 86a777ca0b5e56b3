"""Block-size scheduling (paper §5.5.4) driving the GPU draft cycle.

The library's host policy picks each cycle's block size from the accepted
lengths of earlier cycles; the synthetic target agrees with every draft with
probability 0.95 for the first cycles and 0.1 after, so the policy moves from
large blocks to small ones.  Every cycle — whichever block size was chosen —
is checked against the float64 oracle (logits within 2e-2 and the 1e-3
regression bar, drafts identical wherever the oracle's top-2 margin exceeds
1e-2, verification bit-exact), and its accepted lengths feed the policy."""
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_4B, make_features, make_tokens
from parity_util import OracleSide, features_for, gpu_draft, gpu_inject, make_gpu, synthetic_target

pytestmark = pytest.mark.gpu


def test_policy_chosen_block_sizes_match_the_oracle():
    import block_diffusion_drafter_dflash_gb300 as df
    cfg, B, ctx, cycles = QWEN3_4B, 2, 1024, 12
    cands = [4, 8, 10, 16]
    pol = df.BlockPolicy(cands, cost_fixed_ms=0.7, cost_per_row_ms=0.02, decay=0.5, prior_accept=0.9,
                         prior_weight=2.0)
    g = make_gpu(cfg, seed=4321, batch=B, capacity=ctx + (cycles + 2) * 16, block=max(cands), max_rows=B * ctx)
    feats = features_for(cfg, [ctx] * B, seed=4322)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in range(B):
        orc.inject(b, feats[b].cpu())
    del feats
    anchors = make_tokens(cfg, B, seed=4323, device="cuda")
    tau = torch.empty(B, dtype=torch.int32, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    chosen = []
    for c in range(cycles):
        block, _ = pol.choose(B)
        chosen.append(block)
        drafts, logits = gpu_draft(g, anchors, block)
        torch.cuda.synchronize()
        an = anchors.cpu().numpy()
        for b in range(B):
            orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy())
        p = 0.95 if c < cycles // 2 else 0.1
        y = synthetic_target(cfg, drafts.cpu(), [p] * B, seed=4400 + c).cuda()
        out = torch.empty((B, block), dtype=torch.int32, device="cuda")
        df.dflash_verify_greedy(drafts, y, tau, out, nxt)
        th = tau.cpu().tolist()
        dh, yh = drafts.cpu().numpy(), y.cpu().numpy()
        for b in range(B):
            assert (th[b], out[b].cpu().tolist(), int(nxt[b])) == oracle.verify_greedy(dh[b], yh[b])
        pol.observe(block, th)
        new = make_features(cfg, B * block, seed=4500 + c, device="cuda")
        gpu_inject(g, [new], max_rows=B * block, host_counts=False, n_new_dev=tau)
        start = 0
        for b in range(B):
            orc.inject(b, new[start:start + th[b]].cpu())
            start += th[b]
        anchors = nxt.clone()
    print("block sizes chosen:", chosen)
    assert chosen[0] == 16 and chosen[-1] < 16           # the policy followed the acceptance
    assert len(set(chosen)) >= 2
    assert df.dflash_get_status(g.model) == 0
