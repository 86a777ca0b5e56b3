"""Architectural variants of the drafter (paper §5.5.2 number of draft layers,
§5.5.3 number of target hidden features; QK-norm, a Qwen3 option the pages do
not use) against the float64 oracle: logits within the contract bar and the
regression bar, drafts identical wherever the oracle's top-2 margin exceeds
1e-2, injected K/V within the bars.

* QK-norm: tiny drafter in fp32 and bf16, 4B-shaped bf16 at batch 1 and 3
  (QK-norm models take the multi-kernel path; the per-head norm and RoPE of
  queries, block keys and injected context keys run after the projections).
* 8 draft layers (the paper's Qwen3-Coder drafter depth), 8B-shaped: batch 1
  runs the persistent one-launch path (6 x 8 + 1 phases), batch 2 the
  multi-kernel path.
* 3 target features instead of 5 (W_c 12288 -> 4096), 8B-shaped, both paths.
* Input fusion instead of per-layer KV injection (paper §5.5.5): the injected
  context rows run through every draft layer (causal among the context) and
  each layer caches its own context K/V; tiny drafter in fp32 and bf16 and
  4B-shaped bf16, a setup injection and then per-cycle injections."""
import pytest
import torch

import oracle
from dflash_inputs import QWEN3_4B, QWEN3_8B, TINY, make_features, make_tokens, replace
from parity_util import OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, tol

pytestmark = pytest.mark.gpu


def _cycle(cfg, B, ctx, block, seed, cycles=2):
    """Inject ctx tokens per request, then `cycles` cycles of draft + inject
    the next block's tokens; every draft and the cache checked."""
    import block_diffusion_drafter_dflash_gb300 as df
    g = make_gpu(cfg, seed=seed, batch=B, capacity=ctx + (cycles + 1) * block, block=block, max_rows=B * ctx)
    feats = features_for(cfg, [ctx] * B, seed=seed + 1)
    gpu_inject(g, feats)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), B)
    for b in range(B):
        orc.inject(b, feats[b].cpu())
    del feats
    compare_cache(g, orc.exact, tol(cfg))
    anchors = make_tokens(cfg, B, seed=seed + 2, device="cuda")
    stats = []
    for c in range(cycles):
        drafts, logits = gpu_draft(g, anchors, block)
        torch.cuda.synchronize()
        an = anchors.cpu().numpy()
        for b in range(B):
            stats.append(orc.check_request(b, int(an[b]), block, logits[b].cpu().numpy(), drafts[b].cpu().numpy()))
        n_new = [1 + (c + b) % block for b in range(B)]
        new = features_for(cfg, n_new, seed=seed + 10 + c)
        gpu_inject(g, new)
        for b in range(B):
            orc.inject(b, new[b].cpu())
        compare_cache(g, orc.exact, tol(cfg))
        anchors = make_tokens(cfg, B, seed=seed + 20 + c, device="cuda")
    assert df.dflash_get_status(g.model) == 0
    print(cfg.name, B, stats)
    return stats


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_qk_norm_tiny(dtype):
    cfg = replace(TINY, name=f"tiny-qknorm-{dtype}", dtype=dtype, qk_norm=True)
    _cycle(cfg, B=2, ctx=64, block=4, seed=500)


@pytest.mark.parametrize("B", [1, 3])
def test_qk_norm_4b_shaped(B):
    cfg = replace(QWEN3_4B, name="qwen3-4b-shaped-qknorm", qk_norm=True)
    _cycle(cfg, B=B, ctx=512, block=16, seed=510 + B)


@pytest.mark.parametrize("B", [1, 2])
def test_eight_layer_drafter_8b_shaped(B):
    cfg = replace(QWEN3_8B, name="qwen3-8b-shaped-8-layers", layers=8)
    _cycle(cfg, B=B, ctx=384, block=16, seed=520 + B, cycles=1)


@pytest.mark.parametrize("B", [1, 2])
def test_three_target_features_8b_shaped(B):
    cfg = replace(QWEN3_8B, name="qwen3-8b-shaped-3-features", n_target_feats=3)
    _cycle(cfg, B=B, ctx=384, block=16, seed=530 + B, cycles=1)


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_input_fusion_tiny(dtype):
    cfg = replace(TINY, name=f"tiny-input-fusion-{dtype}", dtype=dtype, input_fusion=True)
    _cycle(cfg, B=2, ctx=64, block=4, seed=540)


@pytest.mark.parametrize("B", [1, 3])
def test_input_fusion_4b_shaped(B):
    cfg = replace(QWEN3_4B, name="qwen3-4b-shaped-input-fusion", input_fusion=True)
    _cycle(cfg, B=B, ctx=256, block=16, seed=550 + B, cycles=2)
