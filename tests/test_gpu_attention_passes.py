"""Split-KV attention when a kv head's query rows span more than one 64-row
pass (query heads per kv head x block > 64): a tiny drafter with 8 query heads
over 2 kv heads at blocks 17 and 32 (68 and 128 rows a group), ragged contexts,
against the oracle."""
import pytest

import oracle
from dflash_inputs import TINY, make_tokens, replace
from parity_util import OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("block", [17, 32])
def test_query_rows_of_a_kv_head_in_two_passes(dtype, block):
    import torch
    cfg = replace(TINY, name=f"tiny-{dtype}-g4", dtype=dtype, n_q_heads=8, n_kv_heads=2)
    ctxs = [0, 65, 130]
    B = len(ctxs)
    g = make_gpu(cfg, seed=8, batch=B, capacity=176, block=block, max_rows=sum(ctxs))
    orc = OracleSide(cfg, oracle.weights_to_numpy(g.weights), B)
    feats = features_for(cfg, ctxs, seed=9)
    gpu_inject(g, feats)
    for b in range(B):
        if ctxs[b]:
            orc.inject(b, feats[b].float().cpu().numpy())
    compare_cache(g, orc.exact, tol(cfg))
    anchors = make_tokens(cfg, B, seed=10, device="cuda")
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    an, lg, dr = anchors.cpu().numpy(), logits.cpu().numpy(), drafts.cpu().numpy()
    for b in range(B):
        orc.check_request(b, int(an[b]), block, lg[b], dr[b])
