"""The one-launch (persistent) path that serves bf16 calls of at most 16 token
rows, against the oracle: ragged batches with B * block <= 16 (including an
empty context and block 1), context injected through many persistent
injection calls of <= 16 rows each (so the persistent fusion and K/V
epilogues write the whole cache), and the multi-kernel path on the same
shapes with the persistent path switched off (DFLASH_PERSIST=0 at model
creation)."""
import contextlib
import os

import pytest
import torch

import oracle
from dflash_inputs import QWEN3_8B, TINY, make_tokens, replace, workloads
from parity_util import OracleSide, compare_cache, features_for, gpu_draft, gpu_inject, make_gpu, tol

pytestmark = pytest.mark.gpu

TINY_BF16 = replace(TINY, name="tiny-bf16", dtype="bf16")


@contextlib.contextmanager
def persist(on: bool):
    old = os.environ.get("DFLASH_PERSIST")
    os.environ["DFLASH_PERSIST"] = "1" if on else "0"
    try:
        yield
    finally:
        if old is None:
            del os.environ["DFLASH_PERSIST"]
        else:
            os.environ["DFLASH_PERSIST"] = old


def _inject_in_chunks(g, feats, rows_per_call: int):
    """Inject every request's features through calls of at most rows_per_call rows."""
    B = len(feats)
    done = [0] * B
    per = max(1, rows_per_call // B)
    while any(done[b] < feats[b].shape[0] for b in range(B)):
        part = []
        for b in range(B):
            n = min(per, feats[b].shape[0] - done[b])
            part.append(feats[b][done[b]:done[b] + n])
            done[b] += n
        gpu_inject(g, part, max_rows=rows_per_call)


def _draft_compare(orc, g, anchors, block):
    drafts, logits = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    an, lg, dr = anchors.cpu().numpy(), logits.cpu().numpy(), drafts.cpu().numpy()
    return [orc.check_request(b, int(an[b]), block, lg[b], dr[b]) for b in range(len(an))]


@pytest.mark.parametrize("on", [True, False], ids=["persistent", "multi-kernel"])
@pytest.mark.parametrize("ctxs,block", [([70], 16), ([0, 33], 8), ([1, 64, 5, 100], 4), ([17, 2, 9], 5),
                                        ([40] * 16, 1), ([3] * 8, 2)])
def test_tiny_bf16_small_batches(on, ctxs, block):
    B = len(ctxs)
    with persist(on):
        g = make_gpu(TINY_BF16, seed=21, batch=B, capacity=128, block=block, max_rows=16)
    orc = OracleSide(TINY_BF16, oracle.weights_to_numpy(g.weights), B)
    feats = features_for(TINY_BF16, ctxs, seed=22)
    _inject_in_chunks(g, feats, 16)
    for b in range(B):
        if ctxs[b]:
            orc.inject(b, feats[b].float().cpu().numpy())
    compare_cache(g, orc.exact, tol(TINY_BF16))
    anchors = make_tokens(TINY_BF16, B, seed=23, device="cuda")
    if block > 1:
        _draft_compare(orc, g, anchors, block)
    else:
        drafts, _ = gpu_draft(g, anchors, block)
        torch.cuda.synchronize()
    import block_diffusion_drafter_dflash_gb300 as df
    assert df.dflash_get_status(g.model) == 0


@pytest.mark.parametrize("on", [True, False], ids=["persistent", "multi-kernel"])
def test_8b_bs1_short_context_chunked_injection(on):
    """8B shapes at batch 1, block 16: 48 context tokens injected 16 per call,
    then one draft; both paths against the oracle."""
    wl = workloads()["8b_bs1"]
    cfg, block, ctx = QWEN3_8B, wl.block, 48
    with persist(on):
        g = make_gpu(cfg, seed=wl.seed, batch=1, capacity=ctx + block, block=block, max_rows=16)
    orc = OracleSide(cfg, oracle.weights_to_host(g.weights), 1)
    feats = features_for(cfg, [ctx], seed=wl.seed + 5)
    _inject_in_chunks(g, feats, 16)
    orc.inject(0, feats[0].cpu())
    compare_cache(g, orc.exact, tol(cfg))
    anchors = make_tokens(cfg, 1, seed=wl.seed + 6, device="cuda")
    print(_draft_compare(orc, g, anchors, block))
    import block_diffusion_drafter_dflash_gb300 as df
    assert df.dflash_get_status(g.model) == 0


def test_persistent_draft_is_deterministic():
    """Two drafts of the same inputs give bit-identical logits (stream-K
    partial tiles are summed in a fixed order)."""
    B, block = 2, 8
    with persist(True):
        g = make_gpu(TINY_BF16, seed=31, batch=B, capacity=64, block=block, max_rows=16)
    _inject_in_chunks(g, features_for(TINY_BF16, [30, 12], seed=32), 16)
    anchors = make_tokens(TINY_BF16, B, seed=33, device="cuda")
    d1, l1 = gpu_draft(g, anchors, block)
    d2, l2 = gpu_draft(g, anchors, block)
    torch.cuda.synchronize()
    assert torch.equal(d1, d2) and torch.equal(l1, l2)
