"""dflash_inject_context_noalloc: the injection entry point for callers that
cannot allocate device memory (it uses the library's fixed static scratch
instead of a caller workspace).  Its cache contents must match those of
dflash_inject_context on the same inputs, over two calls in a row.

Collected last on purpose (file name), so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

from dflash_inputs import QWEN3_8B, TINY, make_features, replace
from parity_util import make_gpu, tol

pytestmark = pytest.mark.gpu


def _pair(cfg, ctx, block):
    import block_diffusion_drafter_dflash_gb300 as df
    a = make_gpu(cfg, seed=11, batch=2, capacity=ctx + 4 * block, block=block, max_rows=max(ctx, block))
    cache_b = df.Cache(a.model, 2, ctx + 4 * block)
    return df, a, cache_b


def _close(x: torch.Tensor, y: torch.Tensor, t: float) -> float:
    x, y = x.float(), y.float()
    den = y.abs().max().clamp_min(1e-30)
    err = float((x - y).abs().max() / den)
    assert err <= t, err
    return err


@pytest.mark.parametrize("cfg", [TINY, replace(TINY, name="tiny-bf16", dtype="bf16"), QWEN3_8B],
                         ids=["tiny-fp32", "tiny-bf16", "8b-bf16"])
def test_noalloc_injection_matches_workspace_injection_twice(cfg):
    block = 16
    ctx = 24 if cfg is QWEN3_8B else 64
    df, a, cache_b = _pair(cfg, ctx, block)
    # call 1: exact host counts; call 2: counts only on the device, padded rows
    f1 = make_features(cfg, ctx, seed=21, device="cuda")
    counts1 = [ctx // 2 + 3, ctx // 2 - 3]
    n1 = torch.tensor(counts1, dtype=torch.int32, device="cuda")
    df.dflash_inject_context(a.model, a.cache, f1, n1, counts1, ctx, a.ws)
    df.dflash_inject_context_noalloc(a.model, cache_b, f1, n1, counts1, ctx)
    f2 = make_features(cfg, block, seed=22, device="cuda")
    n2 = torch.tensor([5, 9], dtype=torch.int32, device="cuda")
    df.dflash_inject_context(a.model, a.cache, f2, n2, None, block, a.ws)
    df.dflash_inject_context_noalloc(a.model, cache_b, f2, n2, None, block)
    torch.cuda.synchronize()
    assert df.dflash_get_status(a.model) == 0
    la, lb = a.cache.ctx_len().cpu().tolist(), cache_b.ctx_len().cpu().tolist()
    assert la == lb == [counts1[0] + 5, counts1[1] + 9]
    for b in range(2):
        c = la[b]
        _close(cache_b.k()[b, :, :, :c], a.cache.k()[b, :, :, :c], tol(cfg))
        _close(cache_b.v()[b, :, :, :c], a.cache.v()[b, :, :, :c], tol(cfg))


def test_noalloc_8b_cycle_injection_of_32_rows():
    """The largest injection of a cycle at batch 2 and block 16 is 32 rows;
    the fixed scratch must hold its plan on this device (the split-K scratch
    grows with the SM count), and the result must match the workspace path."""
    cfg, rows = QWEN3_8B, 32
    df, a, cache_b = _pair(cfg, rows, 16)
    f = make_features(cfg, rows, seed=23, device="cuda")
    counts = [20, 12]
    n = torch.tensor(counts, dtype=torch.int32, device="cuda")
    df.dflash_inject_context(a.model, a.cache, f, n, counts, rows, a.ws)
    df.dflash_inject_context_noalloc(a.model, cache_b, f, n, counts, rows)
    torch.cuda.synchronize()
    assert df.dflash_get_status(a.model) == 0
    assert a.cache.ctx_len().cpu().tolist() == cache_b.ctx_len().cpu().tolist() == counts
    for b in range(2):
        c = counts[b]
        _close(cache_b.k()[b, :, :, :c], a.cache.k()[b, :, :, :c], tol(cfg))
        _close(cache_b.v()[b, :, :, :c], a.cache.v()[b, :, :, :c], tol(cfg))


def test_noalloc_rejects_launches_beyond_its_scratch():
    import block_diffusion_drafter_dflash_gb300 as df
    cfg = QWEN3_8B
    a = make_gpu(cfg, seed=11, batch=1, capacity=4096, block=16, max_rows=16)
    rows = 4096
    f = torch.zeros((rows, cfg.n_target_feats, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    n = torch.tensor([rows], dtype=torch.int32, device="cuda")
    with pytest.raises(df.DFlashError) as e:
        df.dflash_inject_context_noalloc(a.model, a.cache, f, n, [rows], rows)
    assert e.value.code == -3 and "scratch" in str(e.value)
    assert a.cache.ctx_len().cpu().tolist() == [0]          # nothing was launched
    assert df.lib().dflash_noalloc_scratch_bytes() == 8 << 20
