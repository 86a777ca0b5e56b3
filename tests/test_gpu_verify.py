"""Greedy verification kernel vs the oracle: bit-exact, exhaustive on a tiny
vocabulary, and the E[L] closed form by Monte Carlo on the kernel itself."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from dflash_inputs import TINY, make_agreement, make_tokens, replace, synthetic_target_argmax

pytestmark = pytest.mark.gpu


def run_verify(d: torch.Tensor, y: torch.Tensor):
    import block_diffusion_drafter_dflash_gb300 as df
    B, g = y.shape
    d = d.to("cuda", torch.int32).contiguous()
    y = y.to("cuda", torch.int32).contiguous()
    tau = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    out = torch.full((B, g), -9, dtype=torch.int32, device="cuda")
    nxt = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    df.dflash_verify_greedy(d, y, tau, out, nxt)
    torch.cuda.synchronize()
    return tau.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy()


def check_against_oracle(d, y):
    tau, out, nxt = run_verify(d, y)
    dn, yn = d.cpu().numpy(), y.cpu().numpy()
    for b in range(yn.shape[0]):
        t, o, n = oracle.verify_greedy(dn[b], yn[b])
        assert tau[b] == t and list(out[b]) == o and nxt[b] == n, b


@pytest.mark.parametrize("block", [1, 2, 3, 16, 17, 32])
def test_verify_random_blocks_bit_exact(block):
    cfg = replace(TINY, vocab=4)      # a small vocabulary makes long accepted prefixes common
    B = 257
    d = make_tokens(cfg, B * (block - 1), seed=block).reshape(B, block - 1)
    pat = make_agreement(cfg, B, block, [0.8] * B, seed=100 + block)
    y = synthetic_target_argmax(d, pat, cfg.vocab)
    check_against_oracle(d, y)


@pytest.mark.parametrize("block", [1, 2, 4])
def test_verify_exhaustive_tiny_vocab(block):
    V = 3
    pairs = [(dd, yy) for dd in itertools.product(range(V), repeat=block - 1)
             for yy in itertools.product(range(V), repeat=block)]
    d = torch.tensor([p[0] for p in pairs], dtype=torch.int32).reshape(len(pairs), block - 1)
    y = torch.tensor([p[1] for p in pairs], dtype=torch.int32).reshape(len(pairs), block)
    check_against_oracle(d, y)


def test_verify_empty_batch_is_a_no_op():
    run_verify(torch.empty((0, 15), dtype=torch.int32), torch.empty((0, 16), dtype=torch.int32))


@pytest.mark.parametrize("block,p", [(16, 0.9), (16, 0.6), (8, 0.75)])
def test_expected_accept_length_monte_carlo_on_kernel(block, p):
    cfg = replace(TINY, vocab=151936)
    N = 1 << 20
    d = make_tokens(cfg, N * (block - 1), seed=7, device="cuda").reshape(N, block - 1)
    pat = make_agreement(cfg, N, block, [p] * N, seed=8, device="cuda")
    y = synthetic_target_argmax(d, pat, cfg.vocab)
    tau, _, _ = run_verify(d, y)
    tau = tau.astype(np.float64)
    expect = oracle.expected_accept_len([p] * (block - 1))
    assert abs(tau.mean() - expect) < 4 * tau.std() / math.sqrt(N), (tau.mean(), expect)
    assert tau.min() >= 1 and tau.max() <= block


@pytest.mark.parametrize("block,B", [(16, 32), (4, 3), (1, 5), (32, 7)])
def test_synthetic_target_kernel_matches_the_input_recipe(block, B):
    """The benchmark's one-kernel synthetic target equals dflash_inputs'
    torch recipe for every stacked pattern, and advances its counters."""
    import block_diffusion_drafter_dflash_gb300 as df
    cfg = replace(TINY, vocab=151936)
    P = 3
    pats = [make_agreement(cfg, B, block, [0.7] * B, seed=50 + i, device="cuda") for i in range(P)]
    match = torch.stack([p.match for p in pats]).contiguous()
    off = torch.stack([p.off for p in pats]).contiguous()
    bonus = torch.stack([p.bonus for p in pats]).contiguous()
    d = make_tokens(cfg, B * (block - 1), seed=60, device="cuda").reshape(B, block - 1).contiguous()
    pidx = torch.zeros(1, dtype=torch.long, device="cuda")
    tau = torch.arange(1, B + 1, dtype=torch.int32, device="cuda")
    tau_sum = torch.zeros(1, dtype=torch.long, device="cuda")
    y = torch.empty((B, block), dtype=torch.int32, device="cuda")
    for i in range(P + 1):
        df.dflash_synthetic_target(d, match, off, bonus, pidx, y, cfg.vocab, tau=tau, tau_sum=tau_sum)
        ref = synthetic_target_argmax(d, pats[i % P], cfg.vocab)
        assert torch.equal(y, ref), i
    torch.cuda.synchronize()
    assert int(pidx.item()) == (P + 1) % P
    assert int(tau_sum.item()) == (P + 1) * B * (B + 1) // 2
