"""The library's block-size scheduling policy (host C++, dflash_block_policy_*)
against the oracle's definition (oracle.acceptance_update,
oracle.acceptance_estimate, oracle.choose_block) on random cycle histories:
the per-position acceptance estimates to 1e-12 and the chosen block size
exactly wherever the best and second-best scores differ by more than 1e-9
relative.  Host code only: no GPU is touched."""
import numpy as np
import pytest

import oracle


@pytest.fixture(scope="module")
def df():
    import block_diffusion_drafter_dflash_gb300 as df
    try:
        df.lib()
    except RuntimeError as e:
        pytest.skip(str(e))
    return df


def _scores(cands, alpha, B, cf, cr, cq):
    return {g: B * oracle.expected_accept_len(list(alpha[:g - 1])) / (cf + cr * B * g + cq * B) for g in cands}


@pytest.mark.parametrize("seed", range(6))
def test_policy_matches_oracle_over_random_histories(df, seed):
    rng = np.random.default_rng(seed)
    cands = sorted(rng.choice(np.arange(2, 33), size=int(rng.integers(1, 6)), replace=False).tolist())
    f32 = lambda x: float(np.float32(x))          # the C ABI carries these parameters as float
    cf, cr, cq = f32(rng.uniform(0.1, 2.0)), f32(rng.uniform(0.0, 0.05)), f32(rng.uniform(0.0, 0.05))
    decay, prior, weight = f32(rng.uniform(0.5, 1.0)), f32(rng.uniform(0.1, 0.99)), f32(rng.uniform(0.5, 4.0))
    pol = df.BlockPolicy(cands, cf, cr, cq, decay=decay, prior_accept=prior, prior_weight=weight)
    gmax = cands[-1]
    acc, att = np.zeros(gmax - 1), np.zeros(gmax - 1)
    exact = 0
    for cycle in range(40):
        B = int(rng.integers(1, 33))
        g, e = pol.choose(B)
        alpha = oracle.acceptance_estimate(acc, att, prior, weight)
        g_o, e_o = oracle.choose_block(cands, alpha, B, cf, cr, cq)
        sc = sorted(_scores(cands, alpha, B, cf, cr, cq).values())
        if len(sc) == 1 or sc[-1] > sc[-2] * (1 + 1e-9):
            assert (g, pytest.approx(e, rel=1e-12)) == (g_o, e_o)
            exact += 1
        taus = [int(t) for t in rng.integers(1, g + 1, size=B)]
        pol.observe(g, taus)
        acc, att = oracle.acceptance_update(acc, att, g, taus, decay)
        np.testing.assert_allclose(pol.acceptance(gmax - 1), oracle.acceptance_estimate(acc, att, prior, weight),
                                   rtol=1e-12, atol=0)
    assert exact >= 30


def test_policy_rejects_bad_configs_and_observations(df):
    with pytest.raises(df.DFlashError):
        df.BlockPolicy([8, 4], 1.0, 0.01)                     # not ascending
    with pytest.raises(df.DFlashError):
        df.BlockPolicy([4, 64], 1.0, 0.01)                    # beyond DFLASH_POLICY_MAX_BLOCK
    with pytest.raises(df.DFlashError):
        df.BlockPolicy([4, 8], 0.0, 0.0, 0.0)                 # no cost at all
    with pytest.raises(df.DFlashError):
        df.BlockPolicy([4, 8], 1.0, 0.01, decay=0.0)
    pol = df.BlockPolicy([4, 8], 1.0, 0.01)
    with pytest.raises(df.DFlashError):
        pol.observe(8, [9])                                  # tau > block
    with pytest.raises(df.DFlashError):
        pol.observe(16, [3])                                 # block beyond the candidates
    with pytest.raises(df.DFlashError):
        pol.choose(0)


def test_policy_switches_to_small_blocks_when_acceptance_collapses(df):
    pol = df.BlockPolicy([4, 8, 16], cost_fixed_ms=1.0, cost_per_row_ms=0.004, decay=0.8)
    rng = np.random.default_rng(5)
    for _ in range(30):
        pol.observe(16, [int(min(16, 1 + rng.geometric(0.05) - 1)) for _ in range(16)])
    assert pol.choose(16)[0] == 16
    for _ in range(30):
        pol.observe(16, [int(min(16, rng.geometric(0.6))) for _ in range(16)])
    assert pol.choose(16)[0] == 4
