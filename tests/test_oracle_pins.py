"""Pins for the CPU oracle: each function is tied to something other than itself.

Sources: the printed DFlash mask matrix and its case definition (blog page
"Inside DFlash & Block Diffusion Speculative Decoding", section 2), the
verification rule and its worked example (explainer page, "The Target Verifier
Remains the Correctness Anchor"), the E[L] closed form (blog page, section 1),
tau in [1, gamma+1] (paper §3.1), the fusion and injection equations (paper
§7.3) and the memory figures that follow them, plus textbook identities
(complex rotation for RoPE, library scaled-dot-product attention).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from dflash_inputs import TINY, DraftConfig, make_agreement, make_features, make_tokens, make_weights, replace

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return np.array(rows, dtype=np.int64)


# ---------------------------------------------------------------- the mask

def test_mask_matches_printed_4plus4_matrix():
    printed = _read_golden("dflash_mask_4plus4.txt")
    assert np.array_equal(oracle.dflash_mask(4, 4), printed)


@pytest.mark.parametrize("t,K", [(0, 1), (0, 4), (1, 1), (3, 5), (7, 16)])
def test_mask_block_rows_see_context_and_whole_block_only(t, K):
    M = oracle.dflash_mask(t, K)
    assert M.shape == (t + K, t + K)
    # block rows: everything (all context + the whole block, in both directions)
    assert np.all(M[t:, :] == 1)
    # context rows never see a block position (no leakage from the masked block)
    assert np.all(M[:t, t:] == 0)


# ---------------------------------------------------------------- attention

def _rand(*shape):
    return rng.standard_normal(shape)


@pytest.mark.parametrize("c,g,nq,nkv", [(0, 4, 4, 2), (5, 4, 4, 2), (17, 3, 8, 2), (9, 16, 4, 4)])
def test_masked_attention_equals_unmasked_over_context_and_block(c, g, nq, nkv):
    hd = 8
    q = _rand(g, nq, hd)
    kc, vc = _rand(c, nkv, hd), _rand(c, nkv, hd)
    kb, vb = _rand(g, nkv, hd), _rand(g, nkv, hd)
    rows = oracle.dflash_mask(c, g)[c:, :]
    a = oracle.attention_masked(q, np.concatenate([kc, kb]), np.concatenate([vc, vb]), rows)
    b = oracle.attention_block(q, kc, vc, kb, vb)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("c,g,nq,nkv", [(6, 4, 4, 2), (0, 5, 6, 3), (11, 2, 2, 1)])
def test_masked_attention_matches_library_sdpa(c, g, nq, nkv):
    """Full [context; block] sequence through torch's fp64 SDPA with a boolean
    mask built from the case definition; block rows must agree."""
    hd = 16
    n = c + g
    q_full = _rand(n, nq, hd)
    k_all, v_all = _rand(n, nkv, hd), _rand(n, nkv, hd)
    M = oracle.dflash_mask(c, g)
    ours = oracle.attention_masked(q_full[c:], k_all, v_all, M[c:, :])
    rep = nq // nkv
    qt = torch.tensor(q_full).permute(1, 0, 2)                       # [nq, n, hd]
    kt = torch.tensor(k_all).permute(1, 0, 2).repeat_interleave(rep, 0)
    vt = torch.tensor(v_all).permute(1, 0, 2).repeat_interleave(rep, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=torch.tensor(M, dtype=torch.bool))
    np.testing.assert_allclose(ours, ref.permute(1, 0, 2).numpy()[c:], rtol=1e-12, atol=1e-12)


def test_attention_identical_keys_gives_mean_of_values():
    c, g, nq, nkv, hd = 7, 4, 4, 2, 8
    key = _rand(1, 1, hd)
    k_all = np.broadcast_to(key, (c + g, nkv, hd)).copy()
    v_all = _rand(c + g, nkv, hd)
    out = oracle.attention_masked(_rand(g, nq, hd), k_all, v_all, np.ones((g, c + g)))
    for h in range(nq):
        np.testing.assert_allclose(out[:, h, :], np.broadcast_to(v_all[:, h // 2, :].mean(0), (g, hd)), rtol=1e-12)


def test_gqa_equals_mha_with_duplicated_kv_heads():
    c, g, nq, nkv, hd = 5, 4, 8, 2, 8
    q = _rand(g, nq, hd)
    k, v = _rand(c + g, nkv, hd), _rand(c + g, nkv, hd)
    ones = np.ones((g, c + g))
    a = oracle.attention_masked(q, k, v, ones)
    b = oracle.attention_masked(q, np.repeat(k, nq // nkv, axis=1), np.repeat(v, nq // nkv, axis=1), ones)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def test_block_is_bidirectional():
    """Row 0 (the anchor) must depend on the last block position's key/value."""
    c, g, nq, nkv, hd = 3, 4, 2, 1, 8
    q, kc, vc = _rand(g, nq, hd), _rand(c, nkv, hd), _rand(c, nkv, hd)
    kb, vb = _rand(g, nkv, hd), _rand(g, nkv, hd)
    a = oracle.attention_block(q, kc, vc, kb, vb)
    vb2 = vb.copy()
    vb2[-1] += 1.0
    b = oracle.attention_block(q, kc, vc, kb, vb2)
    assert np.max(np.abs(a[0] - b[0])) > 1e-6


# ---------------------------------------------------------------- RoPE, norms

def test_rope_is_the_complex_rotation():
    n, H, hd, theta = 9, 3, 16, 1e6
    x = _rand(n, H, hd)
    pos = rng.integers(0, 40000, n)
    out = oracle.rope(x, pos, theta)
    half = hd // 2
    z = x[..., :half] + 1j * x[..., half:]
    freqs = theta ** (-np.arange(half) * 2.0 / hd)
    zr = z * np.exp(1j * pos[:, None, None] * freqs[None, None, :])
    np.testing.assert_allclose(out[..., :half], zr.real, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(out[..., half:], zr.imag, rtol=1e-11, atol=1e-11)


def test_rope_identity_at_zero_norm_preserving_and_relative():
    n, H, hd, theta = 6, 2, 32, 1e6
    x = _rand(n, H, hd)
    np.testing.assert_allclose(oracle.rope(x, np.zeros(n, int), theta), x, rtol=0, atol=0)
    pos = rng.integers(0, 5000, n)
    r = oracle.rope(x, pos, theta)
    np.testing.assert_allclose(np.linalg.norm(r, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-12)
    q, k = _rand(1, 1, hd), _rand(1, 1, hd)
    for p, s, d in [(3, 10, 100), (0, 7, 12345)]:
        a = np.sum(oracle.rope(q, [p], theta) * oracle.rope(k, [s], theta))
        b = np.sum(oracle.rope(q, [p + d], theta) * oracle.rope(k, [s + d], theta))
        assert abs(a - b) < 1e-9


def test_rmsnorm_unit_rms_scale_invariance_and_gain():
    x = _rand(5, 64)
    y = oracle.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, np.ones(64), 0.0), y, rtol=1e-13)
    g = _rand(64)
    np.testing.assert_allclose(oracle.rms_norm(x, g, 0.0), y * g, rtol=1e-13)
    # eps only matters near zero
    assert np.all(oracle.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-6) == 0)


# ---------------------------------------------------------------- fusion / injection

def test_fuse_context_sums_one_slice_of_wc_per_target_layer():
    """[H^(l1);...;H^(l5)] through W_c is the sum over target layers j of the
    D-column slice j of W_c applied to H^(lj) — pins the concatenation order."""
    m, D, n = 5, 12, 4
    feats = _rand(n, m, D)
    w_c = _rand(D, m * D)
    y = sum(feats[:, j, :] @ w_c[:, j * D:(j + 1) * D].T for j in range(m))
    ref = y / np.sqrt(np.mean(y * y, axis=-1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(oracle.fuse_context(feats, w_c, np.ones(D), 1e-6), ref, rtol=1e-12)
    # a slice of feats belonging to a wrong layer gives a different answer
    bad = sum(feats[:, (j + 1) % m, :] @ w_c[:, j * D:(j + 1) * D].T for j in range(m))
    assert not np.allclose(bad, y)


def test_memory_figures_of_the_projection():
    """Paper §7.3: W_c in R^{D x 5D} at D=2048 in BF16 is 5*2048*2048*2 ~ 42 MB; at
    batch 1, sequence 2048 the projection input/output are about 40 MB / 8 MB."""
    cfg = DraftConfig("d2048", hidden=2048, layers=1, n_q_heads=16, n_kv_heads=4, head_dim=128,
                      ffn=64, vocab=8, dtype="bf16")
    w_c_bytes = cfg.hidden * cfg.n_target_feats * cfg.hidden * cfg.elem_bytes
    assert w_c_bytes == 41_943_040 and round(w_c_bytes / 1e6) == 42
    assert round(2048 * 5 * 2048 * 2 / 2**20) == 40
    assert round(2048 * 2048 * 2 / 2**20) == 8


def _tiny_setup(seed=0, layers=2):
    cfg = replace(TINY, layers=layers)
    w = oracle.weights_to_numpy(make_weights(cfg, seed))
    return cfg, w


def test_incremental_injection_equals_one_shot():
    cfg, w = _tiny_setup()
    f = make_features(cfg, 11, seed=5).float().numpy()
    a = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w, cfg, a, f)
    b = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w, cfg, b, f[:4])
    oracle.inject_context(w, cfg, b, f[4:])
    for i in range(cfg.layers):
        np.testing.assert_allclose(a.k[i], b.k[i], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(a.v[i], b.v[i], rtol=1e-12, atol=1e-12)


def test_context_reaches_block_only_through_kv_and_block_never_enters_cache():
    cfg, w = _tiny_setup()
    f = make_features(cfg, 16, seed=6).float().numpy()
    cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w, cfg, cache, f)
    k_before = [k.copy() for k in cache.k]
    out1 = oracle.draft_forward(w, cfg, cache, anchor=3, block=4)["h"]
    assert cache.length == 16 and all(np.array_equal(a, b) for a, b in zip(k_before, cache.k))
    # perturb the context keys/values only: the block output must move
    cache.v[1] = cache.v[1] + 0.5
    out2 = oracle.draft_forward(w, cfg, cache, anchor=3, block=4)["h"]
    assert np.max(np.abs(out1 - out2)) > 1e-6
    # with every W^V zeroed the value path carries no context: then changing
    # the context values changes nothing
    w0 = dict(w, layers=[dict(lw, w_v=np.zeros_like(lw["w_v"])) for lw in w["layers"]])
    c0 = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w0, cfg, c0, f)
    assert np.all(c0.v[0] == 0)


def test_zero_output_projections_reduce_drafter_to_normed_embedding():
    """Special case: W^O = W^D = 0 in every layer leaves x = E[tokens]; then
    h = RMSNorm(E[tokens]) and every mask row drafts argmax(RMSNorm(E[mask]) W_lm^T)."""
    cfg, w = _tiny_setup()
    w0 = dict(w, layers=[dict(lw, w_o=np.zeros_like(lw["w_o"]), w_d=np.zeros_like(lw["w_d"])) for lw in w["layers"]])
    cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w0, cfg, cache, make_features(cfg, 8, seed=9).float().numpy())
    r = oracle.draft_cycle(w0, cfg, cache, None, anchor=17, block=5)
    e = w["embed"][cfg.mask_id].astype(np.float64)
    he = e / np.sqrt(np.mean(e * e) + cfg.rms_eps)
    logits = w["lm_head"].astype(np.float64) @ he
    assert np.all(r["drafts"] == int(np.argmax(logits)))
    np.testing.assert_allclose(r["logits"][0], logits, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_draft_forward_matches_torch_fp64_restatement(qk_norm):
    """Independent restatement with torch library routines (SDPA, silu,
    functional rms_norm for the per-head QK-norm) in float64 over the tiny
    config; RoPE via complex multiplication."""
    cfg = replace(TINY, layers=2, qk_norm=qk_norm)
    w = oracle.weights_to_numpy(make_weights(cfg, 0))
    feats = make_features(cfg, 64, seed=1).float().numpy()
    cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    oracle.inject_context(w, cfg, cache, feats)
    r = oracle.draft_cycle(w, cfg, cache, None, anchor=5, block=4)

    T = lambda a: torch.tensor(np.asarray(a, dtype=np.float64))
    D, nq, nkv, hd, g = cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, 4

    def rms(x):
        return x * torch.rsqrt((x * x).mean(-1, keepdim=True) + cfg.rms_eps)

    def rot(x, pos):
        half = hd // 2
        z = torch.complex(x[..., :half], x[..., half:])
        f = cfg.rope_theta ** (-torch.arange(half, dtype=torch.float64) * 2.0 / hd)
        z = z * torch.polar(torch.ones_like(f), pos[:, None, None].double() * f)
        return torch.cat([z.real, z.imag], -1)

    x_ctx = T(feats).reshape(64, -1) @ T(w["w_c"]).T
    h_t = rms(x_ctx)
    pos_c = torch.arange(64)
    pos_b = torch.arange(64, 64 + g)
    x = T(w["embed"])[[5] + [cfg.mask_id] * (g - 1)]
    def qkn(x, gain):   # per-head norm of a Qwen3-style q_norm / k_norm (library routine)
        if not qk_norm:
            return x
        return torch.nn.functional.rms_norm(x, (hd,), T(gain), eps=cfg.rms_eps)

    for lw in w["layers"]:
        kc = rot(qkn((h_t @ T(lw["w_k"]).T).reshape(64, nkv, hd), lw.get("g_k")), pos_c)
        vc = (h_t @ T(lw["w_v"]).T).reshape(64, nkv, hd)
        u = rms(x)
        q = rot(qkn((u @ T(lw["w_q"]).T).reshape(g, nq, hd), lw.get("g_q")), pos_b)
        kb = rot(qkn((u @ T(lw["w_k"]).T).reshape(g, nkv, hd), lw.get("g_k")), pos_b)
        vb = (u @ T(lw["w_v"]).T).reshape(g, nkv, hd)
        K = torch.cat([kc, kb]).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
        V = torch.cat([vc, vb]).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
        o = torch.nn.functional.scaled_dot_product_attention(q.permute(1, 0, 2), K, V)
        x = x + o.permute(1, 0, 2).reshape(g, nq * hd) @ T(lw["w_o"]).T
        u = rms(x)
        x = x + (torch.nn.functional.silu(u @ T(lw["w_g"]).T) * (u @ T(lw["w_u"]).T)) @ T(lw["w_d"]).T
    logits = rms(x)[1:] @ T(w["lm_head"]).T
    np.testing.assert_allclose(r["logits"], logits.numpy(), rtol=1e-10, atol=1e-10)
    assert np.array_equal(r["drafts"], torch.argmax(logits, -1).numpy())


def test_lm_head_argmax_breaks_ties_to_lowest_index():
    h = np.array([[1.0, 0.0], [0.0, 1.0]])
    W = np.array([[0.0, 0.0], [1.0, 0.0], [0.5, 0.5], [1.0, 0.0], [0.0, 1.0]])
    _, d = oracle.lm_head_argmax(h, W)
    assert list(d) == [1, 4]
    _, d = oracle.lm_head_argmax(np.zeros((1, 2)), W)
    assert list(d) == [0]


# ---------------------------------------------------------------- verification

def test_verify_worked_example():
    for proposals, first_rej, tau_exp, emitted in _read_golden("verify_worked_example.txt"):
        d = list(range(100, 100 + proposals))
        y = list(d) + [999]                   # target agrees everywhere ...
        y[first_rej - 1] = 555                # ... except at proposal `first_rej`
        tau, out, nxt = oracle.verify_greedy(d, y)
        assert tau == tau_exp
        assert out[:emitted] == d[:first_rej - 1] + [555]     # three kept, target supplies the 4th
        assert all(t == -1 for t in out[emitted:])             # proposals 5.. discarded
        assert nxt == 555


def _brute_tau(d, y):
    """Accepted length from its definition: 1 + the largest n such that the
    first n drafts all equal the target's tokens, over every prefix length."""
    best = 0
    for n in range(len(d) + 1):
        if all(d[k] == y[k] for k in range(n)):
            best = max(best, n)
    return best + 1


@pytest.mark.parametrize("block", [1, 2, 4])
def test_verify_exhaustive_tiny_vocab(block):
    V = 3
    for d in itertools.product(range(V), repeat=block - 1):
        for y in itertools.product(range(V), repeat=block):
            tau, out, nxt = oracle.verify_greedy(d, y)
            assert tau == _brute_tau(d, y)
            assert 1 <= tau <= block                         # paper §3.1: tau in [1, gamma+1]
            assert out[:tau] == list(d[:tau - 1]) + [y[tau - 1]]
            assert nxt == y[tau - 1]


def test_expected_accept_length_closed_form_by_monte_carlo():
    """E[L] = 1 + sum_i prod_{j<=i} alpha_j with independent per-position
    agreement; checked on the oracle's verify over synthetic blocks."""
    cfg = replace(TINY, vocab=50)
    for block, p in [(16, [0.9]), (8, [0.6])]:
        N = 60000
        pat = make_agreement(cfg, N, block, p * N, seed=11)
        d = make_tokens(cfg, N * (block - 1), seed=12).reshape(N, block - 1)
        from dflash_inputs import synthetic_target_argmax
        y = synthetic_target_argmax(d, pat, cfg.vocab)
        dn, yn = d.numpy(), y.numpy()
        taus = np.array([oracle.verify_greedy(dn[i], yn[i])[0] for i in range(N)], dtype=np.float64)
        expect = oracle.expected_accept_len([p[0]] * (block - 1))
        assert abs(taus.mean() - expect) < 4 * taus.std() / math.sqrt(N), (taus.mean(), expect)
    assert abs(oracle.expected_accept_len([0.9] * 15) - 8.14697981114816) < 1e-12


def test_speculative_loop_is_lossless_against_a_fake_target():
    """Whatever the drafts are, the emitted stream equals plain greedy decoding
    of the (deterministic) target: explainer step 4-5 and the lossless rule."""
    V = 7

    def target_next(prefix):                       # a deterministic "greedy target"
        h = 0
        for t in prefix[-3:]:
            h = (h * 31 + t + 1) % 1000003
        return (h * 2654435761) % V

    prompt = [1, 2, 3]
    ref = list(prompt)
    while len(ref) < 60:
        ref.append(target_next(ref))

    r = np.random.default_rng(0)
    for block in (1, 2, 5, 16):
        seq = list(prompt)
        anchor = target_next(seq)                  # the first target token is the first anchor
        while len(seq) < 60:
            good = r.random() < 0.7
            drafts, ctx = [], seq + [anchor]
            for _ in range(block - 1):             # drafts: right w.p. ~0.7 per position, else random
                t = target_next(ctx) if (good and r.random() < 0.8) else int(r.integers(V))
                drafts.append(t)
                ctx = ctx + [t]
            ys, ctx = [], seq + [anchor]
            for k in range(block):                 # target's greedy token after each block position
                ys.append(target_next(ctx))
                if k < block - 1:
                    ctx = ctx + [drafts[k]]
            tau, out, nxt = oracle.verify_greedy(drafts, ys)
            seq = seq + [anchor] + out[:tau - 1]   # committed: anchor + accepted drafts
            anchor = nxt                           # correction / bonus is the next anchor
        assert seq[:60] == ref[:60]


# ---------------------------------------------------------------- storage rounding

def test_store_rounding_matches_library_conversions():
    """bf16 storage = torch's float32 -> bfloat16 conversion (round to nearest
    even), applied after rounding to float32; fp32 storage = float32 cast."""
    x = np.concatenate([rng.standard_normal(20000) * 10.0 ** rng.integers(-8, 8, 20000),
                        np.array([0.0, -0.0, 1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 65504.0, -3.0e-38])])
    f32 = x.astype(np.float32)
    ref = torch.tensor(f32).to(torch.bfloat16).float().numpy().astype(np.float64)
    np.testing.assert_array_equal(oracle.store(x, "bf16"), ref)
    np.testing.assert_array_equal(oracle.store(x, "fp32"), f32.astype(np.float64))
    assert oracle.store(x, "f64") is x
    # ties go to even: 1 + 2^-8 sits halfway between two bf16 neighbours
    assert oracle.store(np.array([1.0 + 2.0 ** -8]), "bf16")[0] == 1.0
    assert oracle.store(np.array([1.0 + 3 * 2.0 ** -8]), "bf16")[0] == 1.0 + 2.0 ** -6


def test_storage_mode_only_rounds_between_steps():
    """With fp32 storage the drafter stays within float32 rounding of the
    exact definition, and bf16 storage within bf16 rounding (tiny config)."""
    cfg, w = _tiny_setup()
    f = make_features(cfg, 16, seed=3).float().numpy()
    res = {}
    for mode in ("f64", "fp32", "bf16"):
        c = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
        res[mode] = oracle.draft_cycle(w, cfg, c, f, anchor=9, block=4, mode=mode)["logits"]
    scale = np.max(np.abs(res["f64"]))
    assert np.max(np.abs(res["fp32"] - res["f64"])) / scale < 1e-5
    err = np.max(np.abs(res["bf16"] - res["f64"])) / scale
    assert 1e-5 < err < 5e-2


# ---------------------------------------------------------------------------
# Stochastic lossless verification (explainer, "The Target Verifier Remains the
# Correctness Anchor"): pinned to the losslessness theorem of speculative
# sampling and to its special cases, with the oracle's own decisions counted
# over fine grids of the two uniforms (no random sampling, no retyped formula).
# ---------------------------------------------------------------------------

_GRID = (np.arange(4000) + 0.5) / 4000          # midpoints: fractions exact to 1/4000


def _dist(rng, V, zeros=0):
    p = rng.dirichlet(np.ones(V))
    if zeros:
        p[rng.choice(V, zeros, replace=False)] = 0.0
        p /= p.sum()
    return p


def _accept_fraction(d, pd, pt):
    """Share of u_accept values for which the oracle keeps draft d (block of 1 draft)."""
    P_d, P_t = pd[None, :], np.stack([pt, pt])
    return np.mean([oracle.verify_sampled([d], P_d, P_t, [u], 0.5)[0] == 2 for u in _GRID])


def _correction_dist(d, pd, pt, V):
    """Distribution of the correction after a rejection of draft d, over u_sample."""
    P_d, P_t = pd[None, :], np.stack([pt, pt])
    toks = [oracle.verify_sampled([d], P_d, P_t, [1.0 - 1e-12], u)[2] for u in _GRID]
    return np.bincount(toks, minlength=V) / len(_GRID)


@pytest.mark.parametrize("seed,zeros", [(0, 0), (1, 1), (2, 2)])
def test_sampled_verify_is_lossless(seed, zeros):
    """The first emitted token is distributed exactly as the target's p_t,
    whatever the drafter's p_d: accepted drafts plus corrections."""
    rng = np.random.default_rng(seed)
    V = 5
    pd, pt = _dist(rng, V, zeros), _dist(rng, V, zeros)
    emitted = np.zeros(V)
    for d in range(V):
        if pd[d] == 0.0:
            continue
        a = _accept_fraction(d, pd, pt)
        emitted[d] += pd[d] * a
        if a < 1.0:
            emitted += pd[d] * (1.0 - a) * _correction_dist(d, pd, pt, V)
    assert np.allclose(emitted, pt, atol=2e-3), (emitted, pt)


def test_sampled_verify_acceptance_is_the_overlap_of_the_distributions():
    rng = np.random.default_rng(3)
    V = 6
    pd, pt = _dist(rng, V), _dist(rng, V)
    accept = sum(pd[d] * _accept_fraction(d, pd, pt) for d in range(V))
    assert abs(accept - np.minimum(pd, pt).sum()) < 1e-3


def test_sampled_verify_bonus_follows_the_target_when_every_draft_survives():
    rng = np.random.default_rng(4)
    V, n = 5, 3
    P = np.stack([_dist(rng, V) for _ in range(n + 1)])
    drafts = [1, 3, 0]
    toks = []
    for u in _GRID:
        tau, out, nxt = oracle.verify_sampled(drafts, P[:n], P, [0.999999] * n, u)   # p_d = p_t: always kept
        assert tau == n + 1 and out[:n] == drafts and out[n] == nxt
        toks.append(nxt)
    assert np.allclose(np.bincount(toks, minlength=V) / len(_GRID), P[n], atol=1e-3)


def test_sampled_verify_with_one_hot_distributions_is_greedy_verify():
    rng = np.random.default_rng(5)
    V = 4
    for _ in range(300):
        g = int(rng.integers(1, 6))
        drafts = rng.integers(0, V, g - 1).tolist()
        target = rng.integers(0, V, g).tolist()
        P_d = np.eye(V)[drafts].reshape(g - 1, V)
        P_t = np.eye(V)[target]
        got = oracle.verify_sampled(drafts, P_d, P_t, rng.random(g - 1), float(rng.random()))
        assert got == oracle.verify_greedy(drafts, target)


def test_sampled_verify_rejects_a_token_the_target_never_emits():
    """p_t(d) = 0: rejected for every u; with a one-hot drafter the residual is p_t itself."""
    rng = np.random.default_rng(6)
    V, d = 5, 2
    pt = _dist(rng, V)
    pt[d] = 0.0
    pt /= pt.sum()
    pd = np.eye(V)[d]
    assert _accept_fraction(d, pd, pt) == 0.0
    assert np.allclose(_correction_dist(d, pd, pt, V), pt, atol=1e-3)


# ---------------------------------------------------------------- softmax at a temperature
def test_softmax_matches_library_and_two_token_closed_form():
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    for T in (0.5, 1.0, 1.7):
        x = rng.normal(0.0, 3.0, size=(5, 257))
        np.testing.assert_allclose(oracle.softmax(x, T), scipy_special.softmax(x / T, axis=-1), rtol=1e-13, atol=0)
    # two tokens: p_0 = 1 / (1 + exp((l_1 - l_0) / T)), the logistic function
    for l0, l1, T in [(0.3, -1.2, 1.0), (5.0, 5.5, 0.25), (-2.0, 3.0, 2.0)]:
        p = oracle.softmax(np.array([l0, l1]), T)
        assert p[0] == pytest.approx(1.0 / (1.0 + math.exp((l1 - l0) / T)), rel=1e-14)
        assert p.sum() == pytest.approx(1.0, abs=1e-15)


def test_softmax_shift_invariance_and_zero_temperature_limit():
    rng = np.random.default_rng(8)
    x = rng.normal(0.0, 2.0, size=(3, 100))
    np.testing.assert_allclose(oracle.softmax(x + 123.0, 1.0), oracle.softmax(x, 1.0), rtol=1e-12)
    # T -> 0: all mass on the largest logit (greedy decoding)
    p = oracle.softmax(x, 1e-4)
    np.testing.assert_array_equal(np.argmax(p, axis=-1), np.argmax(x, axis=-1))
    assert np.all(p.max(axis=-1) > 1.0 - 1e-12)


# ---------------------------------------------------------------- block-size scheduling
def _simulate_blocks(alpha, block, n, rng):
    """Accepted lengths of n blocks whose draft j is kept with probability
    alpha[j-1] given the drafts before it were (left to right, stop at the
    first rejection)."""
    taus = []
    for _ in range(n):
        k = 0
        while k < block - 1 and rng.random() < alpha[k]:
            k += 1
        taus.append(k + 1)
    return taus


def test_acceptance_estimate_recovers_the_per_position_rates():
    # with no prior and no forgetting the estimate converges to the rates
    # that generated the blocks; a wrong attempt/keep index would bias it
    rng = np.random.default_rng(21)
    alpha = [0.95, 0.9, 0.85, 0.8, 0.7, 0.6, 0.5]
    acc, att = np.zeros(7), np.zeros(7)
    for block in (8, 6, 8):
        acc, att = oracle.acceptance_update(acc, att, block, _simulate_blocks(alpha, block, 20000, rng), 1.0)
    est = oracle.acceptance_estimate(acc, att, 0.5, 1e-9)
    for j in range(7):
        sd = math.sqrt(alpha[j] * (1 - alpha[j]) / att[j])
        assert abs(est[j] - alpha[j]) < 5 * sd, (j, est[j], alpha[j])
    # positions past a block's last draft are never attempted
    acc2, att2 = oracle.acceptance_update(np.zeros(7), np.zeros(7), 3, [3, 3, 1], 1.0)
    assert att2.tolist() == [3, 2, 0, 0, 0, 0, 0] and acc2.tolist() == [2, 2, 0, 0, 0, 0, 0]


def test_acceptance_estimate_forgets_at_the_decay_rate():
    rng = np.random.default_rng(22)
    acc, att = np.zeros(3), np.zeros(3)
    for _ in range(200):
        acc, att = oracle.acceptance_update(acc, att, 4, _simulate_blocks([0.95] * 3, 4, 8, rng), 0.8)
    for _ in range(60):
        acc, att = oracle.acceptance_update(acc, att, 4, _simulate_blocks([0.3] * 3, 4, 8, rng), 0.8)
    assert abs(oracle.acceptance_estimate(acc, att, 0.5, 1.0)[0] - 0.3) < 0.1
    # one update with decay d scales earlier counts by d
    a1, t1 = oracle.acceptance_update(np.array([4.0, 2.0]), np.array([5.0, 4.0]), 3, [], 0.5)
    assert a1.tolist() == [2.0, 1.0] and t1.tolist() == [2.5, 2.0]


def test_choose_block_maximises_simulated_throughput():
    # brute force: accepted tokens per unit cost of each candidate by Monte
    # Carlo; the choice must be the best one wherever the margin is clear
    rng = np.random.default_rng(23)
    cands = [4, 8, 10, 16]
    checked = 0
    for alpha0, c_row in [(0.98, 0.001), (0.9, 0.01), (0.6, 0.02), (0.3, 0.05), (0.8, 0.0), (0.95, 0.03)]:
        alpha = [alpha0 * (0.99 ** j) for j in range(15)]
        B, cf, creq = 8, 1.0, 0.01
        thr = {}
        for g in cands:
            taus = _simulate_blocks(alpha, g, 20000, rng)
            thr[g] = B * np.mean(taus) / (cf + c_row * B * g + creq * B)
        g_best = max(thr, key=thr.get)
        second = sorted(thr.values())[-2]
        g, e = oracle.choose_block(cands, alpha, B, cf, c_row, creq)
        assert e == pytest.approx(oracle.expected_accept_len(alpha[:g - 1]))
        if thr[g_best] > 1.01 * second:
            assert g == g_best, (alpha0, c_row, thr)
            checked += 1
    assert checked >= 4


def test_choose_block_special_cases():
    cands = [2, 4, 8, 16]
    # free rows and any acceptance: the largest block (E[tau] never falls with g)
    assert oracle.choose_block(cands, [0.5] * 15, 4, 1.0, 0.0, 0.0)[0] == 16
    # nothing is ever accepted: E[tau] = 1 for every g, so the cheapest block
    assert oracle.choose_block(cands, [0.0] * 15, 4, 1.0, 0.1, 0.0) == (2, 1.0)
    # every draft accepted and rows free: tau = g
    assert oracle.choose_block(cands, [1.0] * 15, 1, 1.0, 0.0, 0.0) == (16, 16.0)


def test_qk_norm_makes_the_drafter_invariant_to_the_scale_of_w_q_and_w_k():
    """Special case of the per-head norm: scaling W^Q or W^K by a positive
    constant changes nothing once every query and key head is normalised
    (without QK-norm the same scaling changes the logits).  Exact with
    eps = 0: eps is what breaks the scale invariance of an RMS norm."""
    for qk in (True, False):
        cfg = replace(TINY, layers=2, qk_norm=qk, rms_eps=0.0)
        w = oracle.weights_to_numpy(make_weights(cfg, 3))
        feats = make_features(cfg, 16, seed=4).float().numpy()
        w2 = dict(w, layers=[dict(lw, w_q=lw["w_q"] * 4.0, w_k=lw["w_k"] * 2.0) for lw in w["layers"]])
        out = []
        for ww in (w, w2):
            cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
            out.append(oracle.draft_cycle(ww, cfg, cache, feats, anchor=9, block=4)["logits"])
        if qk:
            np.testing.assert_allclose(out[1], out[0], rtol=1e-9, atol=1e-11)
        else:
            assert np.max(np.abs(out[1] - out[0])) > 1e-4


# ---------------------------------------------------------------- packed training attention
def _packed_inputs(S, anchors, g, nq, nkv, hd, seed=31):
    r = np.random.default_rng(seed)
    N = len(anchors)
    return (r.standard_normal((N * g, nq, hd)), r.standard_normal((S, nkv, hd)), r.standard_normal((S, nkv, hd)),
            r.standard_normal((N * g, nkv, hd)), r.standard_normal((N * g, nkv, hd)))


@pytest.mark.parametrize("S,anchors,g", [(20, [3, 11, 0, 19], 4), (9, [9, 2], 3), (40, [5, 6, 7, 30, 12], 5)])
def test_packed_attention_equals_one_inference_block_per_anchor(S, anchors, g):
    """The packed forward reproduces, block by block, the inference-time block
    attention over the context truncated at the anchor (no mask involved)."""
    nq, nkv, hd = 4, 2, 8
    q, kc, vc, kb, vb = _packed_inputs(S, anchors, g, nq, nkv, hd)
    out = oracle.attention_packed(q, kc, vc, kb, vb, anchors)
    for n, a in enumerate(anchors):
        rows = slice(n * g, (n + 1) * g)
        ref = oracle.attention_block(q[rows], kc[:a], vc[:a], kb[rows], vb[rows])
        np.testing.assert_allclose(out[rows], ref, rtol=1e-12, atol=1e-12)


def test_packed_attention_matches_library_sdpa_with_the_mask():
    S, anchors, g, nq, nkv, hd = 17, [4, 9, 16], 4, 4, 2, 8
    q, kc, vc, kb, vb = _packed_inputs(S, anchors, g, nq, nkv, hd, seed=32)
    M = oracle.packed_block_mask(S, anchors, g)
    K, V = np.concatenate([kc, kb]), np.concatenate([vc, vb])
    rep = nq // nkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q).permute(1, 0, 2), torch.tensor(K).permute(1, 0, 2).repeat_interleave(rep, 0),
        torch.tensor(V).permute(1, 0, 2).repeat_interleave(rep, 0), attn_mask=torch.tensor(M, dtype=torch.bool))
    np.testing.assert_allclose(oracle.attention_packed(q, kc, vc, kb, vb, anchors), ref.permute(1, 0, 2).numpy(),
                               rtol=1e-12, atol=1e-12)


def test_packed_mask_follows_the_explainers_example():
    """Explainer, "Training Rehearses the Same Masked Blocks...": a block
    anchored at r_2 sees its own block (the anchor r_2 included) and the clean
    context before it, never the neighbouring block that begins at r_3."""
    S, g, r2, r3 = 12, 3, 4, 7
    M = oracle.packed_block_mask(S, [r2, r3], g)
    assert M.shape == (2 * g, S + 2 * g)
    for i in range(g):
        assert M[i, :r2].all() and not M[i, r2:S].any()            # context strictly before the anchor
        assert M[i, S:S + g].all()                                  # its own block, bidirectionally
        assert not M[i, S + g:].any()                               # not the block starting at r_3
        assert M[g + i, :r3].all() and not M[g + i, r3:S].any() and M[g + i, S + g:].all() and not M[g + i, S:S + g].any()
    # the same facts seen through the attention output: moving the r_3 block's
    # keys and values, or context at or after r_2, leaves the r_2 block unchanged
    q, kc, vc, kb, vb = _packed_inputs(S, [r2, r3], g, 2, 1, 8, seed=33)
    base = oracle.attention_packed(q, kc, vc, kb, vb, [r2, r3])
    kb2, vb2, vc2 = kb.copy(), vb.copy(), vc.copy()
    kb2[g:] += 1.0
    vb2[g:] -= 2.0
    vc2[r2:] += 3.0
    moved = oracle.attention_packed(q, kc, vc2, kb2, vb2, [r2, r3])
    np.testing.assert_allclose(moved[:g], base[:g], rtol=0, atol=0)
    assert np.max(np.abs(moved[g:] - base[g:])) > 1e-3


def test_per_class_storage_rounding_covers_every_rounding_point():
    """The study mode's classes partition the rounding points: every class in
    bf16 equals the all-bf16 mode, every class exact equals the exact path."""
    cfg, w = _tiny_setup(seed=2)
    feats = make_features(cfg, 12, seed=3).float().numpy()
    out = {}
    for name, mode in [("all", "bf16"), ("each", {c: "bf16" for c in oracle.STORE_CLASSES}),
                       ("exact", "f64"), ("none", {})]:
        cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
        out[name] = oracle.draft_cycle(w, cfg, cache, feats, anchor=4, block=4, mode=mode)["logits"]
    np.testing.assert_array_equal(out["each"], out["all"])
    np.testing.assert_array_equal(out["none"], out["exact"])
    assert np.max(np.abs(out["all"] - out["exact"])) > 0


# ---------------------------------------------------------------- input-fusion ablation
def test_input_fusion_cached_form_equals_the_full_sequence_definition():
    """Injecting the context through the layers once (cached per-layer K/V,
    extended incrementally) and then drafting equals running every layer over
    the whole [context ; block] sequence under the DFlash mask."""
    cfg = replace(TINY, layers=2, input_fusion=True)
    w = oracle.weights_to_numpy(make_weights(cfg, 5))
    feats = make_features(cfg, 23, seed=6).float().numpy()
    cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    for s0, s1 in [(0, 9), (9, 10), (10, 23)]:                  # three injections
        oracle.inject_context(w, cfg, cache, feats[s0:s1])
    r = oracle.draft_cycle(w, cfg, cache, None, anchor=7, block=5)
    full = oracle.draft_forward_full_sequence(w, cfg, feats, anchor=7, block=5)
    logits_full, _ = oracle.lm_head_argmax(full["h"][1:], w["lm_head"])
    np.testing.assert_allclose(r["logits"], logits_full, rtol=1e-10, atol=1e-12)


def test_input_fusion_with_zero_output_projections_gives_the_injected_cache():
    """Special case linking the two conditioning modes: with W_O = W_D = 0 the
    context hidden states stay H_t through every layer, so layer i's context
    keys and values are W^K_i, W^V_i applied to RMSNorm(H_t) — KV injection's
    cache up to the norm's epsilon (exact with eps = 0, H_t having unit RMS)."""
    base = replace(TINY, layers=2, rms_eps=0.0)
    w = oracle.weights_to_numpy(make_weights(base, 8))
    w0 = dict(w, layers=[dict(lw, w_o=np.zeros_like(lw["w_o"]), w_d=np.zeros_like(lw["w_d"])) for lw in w["layers"]])
    feats = make_features(base, 11, seed=9).float().numpy()
    caches = []
    for cfg in (base, replace(base, input_fusion=True)):
        cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
        oracle.inject_context(w0, cfg, cache, feats)
        caches.append(cache)
    for i in range(base.layers):
        np.testing.assert_allclose(caches[1].k[i], caches[0].k[i], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(caches[1].v[i], caches[0].v[i], rtol=1e-11, atol=1e-12)
    # and with the projections on, the two modes differ (the ablation is not a no-op)
    c2 = oracle.RequestCache(base.layers, base.n_kv_heads, base.head_dim)
    oracle.inject_context(w, replace(base, input_fusion=True), c2, feats)
    assert np.max(np.abs(c2.k[1] - caches[0].k[1])) > 1e-3


def test_input_fusion_cache_storage_rounding():
    """With the cached K/V stored in bf16 (storage class "kv"), the input-fusion
    path caches what the exact path computes, rounded: layer 0's context K/V
    (which depend on nothing cached) are exactly the rounded exact values,
    every cached value is a bf16, and deeper layers read the rounded cache
    (so they differ from merely rounding the exact deeper layers)."""
    cfg = replace(TINY, layers=2, input_fusion=True)
    w = oracle.weights_to_numpy(make_weights(cfg, 12))
    feats = make_features(cfg, 14, seed=13).float().numpy()
    ex = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    st = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
    for s0, s1 in [(0, 9), (9, 14)]:
        oracle.inject_context(w, cfg, ex, feats[s0:s1])
        oracle.inject_context(w, cfg, st, feats[s0:s1], {"kv": "bf16"})
    for i in range(cfg.layers):
        for a in (st.k[i], st.v[i]):
            np.testing.assert_array_equal(a, oracle.store(a, "bf16"))
    np.testing.assert_array_equal(st.k[0], oracle.store(ex.k[0], "bf16"))
    np.testing.assert_array_equal(st.v[0], oracle.store(ex.v[0], "bf16"))
    assert not np.array_equal(st.k[1], oracle.store(ex.k[1], "bf16"))
    assert np.max(np.abs(st.k[1] - ex.k[1]) / np.max(np.abs(ex.k[1]))) < 2.0 ** -7


def test_input_fusion_context_rows_are_causal():
    """A later context token never changes an earlier one's cached K/V."""
    cfg = replace(TINY, layers=2, input_fusion=True)
    w = oracle.weights_to_numpy(make_weights(cfg, 10))
    feats = make_features(cfg, 12, seed=11).float().numpy()
    f2 = feats.copy()
    f2[8:] += 1.0
    cs = []
    for f in (feats, f2):
        cache = oracle.RequestCache(cfg.layers, cfg.n_kv_heads, cfg.head_dim)
        oracle.inject_context(w, cfg, cache, f)
        cs.append(cache)
    for i in range(cfg.layers):
        np.testing.assert_array_equal(cs[0].k[i][:8], cs[1].k[i][:8])
        assert np.max(np.abs(cs[0].k[i][8:] - cs[1].k[i][8:])) > 1e-3
